"""Multi-rank host logic of bench.py on CPU: two gloo ranks (replicas only,
no collective on the data path; only the timing reduction crosses ranks)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        bench.barrier(w)
        ms = bench.max_over_ranks(10.0 + 5.0 * r, w)  # rank 1 is the slower one
        q.put((r, w, local, ms, bench.whole_job_us_per_step(ms, 100, w)))
        bench.barrier(w)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_whole_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(2))
    for r, (rank, world, local, ms, us) in enumerate(out):
        assert (rank, world, local) == (r, 2, r)
        assert ms == 15.0                       # the slowest rank's time
        assert us == pytest.approx(1000.0 * 15.0 / 200)  # 2 replicas x 100 steps


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_us_per_step(2.0, 100, 1) == pytest.approx(20.0)


def test_reference_arm_runs_only_on_rank_zero(monkeypatch, capsys):
    class A:
        steps, warmup = 1, 3
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(A, bench.inputs.WORKLOADS["toy_b1_ctx128"])
    assert capsys.readouterr().out == ""
