"""Benchmark: INT4 decode block-step on GB300.

Default workload: one Llama-3.1-8B-shaped decoder block (hidden 4096, 32/8
heads, head_dim 128, SwiGLU 14336), batch 1, 1024 cached positions in the INT4
rotated KV cache.  A step is one futr_decode_block call (QKV + RoPE + rotation
+ INT4 KV append, attention, O + residual, gate/up + SwiGLU, down + residual).

Timing: K steps are captured in one CUDA graph (5 kernels per step,
programmatic dependent launch between them); the graph is replayed R times
(--reps, default 10), each replay one timed region of exactly K steps between
CUDA events, bracketed by a barrier and a device synchronize; the value is the
median (min and max reported).  Steps cycle over distinct copies of the layer
(weights and cache) totalling more than 4x the L2, so every step streams from
HBM.  One JSON line on stdout (rank 0).

After the headline workload the same run times the other block and complete
8B-step workloads (the "sweep" object: 8B batch 8 and 32, 70B batch 1, 8 and
32, the 32-layer 8B step at batch 1 and 16), each with its roofline fractions,
clock record and a bounded CPU-oracle sample; --no-sweep skips it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--reps R] [--workload NAME] [--no-sweep]
                  [--impl futr|reference]

The llama8b_x32_* workloads time the complete model step instead (32 blocks,
embedding, final norm and bf16 LM head; futr_decode_step, 164 kernels per step).

--impl reference times the float64 CPU oracle on the host cores instead.
Under torchrun (N > 1) every rank runs an independent replica (no collective
on the data path); elapsed time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from int4_weight_kv_w4a16_gb300 import inputs  # noqa: E402

METRIC = "INT4 decode µs/block-step (8B/70B, batch 1–32); achieved HBM TB/s vs peak"
UNIT = "us/block-step"
N_LAYERS_MODEL = {4096: 32, 8192: 80}


# ------------------------------------------------------------- byte model --

def proj_bytes(rows: int, cols: int) -> int:
    """INT4 codes + fp16 group-128 scales of one projection."""
    return rows * cols // 2 + rows * (cols // 128) * 2


def stage_bytes(shape, lengths) -> dict:
    """Algorithmic HBM bytes of each kernel of one block-step: weights, KV
    codes + scales read (new token included) and written, activations read
    and written once."""
    b = len(lengths)
    H, I, Hq, Hkv, d = shape.hidden, shape.inter, shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    kv_tok = Hkv * (d + 4)
    kv_read = int(sum(int(L) + 1 for L in lengths)) * kv_tok
    qd = Hq * d
    return {
        "qkv": proj_bytes(shape.qkv_rows, H) + b * H * 2 + b * qd * 2 + b * kv_tok,
        "attention": b * qd * 2 + kv_read + b * qd * 2,
        "o": proj_bytes(H, qd) + b * qd * 2 + b * H * 2 + b * H * 2,
        "gate_up": proj_bytes(2 * I, H) + b * H * 2 + b * I * 2,
        "down": proj_bytes(H, I) + b * I * 2 + b * H * 2 + b * H * 2,
    }


STAGES = ["qkv", "attention", "o", "gate_up", "down"]


# ------------------------------------------------------------------ peaks --

def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu record, or
    None when it was taken on another workload or the kernel's sources have
    changed since."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("workload") != workload:
        return None
    h = hashlib.sha256(b"".join(open(os.path.join(ROOT, f), "rb").read() for f in rec["kernel_sources"]))
    return int(rec["dram_bytes_per_launch"]) if h.hexdigest()[:16] == rec["source_sha256_16"] else None


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            f = getattr(self, "f", None)
            if f is not None:
                f.close()
                os.unlink(f.name)
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(", ") for r in self.f.read().strip().splitlines() if r.strip()]
        self.f.close()
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------- distributed glue --

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, world: int) -> float:
    """Max of a float over the process group (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_us_per_step(ms_max: float, steps: int, world: int) -> float:
    """Whole-job µs per block-step: every rank runs `steps` block-steps of its
    own replica in parallel, so N ranks finish N*steps block-steps in the
    slowest rank's time."""
    return 1000.0 * ms_max / (steps * world)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------- CPU baseline --

def host_info() -> dict:
    """CPU model, BLAS library and BLAS thread setting of the host that times the oracle."""
    import platform
    import subprocess
    model = platform.machine()
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        names = [ln.split(":", 1)[1].strip() for ln in out.splitlines() if ln.startswith("Model name:")]
        if names:
            model = f"{names[0]} ({platform.machine()})"
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        blas = np.show_config(mode="dicts")["Build Dependencies"]["blas"]["name"]
    except Exception:  # older numpy: no dict form of the build configuration
        blas = "unknown"
    threads = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS") or "library default"
    return {"cpu_model": model, "blas": blas, "blas_threads": threads}


def _cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def _time_oracle_block(x, wdq, cache, pos, shape, budget_s: float, max_steps: int, min_steps: int = 1):
    import oracle
    times = []
    t_all = time.perf_counter()
    while len(times) < max_steps and (len(times) < min_steps or time.perf_counter() - t_all < budget_s):
        t0 = time.perf_counter()
        oracle.decode_block(x, wdq, cache, pos, shape)
        times.append(time.perf_counter() - t0)
    return times


def oracle_baseline(wl, budget_s: float = 15.0, max_steps: int = 20, min_steps: int = 1):
    """Time the float64 oracle's decode_block on the host cores, on the same
    workload, for a bounded number of block-steps."""
    import oracle
    shape = wl.shape
    lengths = inputs.context_lengths(wl)
    w = inputs.block_weights(shape, 0)
    wdq = oracle.dequant_block(oracle.pack_block(w))
    del w
    x = inputs.activations(shape, wl.batch, 0)
    hist = inputs.kv_history(shape, lengths, n_outlier=wl.n_outlier, seed=0)
    cache = oracle.build_cache(hist, shape)
    del hist
    times = _time_oracle_block(x, wdq, cache, np.asarray(lengths), shape, budget_s, max_steps, min_steps)
    return {"value": 1e6 * statistics.mean(times), "unit": UNIT, "cores": _cores(), "kind": "oracle",
            "sample": f"{len(times)} full block-steps of {wl.name} (float64 numpy, weights pre-dequantized "
                      f"outside the timed region)", **host_info()}


def random_int4_operands(shape, lengths, batch: int, seed: int = 0):
    """Operands of the oracle's decode_block drawn directly as INT4 codes in
    [-8, 7] with fp16 scales (weights per 128-input group, cache per token and
    kv-head): the same shapes as the packed workload without the host-side
    packing of seeded fp32 weights, which would take minutes at the 70B shape.
    The oracle's time does not depend on the values."""
    import oracle
    r = np.random.default_rng(seed)
    H, I, d, Hkv = shape.hidden, shape.inter, shape.head_dim, shape.n_kv_heads

    def proj(n, k):
        c = r.integers(-8, 8, size=(n, k), dtype=np.int8)
        s = r.uniform(1e-3, 4e-3, size=(n, k // 128)).astype(np.float16)
        return oracle.dequant(c, s, 128)

    wdq = {"qkv": proj(shape.qkv_rows, H), "o": proj(H, shape.q_rows), "gate": proj(I, H), "up": proj(I, H),
           "down": proj(H, I)}
    cache = []
    for L in lengths:
        L = int(L)
        cache.append({"k_codes": r.integers(-8, 8, size=(Hkv, L, d), dtype=np.int8),
                      "k_scales": r.uniform(0.1, 1.0, size=(Hkv, L)).astype(np.float16),
                      "v_codes": r.integers(-8, 8, size=(Hkv, L, d), dtype=np.int8),
                      "v_scales": r.uniform(0.1, 1.0, size=(Hkv, L)).astype(np.float16)})
    x = inputs.activations(shape, batch, seed)
    return x, wdq, cache


def oracle_sample_baseline(wl, budget_s: float = 4.0, max_steps: int = 5):
    """The oracle's decode_block on random INT4 operands of this workload's
    shapes (see random_int4_operands), a bounded number of block-steps."""
    lengths = inputs.context_lengths(wl)
    x, wdq, cache = random_int4_operands(wl.shape, lengths, wl.batch)
    times = _time_oracle_block(x, wdq, cache, np.asarray(lengths), wl.shape, budget_s, max_steps)
    return {"value": round(1e6 * statistics.mean(times), 1), "unit": UNIT, "cores": _cores(), "kind": "oracle",
            "sample": f"{len(times)} full block-steps of {wl.name} on random INT4 codes and fp16 scales of its "
                      f"shapes (float64 numpy, weights dequantized outside the timed region)", **host_info()}


# ------------------------------------------------------------- GPU bench --

def time_replays(torch, g, reps: int, world: int):
    """Replay the captured K-step graph `reps` times; each replay is one timed
    region of exactly K steps between CUDA events on the current stream,
    bracketed by a barrier and a device synchronize.  ms per replay (max over
    ranks)."""
    out = []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(reps):
        barrier(world)
        torch.cuda.synchronize()
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        barrier(world)
        out.append(max_over_ranks(e0.elapsed_time(e1), world))
    return out


def capture(torch, step, steps: int, warmup: int):
    """W eager warm-up steps, then K steps captured in one CUDA graph, replayed
    once untimed (uploads the executable graph)."""
    for k in range(warmup):
        step(k)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
            for k in range(steps):
                step(k)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    return g


def replay_stats(ms_list, steps: int) -> dict:
    us = sorted(1000.0 * m / steps for m in ms_list)
    return {"replays": len(us), "median": round(statistics.median(us), 3), "min": round(us[0], 3),
            "max": round(us[-1], 3)}


class Bench:
    def __init__(self, wl, device: int, device_weights: bool = False):
        import torch
        from int4_weight_kv_w4a16_gb300 import build, futr
        build.build()
        self.torch, self.futr = torch, futr
        torch.cuda.set_device(device)
        self.wl, self.shape = wl, wl.shape
        self.cs = futr.make_shape(self.shape)
        self.lengths = inputs.context_lengths(wl)
        self.b = wl.batch
        self.cap = int(max(self.lengths)) + 16
        blob_bytes = futr.futr_weights_size(self.cs)
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        self.n_copies = max(2, math.ceil(4 * l2 / blob_bytes))
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        self.blobs = [futr.alloc_bytes(blob_bytes) for _ in range(self.n_copies)]
        wd = inputs.block_weights_device(self.shape, 0) if device_weights else \
            {k: dev(v) for k, v in inputs.block_weights(self.shape, 0).items()}
        futr.futr_pack_weights(self.cs, wd["wq"], wd["wk"], wd["wv"], wd["wo"], wd["wgate"], wd["wup"],
                               wd["wdown"], wd["g_attn"], wd["g_mlp"], self.blobs[0])
        del wd
        for bl in self.blobs[1:]:
            bl.copy_(self.blobs[0])
        self.kv = futr.futr_kv_init(self.cs, self.n_copies, self.b, self.cap,
                                    futr.alloc_bytes(futr.futr_kv_size(self.cs, self.n_copies, self.b, self.cap)))
        self.ws = futr.futr_workspace_init(self.cs, self.b, self.cap,
                                           futr.alloc_bytes(futr.futr_workspace_size(self.cs, self.b, self.cap)))
        zero = torch.zeros(1, dtype=torch.int32, device="cuda")
        if device_weights:
            for layer in range(self.n_copies):
                for s, L in enumerate(self.lengths):
                    k, v = inputs.kv_history_device(self.shape, int(L), seed=s, n_outlier=wl.n_outlier)
                    futr.futr_kv_append(self.kv, layer, s, 1, zero, int(L), k, v)
        else:
            hist = inputs.kv_history(self.shape, self.lengths, n_outlier=wl.n_outlier, seed=0)
            for layer in range(self.n_copies):
                for s, (kb, vb) in enumerate(hist):
                    futr.futr_kv_append(self.kv, layer, s, 1, zero, kb.shape[1], dev(kb), dev(vb))
            del hist
        self.x = dev(inputs.activations(self.shape, self.b, 0).view(np.int16))
        self.pos = dev(np.asarray(self.lengths, np.int32))
        self.y = torch.empty_like(self.x)
        torch.cuda.synchronize()
        st = futr.futr_check(self.ws, self.kv)
        if st != 0:
            raise RuntimeError(futr.futr_status_string(st))
        self.bytes = stage_bytes(self.shape, self.lengths)
        self.blob_bytes = blob_bytes

    def step(self, k: int):
        layer = k % self.n_copies
        self.futr.futr_decode_block(self.x, self.blobs[layer], self.kv, layer, self.b, self.pos, self.y, self.ws)

    def timed(self, steps: int, warmup: int):
        g = capture(self.torch, self.step, steps, warmup)
        st = self.futr.futr_check(self.ws, self.kv)
        if st != 0:
            raise RuntimeError(self.futr.futr_status_string(st))
        return g

    def stage_times(self, n: int):
        acc = np.zeros(5)
        for k in range(n):
            layer = k % self.n_copies
            acc += np.array(self.futr.futr_decode_block_timed(self.x, self.blobs[layer], self.kv, layer, self.b,
                                                              self.pos, self.y, self.ws))
        return acc / n

    def e2e(self, n: int):
        torch = self.torch
        xh = self.x.cpu().pin_memory()
        ph = self.pos.cpu().pin_memory()
        yh = torch.empty_like(xh).pin_memory()
        # untimed warm-up: a pass over the layer copies
        for k in range(self.n_copies + 1):
            self.futr.futr_decode_block_host(xh, self.blobs[k % self.n_copies], self.kv, k % self.n_copies, self.b,
                                             ph, yh, self.ws)
        t0 = time.perf_counter()
        for k in range(n):
            layer = k % self.n_copies
            self.futr.futr_decode_block_host(xh, self.blobs[layer], self.kv, layer, self.b, ph, yh, self.ws)
        dt = time.perf_counter() - t0
        return {"value": 1e6 * dt / n, "unit": UNIT, "h2d_bytes_per_step": int(self.b * self.shape.hidden * 2 + self.b * 4),
                "d2h_bytes_per_step": int(self.b * self.shape.hidden * 2)}


def block_point(B, args, world: int, pk: dict) -> dict:
    """Time one block workload: R replays of the K-step graph, per-kernel event
    times, and the roofline fractions of the step and of its dominant kernel."""
    torch = B.torch
    g = B.timed(args.steps, args.warmup)
    clocks = ClockSampler(torch.cuda.current_device())
    time.sleep(0.2)
    ms = time_replays(torch, g, args.reps, world)
    clk = clocks.stop()
    st = B.futr.futr_check(B.ws, B.kv)
    if st != 0:
        raise RuntimeError(B.futr.futr_status_string(st))
    stats = replay_stats(ms, args.steps)
    us_step = stats["median"]
    stage_ms = B.stage_times(min(args.steps, 20))
    total = sum(B.bytes.values())
    dom = int(np.argmax(stage_ms))
    dom_name = STAGES[dom]
    dom_gbs = B.bytes[dom_name] / (stage_ms[dom] * 1e-3) / 1e9
    return {"ms_list": ms, "stats": stats, "us_step": us_step, "clocks": clk, "stage_ms": stage_ms,
            "total_bytes": total, "block_gbs": total / (us_step * 1e-6) / 1e9, "dom_name": dom_name,
            "dom_gbs": dom_gbs, "dom_us": stage_ms[dom] * 1e3, "peak": pk["hbm_gbs"]}


def run_futr(args, wl):
    rank, world, local = dist_env()
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    pk = peaks()
    B = Bench(wl, local)
    P = block_point(B, args, world, pk)
    us_step = P["us_step"]
    value = whole_job_us_per_step(us_step * args.steps / 1000.0, args.steps, world)
    e2e = B.e2e(min(args.steps, 50))
    sh = B.shape
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(us_step / 1000.0, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "hidden": sh.hidden, "n_q_heads": sh.n_q_heads, "n_kv_heads": sh.n_kv_heads,
                   "head_dim": sh.head_dim, "inter": sh.inter, "batch": B.b,
                   "ctx": "ragged %d-%d (mean %.0f)" % (wl.ragged[0], wl.ragged[1], np.mean(B.lengths))
                   if wl.ragged else int(wl.ctx),
                   "weights": "int4 group-128 fp16 scales", "kv_cache": "int4 Hadamard-rotated, fp16 scale per token-head",
                   "l2": f"steps cycle {B.n_copies} distinct layer copies ({B.n_copies * B.blob_bytes / 1e6:.0f} MB of weights) "
                         f"> 4x L2",
                   "timing": f"median of {args.reps} timed regions, each exactly K={args.steps} steps of one CUDA "
                             f"graph (5 kernels/step, programmatic dependent launch)",
                   "parallelism": f"replicas x{world}"},
        "replays_us_per_step": P["stats"],
        "block_roofline": {"bound": "hbm", "algorithmic_bytes": int(P["total_bytes"]),
                           "achieved": round(P["block_gbs"], 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                           "frac": round(P["block_gbs"] / pk["hbm_gbs"], 4), "peak_source": pk["source"]},
        "roofline": {"kernel": P["dom_name"], "bound": "hbm", "achieved": round(P["dom_gbs"], 1),
                     "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(P["dom_gbs"] / pk["hbm_gbs"], 4),
                     "traffic": profiled_traffic(P["dom_name"], wl.name),
                     "algorithmic_bytes": int(B.bytes[P["dom_name"]]), "avg_launch_us": round(P["dom_us"], 3),
                     "peak_source": pk["source"]},
        "stage_us": {n: round(float(t) * 1e3, 3) for n, t in zip(STAGES, P["stage_ms"])},
        "tokens_per_s_blocks_only": round(B.b / (us_step * 1e-6 * N_LAYERS_MODEL.get(sh.hidden, 32)), 1),
        "e2e": e2e, "clocks": P["clocks"], "gpu_launches": 5 * args.steps * args.reps,
    }
    del B
    if world == 1 and not args.no_sweep:
        line["sweep"] = run_sweep(args, world, pk)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(wl)
    if rank == 0:
        out = json.dumps(line)
        print(out, flush=True)
        if args.out:
            with open(args.out, "a") as f:
                f.write(out + "\n")
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


SWEEP = ["llama8b_b8_ctx1024", "llama8b_b32_ragged512-4096", "llama70b_b1_ctx2048", "llama70b_b8_ctx2048",
         "llama70b_b32_ctx2048", "llama8b_x32_b1_ctx2048", "llama8b_x32_b16_ctx2048"]


def run_sweep(args, world: int, pk: dict) -> dict:
    """The other block and complete-step workloads, each timed like the
    headline (R regions of exactly K steps) in this run; weights and cache
    histories drawn on the device.  Each point carries its own clock record
    and a bounded CPU-oracle sample."""
    import gc
    import torch
    out = {}
    for name in SWEEP:
        wl = inputs.WORKLOADS[name]
        if wl.vocab > 0:
            B = StepBench(wl, torch.cuda.current_device())
            g = B.timed(args.steps, args.warmup)
            clocks = ClockSampler(torch.cuda.current_device())
            time.sleep(0.2)
            ms = time_replays(torch, g, args.reps, world)
            clk = clocks.stop()
            st = B.futr.futr_check(B.ws, B.kv)
            if st != 0:
                raise RuntimeError(B.futr.futr_status_string(st))
            stats = replay_stats(ms, args.steps)
            total = sum(B.bytes.values())
            gbs = total / (stats["median"] * 1e-6) / 1e9
            rec = {"unit": STEP_UNIT, "us_per_step": stats, "batch": wl.batch, "layers": wl.n_layers,
                   "tokens_per_s": round(wl.batch / (stats["median"] * 1e-6), 1),
                   "step_roofline": {"algorithmic_bytes": int(total), "achieved": round(gbs, 1), "unit": "GB/s",
                                     "frac": round(gbs / pk["hbm_gbs"], 4)},
                   "clocks": clk}
            del g, B
            gc.collect()
            torch.cuda.empty_cache()
            if not args.no_cpu_baseline:
                rec["cpu_baseline"] = step_oracle_sample(wl)
        else:
            B = Bench(wl, torch.cuda.current_device(), device_weights=True)
            P = block_point(B, args, world, pk)
            rec = {"unit": UNIT, "us_per_step": P["stats"], "batch": wl.batch,
                   "block_roofline": {"algorithmic_bytes": int(P["total_bytes"]), "achieved": round(P["block_gbs"], 1),
                                      "unit": "GB/s", "frac": round(P["block_gbs"] / pk["hbm_gbs"], 4)},
                   "dominant": {"kernel": P["dom_name"], "achieved": round(P["dom_gbs"], 1),
                                "frac": round(P["dom_gbs"] / pk["hbm_gbs"], 4), "avg_launch_us": round(P["dom_us"], 3)},
                   "stage_us": {n: round(float(t) * 1e3, 3) for n, t in zip(STAGES, P["stage_ms"])},
                   "tokens_per_s_blocks_only": round(
                       wl.batch / (P["us_step"] * 1e-6 * N_LAYERS_MODEL.get(wl.shape.hidden, 32)), 1),
                   "clocks": P["clocks"]}
            del B
            gc.collect()
            torch.cuda.empty_cache()
            if not args.no_cpu_baseline:
                rec["cpu_baseline"] = oracle_sample_baseline(wl)
        rec["peak_gbs"] = pk["hbm_gbs"]
        out[name] = rec
    return out


# --------------------------------------------------- complete decode step --

STEP_METRIC = "INT4 decode µs/step, complete 8B model (32 INT4 blocks + embedding + bf16 LM head)"
STEP_UNIT = "us/step"


class StepBench:
    """The complete model: n_layers packed blocks (weights drawn on the GPU,
    one seed per layer), one INT4 cache with every layer's history, embedding,
    final gain and bf16 LM head; a step is one futr_decode_step call."""

    def __init__(self, wl, device: int):
        import torch
        from int4_weight_kv_w4a16_gb300 import build, futr
        build.build()
        self.torch, self.futr = torch, futr
        torch.cuda.set_device(device)
        self.wl, self.shape, self.b, self.vocab = wl, wl.shape, wl.batch, wl.vocab
        self.cs = futr.make_shape(self.shape)
        self.lengths = inputs.context_lengths(wl)
        self.cap = int(max(self.lengths)) + 16
        nbytes = futr.futr_weights_size(self.cs)
        self.blobs = []
        for l in range(wl.n_layers):
            w = inputs.block_weights_device(self.shape, l)
            blob = futr.alloc_bytes(nbytes)
            futr.futr_pack_weights(self.cs, w["wq"], w["wk"], w["wv"], w["wo"], w["wgate"], w["wup"], w["wdown"],
                                   w["g_attn"], w["g_mlp"], blob)
            del w
            self.blobs.append(blob)
        self.kv = futr.futr_kv_init(self.cs, wl.n_layers, self.b, self.cap,
                                    futr.alloc_bytes(futr.futr_kv_size(self.cs, wl.n_layers, self.b, self.cap)))
        self.ws = futr.futr_workspace_init(self.cs, self.b, self.cap,
                                           futr.alloc_bytes(futr.futr_workspace_size(self.cs, self.b, self.cap)))
        zero = torch.zeros(1, dtype=torch.int32, device="cuda")
        for l in range(wl.n_layers):
            for s in range(self.b):
                k, v = inputs.kv_history_device(self.shape, int(self.lengths[s]), seed=1000 * l + s)
                futr.futr_kv_append(self.kv, l, s, 1, zero, int(self.lengths[s]), k, v)
        g = torch.Generator(device="cuda").manual_seed(12345)
        self.embedding = torch.randn((self.vocab, self.shape.hidden), generator=g, device="cuda").to(torch.bfloat16)
        self.lm_head = (torch.randn((self.vocab, self.shape.hidden), generator=g, device="cuda") * 0.02).to(
            torch.bfloat16)
        self.g_final = torch.rand(self.shape.hidden, generator=g, device="cuda") + 0.5
        self.tokens = torch.from_numpy((np.arange(self.b) * 7919 + 11) % self.vocab).int().cuda()
        self.pos = torch.from_numpy(np.asarray(self.lengths, np.int32)).cuda()
        self.logits = torch.empty((self.b, self.vocab), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        st = futr.futr_check(self.ws, self.kv)
        if st != 0:
            raise RuntimeError(futr.futr_status_string(st))
        blk = stage_bytes(self.shape, self.lengths)
        H = self.shape.hidden
        self.bytes = {"blocks": wl.n_layers * sum(blk.values()), "embedding": self.b * H * 2,
                      "lm_head": self.vocab * H * 2 + self.b * H * 2 + self.b * self.vocab * 4}

    def step(self, tokens=None, pos=None, logits=None):
        self.futr.futr_decode_step(self.tokens if tokens is None else tokens, self.embedding, self.vocab, self.blobs,
                                   self.kv, self.b, self.pos if pos is None else pos, self.g_final, self.lm_head,
                                   self.logits if logits is None else logits, self.ws)

    def timed(self, steps: int, warmup: int):
        g = capture(self.torch, lambda k: self.step(), steps, warmup)
        st = self.futr.futr_check(self.ws, self.kv)
        if st != 0:
            raise RuntimeError(self.futr.futr_status_string(st))
        return g

    def e2e(self, n: int):
        """Tokens and positions from pinned host memory, logits back to the host,
        every step (wall clock)."""
        torch = self.torch
        th = self.tokens.cpu().pin_memory()
        ph = self.pos.cpu().pin_memory()
        lh = torch.empty((self.b, self.vocab), dtype=torch.float32).pin_memory()
        td, pd = torch.empty_like(self.tokens), torch.empty_like(self.pos)
        for k in range(n + 3):
            if k == 3:
                torch.cuda.synchronize()
                t0 = time.perf_counter()
            td.copy_(th, non_blocking=True)
            pd.copy_(ph, non_blocking=True)
            self.step(td, pd)
            lh.copy_(self.logits, non_blocking=True)
            torch.cuda.current_stream().synchronize()
        dt = time.perf_counter() - t0
        return {"value": 1e6 * dt / n, "unit": STEP_UNIT, "h2d_bytes_per_step": int(8 * self.b),
                "d2h_bytes_per_step": int(4 * self.b * self.vocab)}


def step_oracle_baseline(wl, budget_rows: int = 8192):
    """The oracle on the host cores, extrapolated: one block-step of this shape
    and batch (weights pre-dequantized) times n_layers, plus the final norm and
    LM head on ``budget_rows`` vocabulary rows scaled to the full vocabulary."""
    import oracle
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sh = wl.shape
    lengths = inputs.context_lengths(wl)
    w = inputs.block_weights(sh, 0)
    wdq = oracle.dequant_block(oracle.pack_block(w))
    del w
    x = inputs.activations(sh, wl.batch, 0)
    cache = oracle.build_cache(inputs.kv_history(sh, lengths, n_outlier=wl.n_outlier, seed=0), sh)
    pos = np.asarray(lengths)
    oracle.decode_block(x, wdq, cache, pos, sh)
    t0 = time.perf_counter()
    out = oracle.decode_block(x, wdq, cache, pos, sh)
    t_block = time.perf_counter() - t0
    r = np.random.default_rng(0)
    w_rows = inputs.to_bf16_bits(r.standard_normal((budget_rows, sh.hidden)).astype(np.float32) * 0.02)
    g = r.uniform(0.5, 1.5, sh.hidden).astype(np.float32)
    t0 = time.perf_counter()
    oracle.final_logits(out["y"], g, w_rows, sh.rms_eps)
    t_head = (time.perf_counter() - t0) * wl.vocab / budget_rows
    us = 1e6 * (t_block * wl.n_layers + t_head)
    return {"value": round(us, 1), "unit": STEP_UNIT, "cores": cores, "kind": "oracle",
            "sample": f"1 block-step of {sh.hidden}-hidden batch {wl.batch} x {wl.n_layers} layers + final norm and "
                      f"LM head on {budget_rows} of {wl.vocab} rows scaled to the vocabulary (float64 numpy)",
            **host_info()}


def step_oracle_sample(wl, budget_rows: int = 8192):
    """As step_oracle_baseline, on random INT4 operands of the block's shapes
    (random_int4_operands) instead of packed seeded weights."""
    import oracle
    sh = wl.shape
    lengths = inputs.context_lengths(wl)
    x, wdq, cache = random_int4_operands(sh, lengths, wl.batch)
    pos = np.asarray(lengths)
    t_block = min(_time_oracle_block(x, wdq, cache, pos, sh, 0.0, 2, 2))
    y = oracle.decode_block(x, wdq, cache, pos, sh)["y"]
    r = np.random.default_rng(0)
    w_rows = inputs.to_bf16_bits(r.standard_normal((budget_rows, sh.hidden)).astype(np.float32) * 0.02)
    g = r.uniform(0.5, 1.5, sh.hidden).astype(np.float32)
    t0 = time.perf_counter()
    oracle.final_logits(y, g, w_rows, sh.rms_eps)
    t_head = (time.perf_counter() - t0) * wl.vocab / budget_rows
    return {"value": round(1e6 * (t_block * wl.n_layers + t_head), 1), "unit": STEP_UNIT, "cores": _cores(),
            "kind": "oracle",
            "sample": f"the faster of 2 block-steps of {sh.hidden}-hidden batch {wl.batch} on random INT4 codes and "
                      f"fp16 scales x {wl.n_layers} layers + final norm and LM head on {budget_rows} of {wl.vocab} "
                      f"rows scaled to the vocabulary (float64 numpy)", **host_info()}


def run_step(args, wl):
    rank, world, local = dist_env()
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    B = StepBench(wl, local)
    g = B.timed(args.steps, args.warmup)
    clocks = ClockSampler(local)
    time.sleep(0.3)
    ms_list = time_replays(torch, g, args.reps, world)
    clk = clocks.stop()
    st = B.futr.futr_check(B.ws, B.kv)
    if st != 0:
        raise RuntimeError(B.futr.futr_status_string(st))
    stats = replay_stats(ms_list, args.steps)
    us_step = stats["median"]
    ms = us_step * args.steps / 1000.0
    value = whole_job_us_per_step(ms, args.steps, world)
    pk = peaks()
    total = sum(B.bytes.values())
    gbs = total / (us_step * 1e-6) / 1e9
    e2e = B.e2e(min(args.steps, 20))
    line = {
        "metric": STEP_METRIC, "value": round(value, 3), "unit": STEP_UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "layers": wl.n_layers, "vocab": wl.vocab, "batch": B.b, "ctx": int(wl.ctx),
                   "weights": "int4 group-128 fp16 scales; bf16 embedding and LM head",
                   "l2": f"{sum(B.bytes.values()) / 1e9:.2f} GB streamed per step > L2",
                   "timing": f"median of {args.reps} timed regions, each exactly K={args.steps} steps of one CUDA "
                             f"graph ({2 + 5 * wl.n_layers + 2} kernels/step, programmatic dependent launch)",
                   "parallelism": f"replicas x{world}"},
        "replays_us_per_step": stats,
        "roofline": {"kernel": "whole step", "bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4), "traffic": None,
                     "algorithmic_bytes": int(total), "peak_source": pk["source"]},
        "tokens_per_s": round(B.b / (us_step * 1e-6), 1),
        "e2e": e2e, "clocks": clk, "gpu_launches": (2 + 5 * wl.n_layers + 2) * args.steps * args.reps,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = step_oracle_baseline(wl)
    if rank == 0:
        out = json.dumps(line)
        print(out, flush=True)
        if args.out:
            with open(args.out, "a") as f:
                f.write(out + "\n")
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    import oracle
    shape = wl.shape
    lengths = inputs.context_lengths(wl)
    w = inputs.block_weights(shape, 0)
    wdq = oracle.dequant_block(oracle.pack_block(w))
    del w
    x = inputs.activations(shape, wl.batch, 0)
    hist = inputs.kv_history(shape, lengths, n_outlier=wl.n_outlier, seed=0)
    cache = oracle.build_cache(hist, shape)
    pos = np.asarray(lengths)
    for _ in range(args.warmup):
        oracle.decode_block(x, wdq, cache, pos, shape)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode_block(x, wdq, cache, pos, shape)
    dt = time.perf_counter() - t0
    us = 1e6 * dt / args.steps
    line = {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1000, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "batch": wl.batch},
            "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} full block-steps of {wl.name}, float64 numpy oracle",
                             **host_info()},
            "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="llama8b_b1_ctx1024", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--impl", default="futr", choices=["futr", "reference"])
    ap.add_argument("--out", default=None, help="also append the JSON line to this file")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reps", type=int, default=10, help="timed regions of exactly K steps (median reported)")
    ap.add_argument("--no-sweep", action="store_true", help="time the chosen workload only")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = inputs.WORKLOADS[args.workload]
    if wl.vocab > 0:  # the complete model step
        if args.impl == "reference":
            rank, world, _ = dist_env()
            if rank == 0:
                base = step_oracle_baseline(wl)
                print(json.dumps({"impl": "reference", "metric": STEP_METRIC, "value": base["value"],
                                  "unit": STEP_UNIT, "n_gpus": world, "steps": 1, "warmup": 1,
                                  "ms_per_step": round(base["value"] / 1000, 3), "higher_is_better": False,
                                  "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                                  "config": {"workload": wl.name, "batch": wl.batch}, "cpu_baseline": base,
                                  "e2e": {"value": base["value"], "unit": STEP_UNIT, "h2d_bytes_per_step": 0,
                                          "d2h_bytes_per_step": 0}}), flush=True)
        else:
            run_step(args, wl)
        return
    if args.impl == "reference":
        if args.steps > 20:
            args.steps = 20  # bounded CPU sample
        run_reference(args, wl)
    else:
        run_futr(args, wl)


if __name__ == "__main__":
    main()
