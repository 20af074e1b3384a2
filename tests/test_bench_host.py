"""Host-side pieces of bench.py that the reported numbers rest on, on CPU: the
algorithmic byte count (the roofline numerator), the ncu traffic record's
source check, and the clock sampler's throttle-reason parsing."""
import hashlib
import json
import os
import tempfile

import pytest

import bench
from int4_weight_kv_w4a16_gb300.inputs import LLAMA8B, TOY


def test_block_bytes_8b_batch1_hand_count():
    """8B block, batch 1, 1024 cached positions, counted by hand:
    weights (INT4 codes = rows*cols/2, one fp16 scale per row per 128 inputs):
      QKV 6144x4096: 12,582,912 + 393,216;  O 4096x4096: 8,388,608 + 262,144;
      gate/up 28672x4096: 58,720,256 + 1,835,008;  down 4096x14336: 29,360,128 + 917,504
      -> 112,459,776
    KV (per token per kv-head 64 + 64 code bytes + 2 + 2 scale bytes = 132):
      read 1025 positions x 8 heads x 132 = 1,082,400; new token written 8 x 132 = 1,056
    activations, each written once and read once (bf16): x 8,192 (read by QKV and
      by O's residual), q' 8,192 out + in, o 8,192 out + in, h 8,192 out + in (gate/up)
      + in (down residual), a 28,672 out + in, y 8,192 out -> 139,264
    total 113,682,496."""
    st = bench.stage_bytes(LLAMA8B, [1024])
    assert sum(st.values()) == 113_682_496
    assert st["gate_up"] == 58_720_256 + 1_835_008 + 8_192 + 28_672
    assert st["attention"] == 8_192 + 1_082_400 + 8_192


def test_block_bytes_70b_batch1_hand_count():
    """70B block, batch 1, 2048 cached positions, counted by hand:
    weights: QKV 10240x8192: 41,943,040 + 1,310,720;  O 8192x8192: 33,554,432 + 1,048,576;
      gate/up 57344x8192: 234,881,024 + 7,340,032;  down 8192x28672: 117,440,512 + 3,670,016
      -> 441,188,352
    KV: read 2049 positions x 8 kv-heads x 132 = 2,163,744; new token written 8 x 132 = 1,056
    activations (bf16): x 16,384 x 2 reads, q' 16,384 out + in, o 16,384 out + in, h 16,384 out + 2 in,
      a 57,344 out + in, y 16,384 out -> 278,528
    total 443,631,680."""
    from int4_weight_kv_w4a16_gb300.inputs import LLAMA70B
    st = bench.stage_bytes(LLAMA70B, [2048])
    assert sum(st.values()) == 443_631_680
    assert st["gate_up"] == 234_881_024 + 7_340_032 + 16_384 + 57_344


def test_block_bytes_grow_with_context_and_batch():
    one = bench.stage_bytes(TOY, [100])
    # one more cached position of one sequence: Hkv * (d + 4) more KV bytes
    assert sum(bench.stage_bytes(TOY, [101]).values()) - sum(one.values()) == TOY.n_kv_heads * (TOY.head_dim + 4)
    # a second, empty sequence: its new token's KV read and write plus its activations
    two = bench.stage_bytes(TOY, [100, 0])
    weights = sum(bench.proj_bytes(r, c) for r, c in ((TOY.qkv_rows, TOY.hidden),
                                                        (TOY.hidden, TOY.n_q_heads * TOY.head_dim),
                                                        (2 * TOY.inter, TOY.hidden), (TOY.hidden, TOY.inter)))
    assert sum(two.values()) - weights == 2 * (sum(one.values()) - weights) - 100 * TOY.n_kv_heads * (TOY.head_dim + 4)


def _traffic_root(tmp_path, src_text, workload="wl", nbytes=1234):
    os.makedirs(tmp_path / "profiles")
    (tmp_path / "k.cu").write_text(src_text)
    h = hashlib.sha256(src_text.encode()).hexdigest()[:16]
    rec = {"gate_up": {"dram_bytes_per_launch": nbytes, "workload": workload, "kernel_sources": ["k.cu"],
                       "source_sha256_16": h}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))


def test_profiled_traffic_only_for_its_workload_and_sources(tmp_path, monkeypatch):
    _traffic_root(tmp_path, "kernel v1")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("gate_up", "wl") == 1234
    assert bench.profiled_traffic("gate_up", "other") is None
    assert bench.profiled_traffic("down", "wl") is None
    (tmp_path / "k.cu").write_text("kernel v2")  # the kernel changed since the capture
    assert bench.profiled_traffic("gate_up", "wl") is None


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler_with(rows):
    s = object.__new__(bench.ClockSampler)
    s.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    s.f.write("\n".join(rows) + "\n")
    s.p = _Done()
    return s


def test_clock_sampler_reports_median_and_throttle_reasons():
    rows = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 2070, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 1800, 2070, 1390.0, 0x8, Active, Not Active, Not Active, Active",
            "garbage line"]
    c = _sampler_with(rows).stop()
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0 and c["samples"] == 3
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_clock_sampler_without_nvidia_smi():
    s = object.__new__(bench.ClockSampler)
    s.p = None
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]
    s = object.__new__(bench.ClockSampler)
    s.f, s.p = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False), None
    assert s.stop()["sm_mhz"] is None and not os.path.exists(s.f.name)  # its sample file is removed


def test_clock_sampler_removes_its_sample_file():
    s = _sampler_with(["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active"])
    s.stop()
    assert not os.path.exists(s.f.name)


def test_cpu_baseline_names_the_host():
    from int4_weight_kv_w4a16_gb300.inputs import WORKLOADS
    info = bench.host_info()
    assert set(info) == {"cpu_model", "blas", "blas_threads"} and all(isinstance(v, str) and v for v in info.values())
    base = bench.oracle_baseline(WORKLOADS["toy_b1_ctx128"], budget_s=0.5, max_steps=3)
    assert base["kind"] == "oracle" and base["cores"] >= 1 and base["value"] > 0
    assert base["cpu_model"] == info["cpu_model"] and "block-steps of toy_b1_ctx128" in base["sample"]


def test_sweep_oracle_sample_on_random_operands():
    """The sweep's CPU sample times the unmodified oracle on INT4 operands of the
    workload's shapes drawn directly (codes in [-8, 7], fp16 scales)."""
    import dataclasses
    from int4_weight_kv_w4a16_gb300.inputs import WORKLOADS
    wl = WORKLOADS["toy_b1_ctx128"]
    x, wdq, cache = bench.random_int4_operands(wl.shape, [128, 5], 2)
    assert wdq["qkv"].shape == (TOY.qkv_rows, TOY.hidden) and wdq["down"].shape == (TOY.hidden, TOY.inter)
    assert cache[1]["k_codes"].shape == (TOY.n_kv_heads, 5, TOY.head_dim)
    assert cache[0]["k_codes"].min() >= -8 and cache[0]["k_codes"].max() <= 7
    base = bench.oracle_sample_baseline(wl, budget_s=0.2, max_steps=2)
    assert base["kind"] == "oracle" and base["value"] > 0 and "random INT4 codes" in base["sample"]
    step = bench.step_oracle_sample(dataclasses.replace(wl, n_layers=2, vocab=256), budget_rows=64)
    assert step["value"] > 0 and "x 2 layers" in step["sample"]
