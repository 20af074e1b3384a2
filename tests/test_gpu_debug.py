"""Guard words after the workspace and cache regions, and the debug build's
device bounds checks (libfutr_debug.so, FUTR_DEBUG=1)."""
import os
import subprocess
import sys

import numpy as np
import pytest

from int4_weight_kv_w4a16_gb300 import futr, inputs
from int4_weight_kv_w4a16_gb300.inputs import TOY
from tests._gpu_helpers import GpuBlock

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _child(tmp_path, tag, **env):
    out = tmp_path / f"{tag}.npz"
    e = dict(os.environ)
    e.pop("FUTR_DEBUG", None)
    e.update(env)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "_debug_child.py"), str(out)], env=e,
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    return dict(np.load(out))


def test_guard_words_catch_a_write_past_a_region():
    w = inputs.block_weights(TOY, 0)
    gpu = GpuBlock(TOY, w, max_batch=2, capacity=64)
    gpu.decode(inputs.activations(TOY, 2, 1), np.array([0, 3], np.int32))  # every kernel ran: no false alarm
    assert futr.futr_check(gpu.ws, gpu.kv) == futr.FUTR_OK
    # one word of the guard after h, then of the guard after the cache's streams
    gpu.ws._mem[gpu.ws.off_a - 256 + 4] = 0
    assert futr.futr_check(gpu.ws, None) == futr.FUTR_ERR_CORRUPT
    assert futr.futr_check(None, gpu.kv) == futr.FUTR_OK
    gpu.kv._mem[gpu.kv.rope_offset - 1] = 0
    assert futr.futr_check(None, gpu.kv) == futr.FUTR_ERR_CORRUPT


def test_debug_build_matches_release_bit_for_bit(tmp_path):
    """With the same plan the two builds compute the same bits.  The splits are
    fixed here: the planner sizes them from occupancy, and the debug build's
    kernels use other register counts, so its own choice can differ (and with
    it the order of the fp32 sums)."""
    plan = dict(FUTR_SPLITK="4", FUTR_ATTN_SPLIT="2")
    rel = _child(tmp_path, "release", **plan)
    dbg = _child(tmp_path, "debug", FUTR_DEBUG="1", **plan)
    assert str(rel["lib"]) == "libfutr.so" and str(dbg["lib"]) == "libfutr_debug.so"
    for name in ("toy_b3", "8b_b1"):
        assert rel[name + "_status"].tolist() == [0, 0]
        assert dbg[name + "_status"].tolist() == [0, 0], "a bounds check failed on a valid call"
        np.testing.assert_array_equal(dbg[name + "_y"], rel[name + "_y"])


def test_debug_build_bounds_check_reports_and_recovers(tmp_path):
    """FUTR_TEST_SHRINK_OUT=1 (debug build only) checks the outputs of O,
    gate/up and down against a one-element region: their first writes fail
    the check and are skipped, the step reports FUTR_ERR_BOUNDS, and the next
    step is clean."""
    dbg = _child(tmp_path, "shrink", FUTR_DEBUG="1", FUTR_CHILD_SHRINK="1")
    ok = _child(tmp_path, "plain", FUTR_DEBUG="1")
    for name in ("toy_b3", "8b_b1"):
        assert dbg[name + "_status"].tolist() == [futr.FUTR_ERR_BOUNDS, 0], name
        np.testing.assert_array_equal(dbg[name + "_y"], ok[name + "_y"])
