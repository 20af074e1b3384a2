"""Child process of tests/test_gpu_debug.py: loads the library named by the
environment (FUTR_DEBUG=1: the debug build), runs decode steps and saves their
outputs and statuses to the .npz path given as argv[1]."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from int4_weight_kv_w4a16_gb300 import build, futr, inputs  # noqa: E402
from int4_weight_kv_w4a16_gb300.inputs import LLAMA8B, TOY  # noqa: E402
from tests._gpu_helpers import GpuBlock, bits_to_f64  # noqa: E402

CASES = {"toy_b3": (TOY, 3, [5, 70, 129]), "8b_b1": (LLAMA8B, 1, [1024])}


def run(name, shrink=False):
    shape, b, lengths = CASES[name]
    w = inputs.block_weights(shape, 1)
    gpu = GpuBlock(shape, w, max_batch=b, capacity=max(lengths) + 16)
    gpu.append_history(0, inputs.kv_history(shape, lengths, seed=2))
    x = inputs.activations(shape, b, 3)
    pos = np.asarray(lengths, np.int32)
    import torch
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    pd = torch.from_numpy(pos).cuda()
    y = torch.empty_like(xd)
    if shrink:
        os.environ["FUTR_TEST_SHRINK_OUT"] = "1"
    futr.futr_decode_block(xd, gpu.blob, gpu.kv, 0, b, pd, y, gpu.ws)
    st = futr.futr_check(gpu.ws, gpu.kv)
    os.environ.pop("FUTR_TEST_SHRINK_OUT", None)
    # a second step after the check (counters and error words start over)
    futr.futr_decode_block(xd, gpu.blob, gpu.kv, 0, b, pd, y, gpu.ws)
    st2 = futr.futr_check(gpu.ws, gpu.kv)
    return bits_to_f64(y), st, st2


if __name__ == "__main__":
    if os.environ.get("FUTR_DEBUG") == "1":
        build.build(debug=True)
    out = {}
    for name in CASES:
        y, st, st2 = run(name, shrink=os.environ.get("FUTR_CHILD_SHRINK") == "1")
        out[name + "_y"] = y
        out[name + "_status"] = np.array([st, st2])
    out["lib"] = np.array(os.path.basename(futr.lib()._name))
    np.savez(sys.argv[1], **out)
