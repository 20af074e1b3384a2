"""futr_decode_block_noalloc: the decode step for callers that cannot
allocate device memory, using the library's fixed scratch array.

The entry runs the same plans and kernels as futr_decode_block, so its output
must equal that entry's bit for bit on the same inputs, on two calls in a row
(the second call runs on whatever the first left in the shared array).
Collected last on purpose: a failure here leaves every other test run.
"""
import numpy as np
import pytest
import torch

from int4_weight_kv_w4a16_gb300 import futr, inputs
from int4_weight_kv_w4a16_gb300.inputs import LLAMA8B, LLAMA70B, TOY
from tests._gpu_helpers import GpuBlock, dev

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 48 * 2**20


def _block(shape, lengths, seed, device_weights=False):
    """A packed block with its cache and workspace.  device_weights: weights and
    history drawn on the device (the comparison is between two entry points, so
    any weights serve), which avoids the host's multi-GB draw at the 70B shape."""
    batch = len(lengths)
    cap = max(lengths) + 16
    if device_weights:
        gpu = GpuBlock.__new__(GpuBlock)
        gpu.shape, gpu.cs = shape, futr.make_shape(shape)
        gpu.blob = futr.alloc_bytes(futr.futr_weights_size(gpu.cs))
        w = inputs.block_weights_device(shape, seed)
        futr.futr_pack_weights(gpu.cs, w["wq"], w["wk"], w["wv"], w["wo"], w["wgate"], w["wup"], w["wdown"],
                               w["g_attn"], w["g_mlp"], gpu.blob)
        del w
        gpu.kv = futr.futr_kv_init(gpu.cs, 1, batch, cap, futr.alloc_bytes(futr.futr_kv_size(gpu.cs, 1, batch, cap)))
        gpu.ws = futr.futr_workspace_init(gpu.cs, batch, cap,
                                          futr.alloc_bytes(futr.futr_workspace_size(gpu.cs, batch, cap)))
        zero = torch.zeros(1, dtype=torch.int32, device="cuda")
        for s, L in enumerate(lengths):
            if L:
                k, v = inputs.kv_history_device(shape, int(L), seed=1000 + s)
                futr.futr_kv_append(gpu.kv, 0, s, 1, zero, int(L), k, v)
    else:
        gpu = GpuBlock(shape, inputs.block_weights(shape, seed), max_batch=batch, capacity=cap)
        gpu.append_history(0, inputs.kv_history(shape, lengths, seed=seed))
    x = dev(inputs.activations(shape, batch, seed).view(np.int16))
    pos = dev(np.asarray(lengths, np.int32))
    torch.cuda.synchronize()
    return gpu, x, pos


CASES = [(TOY, [5, 130, 0], False), (TOY, [(29 * i) % 170 for i in range(32)], False),
         (LLAMA8B, [1024], False), (LLAMA8B, [512 + 113 * i for i in range(32)], True),
         (LLAMA70B, [2048] * 32, True)]


@pytest.mark.parametrize("shape,lengths,device_weights", CASES,
                         ids=["toy_b3", "toy_b32", "8b_b1", "8b_b32", "70b_b32"])
def test_no_alloc_matches_workspace_entry(shape, lengths, device_weights):
    gpu, x, pos = _block(shape, lengths, seed=11, device_weights=device_weights)
    b = len(lengths)
    y_ref = torch.empty_like(x)
    futr.futr_decode_block(x, gpu.blob, gpu.kv, 0, b, pos, y_ref, gpu.ws)
    assert futr.futr_check(gpu.ws, gpu.kv) == 0
    ref = y_ref.cpu().numpy()
    for _ in range(2):  # the same cache slot is rewritten with the same token
        y = torch.zeros_like(x)
        futr.futr_decode_block_noalloc(x, gpu.blob, gpu.kv, 0, b, pos, y)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(y.cpu().numpy(), ref)


@pytest.mark.parametrize("shape", [LLAMA8B, LLAMA70B], ids=["8b", "70b"])
def test_no_alloc_scratch_covers_batch_32(shape):
    """The 8B- and 70B-shaped blocks need at most the fixed scratch at every
    batch up to 32, whatever the cache capacity."""
    cs = futr.make_shape(shape)
    for cap in (64, 65536):
        assert futr.futr_workspace_size(cs, 32, cap) <= SCRATCH_BYTES


def test_no_alloc_rejects_oversized_scratch():
    """A shape whose workspace exceeds the fixed scratch is refused on the host,
    before any launch.  The refusal is established first from the workspace
    size, so the call below can only return the status (its dummy weight
    blob is never read)."""
    import dataclasses
    wide = dataclasses.replace(LLAMA70B, hidden=32768, n_q_heads=256, n_kv_heads=32, inter=131072)
    cs = futr.make_shape(wide)
    batch, cap = 32, 64
    need = futr.futr_workspace_size(cs, batch, cap)
    assert need > SCRATCH_BYTES, need  # otherwise the call below would run
    kv = futr.futr_kv_init(cs, 1, batch, cap, futr.alloc_bytes(futr.futr_kv_size(cs, 1, batch, cap)))
    x = torch.zeros((batch, wide.hidden), dtype=torch.int16, device="cuda")
    y = torch.empty_like(x)
    pos = torch.zeros(batch, dtype=torch.int32, device="cuda")
    blob = futr.alloc_bytes(256)
    st = futr.lib().futr_decode_block_noalloc(x.data_ptr(), blob.data_ptr(), futr.C.byref(kv), 0, batch,
                                              pos.data_ptr(), y.data_ptr(), None)
    assert st == futr.FUTR_ERR_UNSUPPORTED
