"""The device GPTQ packer against the oracle's GPTQ: codes and scales of every
projection, bit for bit, at the toy shape (all rows) and at the Llama-3-8B
shape (sampled rows; GPTQ treats the rows of a projection independently, so
the oracle on a subset of rows gives those rows' exact result).

Both sides take every code and scale decision in fp32 from a float64 working
weight; the float64 sums come in another order on the device (blocked
Cholesky, triangular inverse, trailing updates as GEMMs), so a decision could
only differ where a quotient lies within ~1e-12 relative of a rounding
boundary, which these seeded inputs do not reach."""
import time

import numpy as np
import pytest
import torch

import oracle
from int4_weight_kv_w4a16_gb300 import futr, inputs
from int4_weight_kv_w4a16_gb300.inputs import LLAMA8B, TOY
from tests._gpu_helpers import dev, ensure_lib

pytestmark = pytest.mark.gpu

PROJ = {"qkv": futr.FUTR_PROJ_QKV, "o": futr.FUTR_PROJ_O, "gate": futr.FUTR_PROJ_GATE,
        "up": futr.FUTR_PROJ_UP, "down": futr.FUTR_PROJ_DOWN}


def _hessians(shape, n, seed):
    """Oracle Hessians from synthetic calibration inputs; input 3 of the block
    input and input 5 of the SwiGLU output are zero in all of them (dead)."""
    xa = inputs.calibration_inputs(shape.hidden, n, seed)
    xa[:, 3] = 0.0
    xo = inputs.calibration_inputs(shape.q_rows, n, seed + 1)
    xm = inputs.calibration_inputs(shape.hidden, n, seed + 2)
    xd = inputs.calibration_inputs(shape.inter, n, seed + 3)
    xd[:, 5] = 0.0
    return {"attn": oracle.gptq_hessian(xa), "o": oracle.gptq_hessian(xo), "mlp": oracle.gptq_hessian(xm),
            "down": oracle.gptq_hessian(xd)}


def _pack_gptq(shape, w, h, damp=0.01):
    """Device GPTQ packing into a zeroed blob; returns (shape struct, blob, seconds)."""
    ensure_lib()
    cs = futr.make_shape(shape)
    blob = torch.zeros(futr.futr_weights_size(cs), dtype=torch.uint8, device="cuda")
    scratch = futr.alloc_bytes(futr.futr_gptq_scratch_size(cs))
    wd = {k: dev(v) for k, v in w.items()}
    hd = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in h.items()}
    torch.cuda.synchronize()
    t = time.perf_counter()
    futr.futr_pack_weights_gptq(cs, wd["wq"], wd["wk"], wd["wv"], wd["wo"], wd["wgate"], wd["wup"], wd["wdown"],
                                wd["g_attn"], wd["g_mlp"], hd["attn"], hd["o"], hd["mlp"], hd["down"], damp,
                                scratch, blob)
    sec = time.perf_counter() - t
    del wd, hd, scratch
    return cs, blob, sec


def _unpack(cs, blob, which, rows, cols):
    codes = torch.empty((rows, cols), dtype=torch.int8, device="cuda")
    scales = torch.empty((rows, cols // 128), dtype=torch.int16, device="cuda")
    futr.futr_unpack_weights(cs, blob, which, codes, scales)
    return codes.cpu().numpy(), scales.cpu().numpy()


def _dims(shape, name):
    return {"qkv": (shape.qkv_rows, shape.hidden), "o": (shape.hidden, shape.q_rows),
            "gate": (shape.inter, shape.hidden), "up": (shape.inter, shape.hidden),
            "down": (shape.hidden, shape.inter)}[name]


def test_gptq_pack_bit_exact_toy():
    w = inputs.block_weights(TOY, 4)
    h = _hessians(TOY, 600, seed=40)
    cs, blob, _ = _pack_gptq(TOY, w, h)
    ref = oracle.pack_block_gptq(w, h)
    rtn = oracle.pack_block(w)
    for name, which in PROJ.items():
        c, s = _unpack(cs, blob, which, *_dims(TOY, name))
        np.testing.assert_array_equal(c, ref[name][0], err_msg=name)
        np.testing.assert_array_equal(s, ref[name][1].view(np.int16), err_msg=name)
        # GPTQ moved codes away from round-to-nearest (the test is not vacuous)
        assert np.mean(c != rtn[name][0]) > 0.05, name
    # the dead inputs' codes are 0
    assert np.all(_unpack(cs, blob, futr.FUTR_PROJ_QKV, *_dims(TOY, "qkv"))[0][:, 3] == 0)
    assert np.all(_unpack(cs, blob, futr.FUTR_PROJ_DOWN, *_dims(TOY, "down"))[0][:, 5] == 0)


def test_gptq_diagonal_hessian_gives_round_to_nearest_blob():
    """With diagonal Hessians no error is spread: the GPTQ blob is the RTN blob,
    byte for byte (header included; both start zeroed, so the alignment gaps
    between sections agree too)."""
    w = inputs.block_weights(TOY, 5)
    r = np.random.default_rng(7)
    h = {k: np.diag(r.uniform(0.5, 2.0, n)) for k, n in
         (("attn", TOY.hidden), ("o", TOY.q_rows), ("mlp", TOY.hidden), ("down", TOY.inter))}
    cs, blob, _ = _pack_gptq(TOY, w, h)
    rtn = torch.zeros_like(blob)
    wd = {k: dev(v) for k, v in w.items()}
    futr.futr_pack_weights(cs, wd["wq"], wd["wk"], wd["wv"], wd["wo"], wd["wgate"], wd["wup"], wd["wdown"],
                           wd["g_attn"], wd["g_mlp"], rtn)
    torch.cuda.synchronize()
    assert torch.equal(blob, rtn)


def test_gptq_not_positive_definite_is_reported():
    w = inputs.block_weights(TOY, 6)
    h = _hessians(TOY, 300, seed=41)
    h["attn"] = -np.eye(TOY.hidden)
    with pytest.raises(futr.FutrError) as e:
        _pack_gptq(TOY, w, h)
    assert e.value.status == futr.FUTR_ERR_NOT_PD


def test_gptq_pack_bit_exact_8b_sampled_rows():
    shape = LLAMA8B
    w = inputs.block_weights(shape, 0)
    h = _hessians(shape, 256, seed=50)
    cs, blob, sec = _pack_gptq(shape, w, h)
    print(f"\n8B block GPTQ pack on the device: {sec:.2f} s")
    r = np.random.default_rng(11)
    q, kv = shape.q_rows, shape.kv_rows
    srcs = {"qkv": (np.concatenate([w["wq"], w["wk"], w["wv"]]), w["g_attn"], "attn",
                    [0, q - 1, q, q + kv - 1, q + kv, shape.qkv_rows - 1]),
            "o": (w["wo"], None, "o", [0, shape.hidden - 1]),
            "gate": (w["wgate"], w["g_mlp"], "mlp", [0, 63, 64, shape.inter - 1]),
            "up": (w["wup"], w["g_mlp"], "mlp", [0, 63, 64, shape.inter - 1]),
            "down": (w["wdown"], None, "down", [0, shape.hidden - 1])}
    for name, (mat, g, hk, edge) in srcs.items():
        rows = np.unique(np.concatenate([edge, r.choice(mat.shape[0], 6, replace=False)]))
        c_ref, s_ref = oracle.gptq_quantize_weight(mat[rows], g, h[hk])
        c, s = _unpack(cs, blob, PROJ[name], *_dims(shape, name))
        np.testing.assert_array_equal(c[rows], c_ref, err_msg=name)
        np.testing.assert_array_equal(s[rows], s_ref.view(np.int16), err_msg=name)
