"""70B-shaped block (hidden 8192, 64/8 heads, SwiGLU 28672) at full size,
batch 1, 8 and 32 with 2048 cached positions: the CUDA path runs the whole
block; the oracle checks sampled outputs one by one, each stage fed the GPU's
own input to that stage (its full float64 evaluation would need ~7 GB of
dequantized weights per call)."""
import numpy as np
import pytest
import torch

import oracle
from int4_weight_kv_w4a16_gb300 import futr, inputs
from int4_weight_kv_w4a16_gb300.inputs import LLAMA70B
from tests._gpu_helpers import GpuBlock, assert_close, bits_to_f64, dev

pytestmark = pytest.mark.gpu

SH = LLAMA70B
CTX = 2048
STAGE_REL = 3e-4
R = np.random.default_rng(70)
Q_HEADS = sorted(R.choice(SH.n_q_heads, 6, replace=False).tolist())
KV_HEADS = sorted({h // (SH.n_q_heads // SH.n_kv_heads) for h in Q_HEADS} | {0, SH.n_kv_heads - 1})
ROWS_H = sorted(R.choice(SH.hidden, 96, replace=False).tolist())
ROWS_I = sorted(R.choice(SH.inter, 96, replace=False).tolist())


@pytest.fixture(scope="module")
def block():
    w = inputs.block_weights(SH, 0)
    gpu = GpuBlock(SH, w, max_batch=32, capacity=CTX + 16)
    hist = inputs.kv_history(SH, [CTX] * 32, seed=0)
    gpu.append_history(0, hist)
    del hist
    return gpu, w


def _dq(w, g, rows):
    c, s = oracle.quantize_weight(w[rows], g, 128)
    return oracle.dequant(c, s, 128)


def test_pack_sampled_rows_bit_exact(block):
    gpu, w = block
    for which, key, g, rows in ((futr.FUTR_PROJ_QKV, None, w["g_attn"], ROWS_H[:32]),
                                (futr.FUTR_PROJ_O, "wo", None, ROWS_H[:32]),
                                (futr.FUTR_PROJ_GATE, "wgate", w["g_mlp"], ROWS_I[:32]),
                                (futr.FUTR_PROJ_UP, "wup", w["g_mlp"], ROWS_I[:32]),
                                (futr.FUTR_PROJ_DOWN, "wdown", None, ROWS_H[:32])):
        src = np.concatenate([w["wq"], w["wk"], w["wv"]]) if key is None else w[key]
        c, s = gpu.unpack(which)
        rc, rs = oracle.quantize_weight(src[rows], g, 128)
        np.testing.assert_array_equal(c[rows], rc)
        np.testing.assert_array_equal(s[rows].view(np.uint16), rs.view(np.uint16))


@pytest.mark.parametrize("batch", [1, 8, 32])
def test_decode_70b_sampled_stages(block, batch):
    gpu, w = block
    x = inputs.activations(SH, batch, 1 + batch)
    pos = np.full(batch, CTX, np.int32)
    y = bits_to_f64(gpu.decode(x, pos))
    inter = gpu.intermediates(batch)
    xf = oracle.bf16_bits_to_float(x)
    d, rep = SH.head_dim, SH.n_q_heads // SH.n_kv_heads
    r1 = oracle.rms_factor(xf, SH.rms_eps)

    # QKV: sampled query heads (RoPE + rotation) and the new token's K/V codes
    for h in Q_HEADS:
        wq = _dq(w["wq"], w["g_attn"], slice(h * d, (h + 1) * d))
        q = oracle.rope((r1[:, None] * (xf @ wq.T))[:, None, :], pos, SH.rope_theta)
        assert_close(inter["q_rot"][:, h], oracle.rotate(q, SH.had_block)[:, 0], f"q_rot head {h}", rel=STAGE_REL)
    caches = [gpu.read_cache(0, i, CTX + 1) for i in range(batch)]
    for kvh in KV_HEADS:
        wk = _dq(w["wk"], w["g_attn"], slice(kvh * d, (kvh + 1) * d))
        wv = _dq(w["wv"], w["g_attn"], slice(kvh * d, (kvh + 1) * d))
        k = oracle.rope((r1[:, None] * (xf @ wk.T))[:, None, :], pos, SH.rope_theta)[:, 0]
        v = r1[:, None] * (xf @ wv.T)
        kc, ks = oracle.kv_quantize(k.astype(np.float32), SH.had_block)
        vc, vs = oracle.kv_quantize(v.astype(np.float32), SH.had_block)
        for i in range(batch):
            for got, ref in ((caches[i]["k_codes"][kvh, CTX], kc[i]), (caches[i]["v_codes"][kvh, CTX], vc[i])):
                assert np.abs(got.astype(int) - ref.astype(int)).max() <= 1
            for got, ref in ((caches[i]["k_scales"][kvh, CTX], ks[i]), (caches[i]["v_scales"][kvh, CTX], vs[i])):
                assert abs(float(got) - float(ref)) <= abs(float(ref)) * 2.0 ** -10

    # attention: sampled kv-heads, on the GPU's query and cache
    for kvh in KV_HEADS:
        for i in range(batch):
            kf = caches[i]["k_codes"][kvh].astype(np.float64) * caches[i]["k_scales"][kvh].astype(np.float64)[:, None]
            vf = caches[i]["v_codes"][kvh].astype(np.float64) * caches[i]["v_scales"][kvh].astype(np.float64)[:, None]
            heads = range(kvh * rep, (kvh + 1) * rep)
            ref = np.stack([oracle.softmax_attention(inter["q_rot"][i, h], kf, vf, 1.0 / np.sqrt(d)) for h in heads])
            ref = oracle.round_bf16(oracle.rotate(ref, SH.had_block))
            got = inter["o"][i].reshape(SH.n_q_heads, d)[kvh * rep:(kvh + 1) * rep]
            assert_close(got, ref, f"o seq {i} kv-head {kvh}", rel=1e-3, flip=True)

    # O + residual, gate/up + SwiGLU, down + residual: sampled output rows
    wo = _dq(w["wo"], None, ROWS_H)
    assert_close(inter["h"][:, ROWS_H], oracle.round_bf16(xf[:, ROWS_H] + inter["o"] @ wo.T), "h",
                 rel=STAGE_REL, flip=True)
    r2 = oracle.rms_factor(inter["h"], SH.rms_eps)[:, None]
    g = r2 * (inter["h"] @ _dq(w["wgate"], w["g_mlp"], ROWS_I).T)
    u = r2 * (inter["h"] @ _dq(w["wup"], w["g_mlp"], ROWS_I).T)
    assert_close(inter["a"][:, ROWS_I], oracle.round_bf16(oracle.silu(g) * u), "a", rel=STAGE_REL, flip=True)
    wd = _dq(w["wdown"], None, ROWS_H)
    assert_close(y[:, ROWS_H], oracle.round_bf16(inter["h"][:, ROWS_H] + inter["a"] @ wd.T), "y",
                 rel=STAGE_REL, flip=True)
    assert futr.futr_check(gpu.ws, gpu.kv) == 0
