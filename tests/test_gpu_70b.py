"""70B-shaped block (hidden 8192, 64/8 heads, SwiGLU 28672) at full size,
batch 1, 8 and 32 with 2048 cached positions: the CUDA path runs the whole
block; the oracle checks each stage on the GPU's own input to that stage, at
every query and kv head and at one sampled output row in every 128-row block
of every projection (plus 96 random rows), since its full float64 evaluation
would need ~7 GB of dequantized weights per call.

Each bf16 output (o, h, a, y) must be the nearest rounding of the oracle's
float64 value, except at near-ties (within 2e-5 relative of a midpoint), where
the kernel's fp32 arithmetic may take the other neighbour."""
import numpy as np
import pytest

import oracle
from int4_weight_kv_w4a16_gb300 import futr, inputs
from int4_weight_kv_w4a16_gb300.inputs import LLAMA70B
from tests._gpu_helpers import GpuBlock, assert_close, assert_rounded, bits_to_f64

pytestmark = pytest.mark.gpu

SH = LLAMA70B
CTX = 2048
STAGE_REL = 3e-4
R = np.random.default_rng(70)


def _rows_every_block(n_rows: int, block: int, extra: int):
    """One random row in each block of `block` rows, plus `extra` random rows."""
    per = [b * block + int(R.integers(block)) for b in range(n_rows // block)]
    return sorted(set(per) | set(R.choice(n_rows, extra, replace=False).tolist()))


# O and down: 64 row blocks of 128 hidden rows.  gate/up: a 128-row block of
# the interleaved section holds 64 gate and 64 up rows of the same 64
# intermediate rows, so one intermediate row per 64 covers every block.
ROWS_H = _rows_every_block(SH.hidden, 128, 96)
ROWS_I = _rows_every_block(SH.inter, 64, 96)


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
    qkv_rows = _rows_every_block(SH.qkv_rows, 128, 32)
    for which, key, g, rows in ((futr.FUTR_PROJ_QKV, None, w["g_attn"], qkv_rows),
                                (futr.FUTR_PROJ_O, "wo", None, ROWS_H),
                                (futr.FUTR_PROJ_GATE, "wgate", w["g_mlp"], ROWS_I),
                                (futr.FUTR_PROJ_UP, "wup", w["g_mlp"], ROWS_I),
                                (futr.FUTR_PROJ_DOWN, "wdown", None, ROWS_H)):
        src = np.concatenate([w["wq"], w["wk"], w["wv"]]) if key is None else w[key]
        c, s = gpu.unpack(which)
        rc, rs = oracle.quantize_weight(src[rows], g, 128)
        np.testing.assert_array_equal(c[rows], rc)
        np.testing.assert_array_equal(s[rows].view(np.uint16), rs.view(np.uint16))


@pytest.mark.parametrize("batch", [1, 8, 32])
def test_decode_70b_every_block_and_head(block, batch):
    gpu, w = block
    x = inputs.activations(SH, batch, 1 + batch)
    pos = np.full(batch, CTX, np.int32)
    y = bits_to_f64(gpu.decode(x, pos))
    inter = gpu.intermediates(batch)
    xf = oracle.bf16_bits_to_float(x)
    d, rep = SH.head_dim, SH.n_q_heads // SH.n_kv_heads
    r1 = oracle.rms_factor(xf, SH.rms_eps)

    # QKV: every query head (RoPE + rotation, kept in fp32) ...
    wq = _dq(w["wq"], w["g_attn"], slice(0, SH.q_rows))
    q = oracle.rope((r1[:, None] * (xf @ wq.T)).reshape(batch, SH.n_q_heads, d), pos, SH.rope_theta)
    assert_close(inter["q_rot"], oracle.rotate(q, SH.had_block), "q_rot", rel=STAGE_REL)
    del wq, q
    # ... and the new token's codes and scales at every kv-head
    caches = [gpu.read_cache(0, i, CTX + 1) for i in range(batch)]
    wk = _dq(w["wk"], w["g_attn"], slice(0, SH.kv_rows))
    wv = _dq(w["wv"], w["g_attn"], slice(0, SH.kv_rows))
    k = oracle.rope((r1[:, None] * (xf @ wk.T)).reshape(batch, SH.n_kv_heads, d), pos, SH.rope_theta)
    v = (r1[:, None] * (xf @ wv.T)).reshape(batch, SH.n_kv_heads, d)
    kc, ks = oracle.kv_quantize(k.astype(np.float32), SH.had_block)
    vc, vs = oracle.kv_quantize(v.astype(np.float32), SH.had_block)
    for i in range(batch):
        for got, ref in ((caches[i]["k_codes"][:, CTX], kc[i]), (caches[i]["v_codes"][:, CTX], vc[i])):
            assert np.abs(got.astype(int) - ref.astype(int)).max() <= 1
            assert np.mean(got != ref) < 0.01
        for got, ref in ((caches[i]["k_scales"][:, CTX], ks[i]), (caches[i]["v_scales"][:, CTX], vs[i])):
            g64, r64 = got.astype(np.float64), ref.astype(np.float64)
            assert np.all(np.abs(g64 - r64) <= np.abs(r64) * 2.0 ** -10)

    # attention: every query head of every sequence, on the GPU's query and cache
    o_exact = np.zeros((batch, SH.n_q_heads, d))
    for i in range(batch):
        for kvh in range(SH.n_kv_heads):
            kf = caches[i]["k_codes"][kvh].astype(np.float64) * caches[i]["k_scales"][kvh].astype(np.float64)[:, None]
            vf = caches[i]["v_codes"][kvh].astype(np.float64) * caches[i]["v_scales"][kvh].astype(np.float64)[:, None]
            for h in range(kvh * rep, (kvh + 1) * rep):
                o_exact[i, h] = oracle.softmax_attention(inter["q_rot"][i, h], kf, vf, 1.0 / np.sqrt(d))
    o_exact = oracle.rotate(o_exact, SH.had_block).reshape(batch, SH.q_rows)
    assert_rounded(inter["o"], o_exact, "o")

    # O + residual, gate/up + SwiGLU, down + residual: a row of every block
    wo = _dq(w["wo"], None, ROWS_H)
    assert_rounded(inter["h"][:, ROWS_H], xf[:, ROWS_H] + inter["o"] @ wo.T, "h")
    r2 = oracle.rms_factor(inter["h"], SH.rms_eps)[:, None]
    g = r2 * (inter["h"] @ _dq(w["wgate"], w["g_mlp"], ROWS_I).T)
    u = r2 * (inter["h"] @ _dq(w["wup"], w["g_mlp"], ROWS_I).T)
    assert_rounded(inter["a"][:, ROWS_I], oracle.silu(g) * u, "a")
    wd = _dq(w["wdown"], None, ROWS_H)
    assert_rounded(y[:, ROWS_H], inter["h"][:, ROWS_H] + inter["a"] @ wd.T, "y")
    assert futr.futr_check(gpu.ws, gpu.kv) == 0
