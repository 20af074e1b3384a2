"""Pins of the float64 oracle against what the mathematics and the method fix.

None of these compares the oracle with itself: each check uses an independent
definition (closed form, library routine, exact rational arithmetic, a pure
Python brute force with different formulas) or an invariant that a dropped
term, a wrong sign, index or transposed operand would break.
"""
import dataclasses
import math
import os
import struct

import numpy as np
import pytest
import torch

import oracle
from int4_weight_kv_w4a16_gb300 import inputs
from tests import _bruteforce as bf

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- rounding --

def test_round_bf16_matches_torch_cast():
    r = np.random.default_rng(1)
    x = np.concatenate([r.standard_normal(20000) * 10.0 ** r.integers(-30, 30, 20000),
                        [0.0, 1.0, -1.0, 1.00390625, 1.01171875, 3.0e38, 1e-40, -1e-39]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x.astype(np.float64)), ref)


def test_round_bf16_ties_to_even_exact():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1.
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3*2^-8 is halfway between 1+2^-7 and 1+2^-6: even is 1+2^-6.
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    for v in np.random.default_rng(2).standard_normal(200):
        assert oracle.round_bf16(v) == bf.bf16(float(v))


def test_round_fp16_matches_struct():
    for v in np.random.default_rng(3).standard_normal(500) * 3:
        assert oracle.round_fp16(v) == struct.unpack("e", struct.pack("e", float(v)))[0]


# ---------------------------------------------------------------- Hadamard --

@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 64, 128, 256])
def test_hadamard_orthogonal(n):
    h = oracle.hadamard(n)
    np.testing.assert_array_equal(h @ h.T, n * np.eye(n, dtype=np.int64))
    assert h.dtype.kind == "i" and set(np.unique(h)) <= {-1, 1}


@pytest.mark.parametrize("n", [2, 8, 64, 128])
def test_hadamard_entries_popcount(n):
    h = oracle.hadamard(n)
    for i in range(n):
        for j in range(n):
            assert h[i, j] == bf.had(i, j)


@pytest.mark.parametrize("n", [8, 64, 128])
def test_fwht_basis_vectors_give_columns(n):
    c = np.float32(1.0 / math.sqrt(n))
    h = oracle.hadamard(n)
    for i in range(n):
        e = np.zeros(n, dtype=np.float32)
        e[i] = 1
        np.testing.assert_array_equal(oracle.fwht_f32(e, n), (h[:, i] * c).astype(np.float32))


def test_fwht_error_bound_and_block_diagonal():
    r = np.random.default_rng(4)
    v = r.standard_normal((7, 256)).astype(np.float32)
    for n in (16, 128, 256):
        got = oracle.fwht_f32(v, n).astype(np.float64)
        ref = oracle.rotate(v.astype(np.float64), n)
        # log2(n) fp32 roundings of partial sums bounded by sum |v| per block
        bound = (math.log2(n) + 1) * 2.0 ** -24 * np.abs(v).reshape(7, -1, n).sum(-1).max() / math.sqrt(n) * 2
        assert np.abs(got - ref).max() <= bound
    # blocks do not mix: a vector supported on block 1 stays there
    w = np.zeros(256, dtype=np.float32)
    w[128:] = r.standard_normal(128)
    out = oracle.fwht_f32(w, 128)
    assert np.all(out[:128] == 0)


def test_fwht_stage_order_bit_exact_vs_pure_python():
    r = np.random.default_rng(5)
    for n, d in ((8, 16), (16, 16), (64, 64)):
        v = r.standard_normal(d).astype(np.float32) * 37
        got = oracle.fwht_f32(v, n)
        ref = np.array(bf.fwht_f32([float(a) for a in v], n), dtype=np.float32)
        np.testing.assert_array_equal(got, ref)


def test_rotation_preserves_dot_products():
    r = np.random.default_rng(6)
    q = r.standard_normal((5, 128))
    k = r.standard_normal((5, 128)) * 20
    qr, kr = oracle.rotate(q, 128), oracle.rotate(k, 128)
    np.testing.assert_allclose(np.sum(qr * kr, -1), np.sum(q * k, -1), rtol=0, atol=1e-12 * np.abs(q * k).sum())
    # orthonormal and symmetric: rotating twice is the identity
    np.testing.assert_allclose(oracle.rotate(qr, 128), q, atol=1e-12)


def test_rotation_spreads_outliers():
    # an outlier channel x20 raises the absmax/rms ratio; the rotation lowers it
    r = np.random.default_rng(7)
    k = r.standard_normal((1000, 128))
    k[:, [3, 50, 77, 120]] *= 20
    ratio = lambda a: np.mean(np.abs(a).max(-1) / np.sqrt(np.mean(a * a, -1)))
    assert ratio(oracle.rotate(k, 128)) < 0.5 * ratio(k)


# --------------------------------------------------------------- quantizer --

def _load_golden():
    cases = []
    with open(os.path.join(HERE, "golden", "quant_rtn_hand_cases.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, vals, scale, codes = [p.strip() for p in line.split("|")]
            cases.append((name, np.array([float(a) for a in vals.split()], dtype=np.float32),
                          float(scale), np.array([int(a) for a in codes.split()])))
    return cases


@pytest.mark.parametrize("case", _load_golden(), ids=lambda c: c[0])
def test_quant_rtn_golden_hand_cases(case):
    name, v, scale, codes = case
    c, s = oracle.quant_rtn(v)
    assert float(s) == scale
    np.testing.assert_array_equal(c, codes)


def test_quant_rtn_matches_struct_emulation():
    r = np.random.default_rng(8)
    for trial in range(300):
        n = int(r.integers(1, 40))
        v = (r.standard_normal(n) * 10.0 ** r.uniform(-6, 3)).astype(np.float32)
        if trial % 10 == 0:
            v[int(r.integers(n))] *= 50
        c, s = oracle.quant_rtn(v)
        rc, rs = bf.quant([float(a) for a in v])
        assert float(s) == rs
        np.testing.assert_array_equal(c, rc)


def test_quant_rtn_error_bound():
    r = np.random.default_rng(9)
    w = (r.standard_normal((64, 4, 128)) * 0.02).astype(np.float32)
    w[3, 1, 5] = 0.9  # single outlier in one group
    c, s = oracle.quant_rtn(w)
    s64 = s.astype(np.float64)[..., None]
    q = w.astype(np.float64) / s64
    assert np.abs(q).max() <= 7.5  # no clamp in play
    err = np.abs(c * s64 - w)
    assert np.all(err <= s64 / 2 * (1 + 1e-6))
    assert c.min() >= -8 and c.max() <= 7
    # the outlier's group: scale follows the outlier, small entries round to 0/+-1
    assert float(s[3, 1]) == float(np.float16(np.float32(0.9) / np.float32(7)))


def test_quant_weight_group_layout():
    # the scale of (row, group) depends only on that row's group of 128 inputs
    r = np.random.default_rng(10)
    w = (r.standard_normal((4, 512)) * 0.02).astype(np.float32)
    w[2, 300] = 5.0
    c, s = oracle.quantize_weight(w, None, 128)
    assert s.shape == (4, 4)
    assert float(s[2, 2]) == float(np.float16(np.float32(5.0) / np.float32(7)))
    others = np.delete(s.astype(np.float64).ravel(), 2 * 4 + 2)
    assert others.max() < 0.02


# ------------------------------------------------ dequantization and cache --

def test_dequant_hand_case():
    # two rows of four codes in groups of two: each value is its code times the
    # scale of its own (row, group)
    codes = np.array([[1, -8, 7, 0], [3, 3, -1, 2]], np.int8)
    scales = np.array([[0.5, 2.0], [0.25, 4.0]], np.float16)
    np.testing.assert_array_equal(oracle.dequant(codes, scales, 2),
                                  [[0.5, -4.0, 14.0, 0.0], [0.75, 0.75, -4.0, 8.0]])


def test_dequant_block_roundtrip_within_half_scale():
    """|dequant(pack(W)) - W diag(g)| <= s/2 with s = fp16(absmax/7) of the
    element's own (row, 128-input group).  The magnitudes differ by powers of
    ten between neighbouring rows and groups, so a scale applied to another
    row or group, or a gain folded into the wrong projection, breaks the bound
    by orders of magnitude.  The bound is taken from the group's absmax, not
    from the packed scales."""
    sh = oracle_shape_tiny(hidden=256, inter=256, head_dim=32, had_block=32, group=128)
    r = np.random.default_rng(18)

    def mk(o, i):
        mag = 10.0 ** (np.arange(o)[:, None] % 3 + 2 * (np.arange(i)[None, :] // 128) - 2)
        return (r.standard_normal((o, i)) * mag).astype(np.float32)

    w = {"wq": mk(sh.q_rows, 256), "wk": mk(sh.kv_rows, 256), "wv": mk(sh.kv_rows, 256),
         "wo": mk(256, sh.q_rows), "wgate": mk(256, 256), "wup": mk(256, 256), "wdown": mk(256, 256),
         "g_attn": r.uniform(0.5, 1.5, 256).astype(np.float32),
         "g_mlp": r.uniform(0.5, 1.5, 256).astype(np.float32)}
    f64 = lambda a: np.asarray(a, np.float64)
    target = {"qkv": np.concatenate([w["wq"], w["wk"], w["wv"]]) * f64(w["g_attn"]),
              "o": f64(w["wo"]), "gate": w["wgate"] * f64(w["g_mlp"]), "up": w["wup"] * f64(w["g_mlp"]),
              "down": f64(w["wdown"])}
    dq = oracle.dequant_block(oracle.pack_block(w))
    for k, t in target.items():
        n, kk = t.shape
        amax = np.abs(t.reshape(n, kk // 128, 128)).max(-1)
        half_s = np.repeat(amax / 14.0 * (1 + 2.0 ** -10), 128, axis=1)
        assert dq[k].shape == t.shape
        assert np.all(np.abs(dq[k] - t) <= half_s + 1e-6 * np.abs(t)), k


def test_build_cache_matches_bruteforce():
    # every cached token and kv-head: fp32 butterflies of the bf16 history
    # vector, then the quantizer, both by the pure-Python brute force
    sh = oracle_shape_tiny()
    r = np.random.default_rng(19)
    hist = []
    for L in (3, 0, 2):
        k = r.standard_normal((sh.n_kv_heads, L, sh.head_dim))
        k[..., 1] *= 20
        hist.append((_bf16_bits(k), _bf16_bits(r.standard_normal((sh.n_kv_heads, L, sh.head_dim)))))
    cache = oracle.build_cache(hist, sh)
    assert len(cache) == len(hist)
    for (kb, vb), c in zip(hist, cache):
        for name, bits in (("k", kb), ("v", vb)):
            vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
            assert c[name + "_codes"].shape == bits.shape
            for h in range(sh.n_kv_heads):
                for t in range(bits.shape[1]):
                    codes, s = bf.quant(bf.fwht_f32(list(vals[h, t]), sh.had_block))
                    assert float(c[name + "_scales"][h, t]) == s
                    np.testing.assert_array_equal(c[name + "_codes"][h, t], codes)


# -------------------------------------------------------------------- GPTQ --

def test_gptq_hessian_quadratic_form():
    # u^T H u is the mean squared output of the linear map u over the
    # calibration inputs, times 2
    x = inputs.calibration_inputs(24, 50, seed=20).astype(np.float64)
    h = oracle.gptq_hessian(x)
    for u in np.random.default_rng(21).standard_normal((5, 24)):
        ref = 2.0 / 50 * sum(float(xi @ u) ** 2 for xi in x)
        assert abs(float(u @ h @ u) - ref) <= 1e-12 * ref
    np.testing.assert_array_equal(h, h.T)


def test_gptq_diagonal_hessian_is_round_to_nearest():
    # uncorrelated inputs: no error is spread, every (row, group) is the
    # round-to-nearest quantizer of its own weights
    r = np.random.default_rng(22)
    w = (r.standard_normal((8, 256)) * 0.02).astype(np.float32)
    h = np.diag(r.uniform(0.1, 10.0, 256))
    c, s = oracle.gptq_quantize(w, h, 128)
    for i in range(8):
        for g in range(2):
            rc, rs = bf.quant([float(a) for a in w[i, 128 * g:128 * (g + 1)]])
            assert float(s[i, g]) == rs
            np.testing.assert_array_equal(c[i, 128 * g:128 * (g + 1)], rc)


@pytest.mark.parametrize("k,group", [(24, 8), (16, 16)])
def test_gptq_matches_least_squares_definition(k, group):
    """The sweep's codes and scales equal those of the definition: after each
    column is fixed, re-solve the least-squares problem for the columns not yet
    quantized (pure Python with numpy linear solves, no Cholesky factor).  One
    input channel is zero in all calibration data."""
    x = inputs.calibration_inputs(k, 200, seed=23 + k).astype(np.float64)
    x[:, 5] = 0.0
    h = oracle.gptq_hessian(x)
    w = (np.random.default_rng(24).standard_normal((4, k)) * 0.5).astype(np.float32)
    c, s = oracle.gptq_quantize(w, h, group)
    assert np.all(c[:, 5] == 0)
    for i in range(4):
        rc, rs = bf.gptq_row([float(a) for a in w[i]], h, group, 0.01)
        np.testing.assert_array_equal(c[i], rc)
        assert [float(a) for a in s[i]] == rs
    # with correlated inputs the sweep departs from round-to-nearest
    assert np.any(c != oracle.quantize_weight(w, None, group)[0])


def test_gptq_lowers_calibration_output_error():
    # the method's purpose: a smaller output error on the calibration inputs
    # (and on fresh inputs of the same distribution) than round-to-nearest
    k, n = 256, 1024
    xs = inputs.calibration_inputs(k, 2 * n, seed=25).astype(np.float64)
    x, held_out = xs[:n], xs[n:]
    w = (np.random.default_rng(26).standard_normal((64, k)) * 0.02).astype(np.float32)
    err = lambda q, xx: float(np.mean(np.sum(((q - w.astype(np.float64)) @ xx.T) ** 2, axis=0)))
    q_gptq = oracle.dequant(*oracle.gptq_quantize(w, oracle.gptq_hessian(x), 128), 128)
    q_rtn = oracle.dequant(*oracle.quantize_weight(w, None, 128), 128)
    assert err(q_gptq, x) < 0.7 * err(q_rtn, x)
    assert err(q_gptq, held_out) < 0.8 * err(q_rtn, held_out)


def test_pack_block_gptq_uses_each_projection_hessian():
    sh = oracle_shape_tiny(hidden=128, inter=128, head_dim=32, had_block=32, group=128)
    r = np.random.default_rng(28)
    mk = lambda o, i: (r.standard_normal((o, i)) * 0.02).astype(np.float32)
    w = {"wq": mk(sh.q_rows, 128), "wk": mk(sh.kv_rows, 128), "wv": mk(sh.kv_rows, 128),
         "wo": mk(128, sh.q_rows), "wgate": mk(128, 128), "wup": mk(128, 128), "wdown": mk(128, 128),
         "g_attn": r.uniform(0.5, 1.5, 128).astype(np.float32), "g_mlp": r.uniform(0.5, 1.5, 128).astype(np.float32)}
    diag = {k: np.diag(r.uniform(0.5, 2.0, 128)) for k in ("attn", "o", "mlp", "down")}
    rtn = oracle.pack_block(w)
    base = oracle.pack_block_gptq(w, diag)
    for k in rtn:  # diagonal Hessians: the round-to-nearest packer, gains included
        np.testing.assert_array_equal(base[k][0], rtn[k][0])
        np.testing.assert_array_equal(base[k][1], rtn[k][1])
    corr = oracle.gptq_hessian(inputs.calibration_inputs(128, 400, seed=29).astype(np.float64))
    for hk, changed in (("attn", {"qkv"}), ("o", {"o"}), ("mlp", {"gate", "up"}), ("down", {"down"})):
        p = oracle.pack_block_gptq(w, dict(diag, **{hk: corr}))
        differs = {k for k in rtn if not np.array_equal(p[k][0], rtn[k][0])}
        assert differs == changed, hk


# ------------------------------------------------------------ gain folding --

def test_gain_folding_equals_rmsnorm_then_matmul():
    r = np.random.default_rng(11)
    H, N = 256, 96
    w = (r.standard_normal((N, H)) * 0.02).astype(np.float32)
    g = r.uniform(0.5, 1.5, H).astype(np.float32)
    x = r.standard_normal((3, H))
    eps = 1e-5
    # textbook RMSNorm with gain, then the projection
    ref = np.stack([w.astype(np.float64) @ (g * xi / np.sqrt(np.mean(xi ** 2) + eps)) for xi in x])
    folded = oracle.fold_gain(w, g).astype(np.float64)
    got = oracle.rms_factor(x, eps)[:, None] * (x @ folded.T)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-6 * np.abs(ref).max())


def test_pack_block_gain_placement():
    sh = oracle_shape_tiny(hidden=128, inter=128, head_dim=32, had_block=32, group=128)
    r = np.random.default_rng(12)
    mk = lambda o, i: (r.standard_normal((o, i)) * 0.02).astype(np.float32)
    w = {"wq": mk(sh.q_rows, 128), "wk": mk(sh.kv_rows, 128), "wv": mk(sh.kv_rows, 128),
         "wo": mk(128, sh.q_rows), "wgate": mk(128, 128), "wup": mk(128, 128), "wdown": mk(128, 128),
         "g_attn": np.ones(128, np.float32), "g_mlp": np.ones(128, np.float32)}
    base = oracle.pack_block(w)
    w2 = dict(w, g_attn=np.full(128, 2.0, np.float32), g_mlp=np.full(128, 4.0, np.float32))
    p2 = oracle.pack_block(w2)
    for k, f in (("qkv", 2.0), ("gate", 4.0), ("up", 4.0), ("o", 1.0), ("down", 1.0)):
        np.testing.assert_array_equal(p2[k][0], base[k][0])
        np.testing.assert_array_equal(p2[k][1].astype(np.float64), base[k][1].astype(np.float64) * f)


# -------------------------------------------------------------------- RoPE --

def test_rope_properties_and_complex_form():
    r = np.random.default_rng(13)
    d, theta = 16, 500000.0
    q = r.standard_normal((1, 1, d))
    k = r.standard_normal((1, 1, d))
    # position 0 is the identity; norms are preserved
    np.testing.assert_allclose(oracle.rope(q, np.array([0]), theta), q, atol=0)
    for p in (1, 7, 1000, 4095):
        rq = oracle.rope(q, np.array([p]), theta)
        np.testing.assert_allclose(np.linalg.norm(rq), np.linalg.norm(q), rtol=1e-13)
        np.testing.assert_allclose(rq[0, 0], bf.rope(list(q[0, 0]), p, theta), atol=1e-12)
    # the score depends only on the position difference
    dot = lambda m, n: float(np.sum(oracle.rope(q, np.array([m]), theta) * oracle.rope(k, np.array([n]), theta)))
    assert abs(dot(10, 3) - dot(107, 100)) < 1e-10
    assert abs(dot(10, 3) - dot(3, 10)) > 1e-6


# --------------------------------------------------------------- attention --

def test_online_softmax_equals_bruteforce():
    r = np.random.default_rng(14)
    for L, chunk in ((1, 4), (5, 2), (37, 8), (100, 16), (129, 64)):
        q = r.standard_normal(16) * 3
        k = r.standard_normal((L, 16)) * 3
        v = r.standard_normal((L, 16))
        a = oracle.softmax_attention(q, k, v, 0.25)
        b = oracle.online_softmax_attention(q, k, v, 0.25, chunk)
        np.testing.assert_allclose(b, a, rtol=0, atol=1e-12)


def test_attention_uniform_and_one_hot():
    r = np.random.default_rng(15)
    v = r.standard_normal((9, 8))
    q = np.zeros(8)
    k = r.standard_normal((9, 8))
    np.testing.assert_allclose(oracle.softmax_attention(q, k, v, 1.0), v.mean(0), atol=1e-15)
    q = np.zeros(8)
    q[0] = 1.0
    k = np.zeros((9, 8))
    k[4, 0] = 1000.0
    np.testing.assert_allclose(oracle.softmax_attention(q, k, v, 1.0), v[4], atol=1e-12)


def test_rotated_attention_equals_unrotated():
    """Rotating q, K, V and rotating the output back changes nothing (exact
    arithmetic): pins the placement of the inverse rotation."""
    r = np.random.default_rng(16)
    d, n = 64, 32
    q = r.standard_normal(d)
    k = r.standard_normal((20, d)) * 2
    v = r.standard_normal((20, d))
    ref = oracle.softmax_attention(q, k, v, 0.125)
    rot = oracle.rotate(oracle.softmax_attention(oracle.rotate(q, n), oracle.rotate(k, n),
                                                 oracle.rotate(v, n), 0.125), n)
    np.testing.assert_allclose(rot, ref, atol=1e-12)


# ------------------------------------------------------------ whole block --

def oracle_shape_tiny(**kw):
    from int4_weight_kv_w4a16_gb300.inputs import BlockShape
    base = dict(hidden=16, n_q_heads=4, n_kv_heads=2, head_dim=8, inter=24, had_block=4, group=8)
    base.update(kw)
    return BlockShape(**base)


def _tiny_case(sh, b, lengths, seed):
    r = np.random.default_rng(seed)
    w = {"qkv": r.integers(-8, 8, (sh.qkv_rows, sh.hidden)) * 0.01,
         "o": r.integers(-8, 8, (sh.hidden, sh.q_rows)) * 0.02,
         "gate": r.integers(-8, 8, (sh.inter, sh.hidden)) * 0.03,
         "up": r.integers(-8, 8, (sh.inter, sh.hidden)) * 0.03,
         "down": r.integers(-8, 8, (sh.hidden, sh.inter)) * 0.02}
    x32 = r.standard_normal((b, sh.hidden)).astype(np.float32)
    import torch as _t
    xb = _t.from_numpy(x32).to(_t.bfloat16).view(_t.int16).numpy().view(np.uint16)
    cache = []
    for L in lengths:
        cache.append({"k_codes": r.integers(-8, 8, (sh.n_kv_heads, L, sh.head_dim)).astype(np.int8),
                      "k_scales": (r.uniform(0.1, 2, (sh.n_kv_heads, L))).astype(np.float16),
                      "v_codes": r.integers(-8, 8, (sh.n_kv_heads, L, sh.head_dim)).astype(np.int8),
                      "v_scales": (r.uniform(0.1, 1, (sh.n_kv_heads, L))).astype(np.float16)})
    return w, xb, cache


@pytest.mark.parametrize("lengths", [[0], [3], [5, 1, 0]])
def test_decode_block_matches_bruteforce(lengths):
    sh = oracle_shape_tiny()
    w, xb, cache = _tiny_case(sh, len(lengths), lengths, seed=17 + len(lengths))
    pos = np.array(lengths)
    out = oracle.decode_block(xb, w, cache, pos, sh)
    x = oracle.bf16_bits_to_float(xb)
    for i, L in enumerate(lengths):
        kd = [[list(cache[i]["k_codes"][h, j].astype(float) * float(cache[i]["k_scales"][h, j]))
               for j in range(L)] for h in range(sh.n_kv_heads)]
        vd = [[list(cache[i]["v_codes"][h, j].astype(float) * float(cache[i]["v_scales"][h, j]))
               for j in range(L)] for h in range(sh.n_kv_heads)]
        wl = {k: [list(row) for row in m] for k, m in w.items()}
        ref = bf.block(list(x[i]), wl, {"k": kd, "v": vd}, int(L), sh)
        np.testing.assert_allclose(out["q_rot"][i], np.array(ref["q_rot"]), atol=1e-12)
        for h in range(sh.n_kv_heads):
            np.testing.assert_array_equal(out["k_codes"][i, h], ref["k_new"][h][0])
            assert float(out["k_scales"][i, h]) == ref["k_new"][h][1]
            np.testing.assert_array_equal(out["v_codes"][i, h], ref["v_new"][h][0])
        for key in ("o", "h", "a", "y"):
            np.testing.assert_allclose(out[key][i], np.array(ref[key]), rtol=0, atol=1e-12, err_msg=key)


def test_decode_block_zero_weights_and_input():
    sh = oracle_shape_tiny()
    w, xb, cache = _tiny_case(sh, 2, [4, 2], seed=30)
    zero = {k: np.zeros_like(v) for k, v in w.items()}
    out = oracle.decode_block(np.zeros_like(xb), zero, cache, np.array([4, 2]), sh)
    assert np.all(out["y"] == 0)
    # Wo = Wdown = 0: the block is the identity on a bf16 input
    w2 = dict(w, o=np.zeros_like(w["o"]), down=np.zeros_like(w["down"]))
    out = oracle.decode_block(xb, w2, cache, np.array([4, 2]), sh)
    np.testing.assert_array_equal(out["y"], oracle.bf16_bits_to_float(xb))


def test_decode_block_batch_permutation():
    sh = oracle_shape_tiny()
    w, xb, cache = _tiny_case(sh, 3, [3, 5, 2], seed=31)
    pos = np.array([3, 5, 2])
    a = oracle.decode_block(xb, w, cache, pos, sh)
    perm = [2, 0, 1]
    b = oracle.decode_block(xb[perm], w, [cache[i] for i in perm], pos[perm], sh)
    np.testing.assert_array_equal(b["y"], a["y"][perm])


# -------------------------------------------------------- full decode step --

def _bf16_bits(x) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_embed_takes_table_rows():
    table = np.random.default_rng(40).integers(0, 2 ** 16, (37, 8)).astype(np.uint16)
    tok = np.array([5, 0, 36, 5])
    np.testing.assert_array_equal(oracle.embed(tok, table), table[[5, 0, 36, 5]])


def test_final_logits_unit_gain_is_rmsnorm_then_matmul():
    # g = 1: bf16(g * y) = y exactly, so the logits are RMSNorm(y) W^T by the
    # definition, evaluated here with explicit Python sums
    r = np.random.default_rng(41)
    H, V, b = 64, 24, 3
    y = oracle.bf16_bits_to_float(_bf16_bits(r.standard_normal((b, H))))
    wb = _bf16_bits(r.standard_normal((V, H)) * 0.05)
    w = oracle.bf16_bits_to_float(wb)
    got = oracle.final_logits(y, np.ones(H, np.float32), wb, 1e-5)
    for i in range(b):
        den = math.sqrt(sum(float(v) * float(v) for v in y[i]) / H + 1e-5)
        ref = [sum(float(w[v, k]) * float(y[i, k]) for k in range(H)) / den for v in range(V)]
        np.testing.assert_allclose(got[i], np.array(ref), rtol=1e-12, atol=1e-12)


def test_final_logits_gain_rounded_once_to_bf16():
    # a general gain: the activation is bf16(fp32(g y)); against the unrounded
    # RMSNorm(y) * g the error per logit is at most r * sum_k |W_vk| |g_k y_k| 2^-8
    r = np.random.default_rng(42)
    H, V, b = 128, 40, 2
    y = oracle.bf16_bits_to_float(_bf16_bits(r.standard_normal((b, H)) * 3))
    g = r.uniform(0.5, 1.5, H).astype(np.float32)
    wb = _bf16_bits(r.standard_normal((V, H)) * 0.05)
    w = oracle.bf16_bits_to_float(wb)
    got = oracle.final_logits(y, g, wb, 1e-5)
    rms = np.sqrt(np.mean(y * y, axis=1) + 1e-5)
    exact = ((y * g.astype(np.float64)) / rms[:, None]) @ w.T
    bound = (np.abs(y * g.astype(np.float64)) @ np.abs(w).T) / rms[:, None] * 2.0 ** -8
    assert np.all(np.abs(got - exact) <= bound + 1e-15)
    assert np.any(got != exact)  # the rounding is there


def test_final_logits_reads_rows_of_the_head():
    # one-hot rows: logit v is r * bf16(fp32(g_k y_k)) for the column k the row
    # selects; the gain differs per column and g_k y_k is not a bf16 value, so
    # a transposed head, a gain of another column, a dropped factor or an
    # activation left unrounded fails.  Rounding by the brute-force helpers.
    H = 16
    y = oracle.bf16_bits_to_float(_bf16_bits(np.arange(1, H + 1, dtype=np.float32) / 4))[None, :]
    w = np.zeros((6, H), np.float32)
    for v in range(6):
        w[v, 3 * v % H] = 1.0
    g = (1.0 + np.arange(H, dtype=np.float32) / np.float32(10.0)).astype(np.float32)
    got = oracle.final_logits(y, g, _bf16_bits(w), 1e-5)[0]
    r = 1.0 / math.sqrt(sum(float(a) ** 2 for a in y[0]) / H + 1e-5)
    act = [bf.bf16(bf.f32(float(g[k]) * float(y[0, k]))) for k in range(H)]
    assert sum(act[k] != float(g[k]) * float(y[0, k]) for k in range(H)) >= 8  # the rounding matters
    np.testing.assert_allclose(got, [r * act[3 * v % H] for v in range(6)], rtol=1e-15)


def test_decode_step_chains_the_blocks():
    sh = oracle_shape_tiny()
    w1, _, c1 = _tiny_case(sh, 2, [3, 1], seed=50)
    w2, _, c2 = _tiny_case(sh, 2, [3, 1], seed=51)
    r = np.random.default_rng(52)
    table = _bf16_bits(r.standard_normal((11, sh.hidden)))
    wlm = _bf16_bits(r.standard_normal((9, sh.hidden)) * 0.05)
    g = r.uniform(0.5, 1.5, sh.hidden).astype(np.float32)
    tok, pos = np.array([4, 10]), np.array([3, 1])
    out = oracle.decode_step(tok, table, [w1, w2], [c1, c2], pos, g, wlm, sh)
    y1 = oracle.decode_block(table[tok], w1, c1, pos, sh)["y"]
    y2 = oracle.decode_block(_bf16_bits(y1), w2, c2, pos, sh)["y"]
    np.testing.assert_array_equal(out["y"][0], y1)
    np.testing.assert_array_equal(out["y"][1], y2)
    np.testing.assert_array_equal(out["logits"], oracle.final_logits(y2, g, wlm, sh.rms_eps))
