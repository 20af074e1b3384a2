"""Plain, slow CPU oracle for the INT4 decode step of a Llama-style block.

TEST INFRASTRUCTURE.  Only the test-suite, the package smoke check and the
benchmark's CPU-baseline leg may import this module.  It shares no code with
the CUDA path and imports nothing from it; both sides only consume the same
seeded inputs.

Sources (cited by title and section):
  [ABS] "FuTransformer: FP8 prefill and INT4 decode for Llama-style inference
        on Hopper" -- the paper's abstract.
  [EN]  "FP8 Prefill + INT4 Decode: New Optimization for Llama Inference on
        Hopper" -- sections "FP8 Prefill: fusing GEMM and epilogue all the way",
        "INT4 Decode: letting dequantization feed directly into MMA operands",
        and the paragraph on the Hadamard transform.

Precision.  Everything is float64 except the two quantizers, whose rounding is
fixed exactly: scale = fp16(absmax / 7) with the division in fp32, codes =
round-half-to-even of the fp32 quotient x / fp16 scale, clamped to [-8, 7].
The fp32 Hadamard butterflies that feed the KV quantizer are emulated in fp32
in a fixed stage order.  The block evaluation rounds only where the block's
activations are stored in bf16 between stages: the attention output o, the
residual stream h, the SwiGLU activation a and the block output y.  The rotated
query is kept at full precision.

Readings of points the pages leave open (the plainest one each time):
  * RMSNorm: r = 1/sqrt(mean(x^2) + eps), eps = 1e-5; the gain g_attn is folded
    into Wq, Wk, Wv and g_mlp into Wgate, Wup; Wo and Wdown get no gain.
  * RoPE: Llama rotate-half convention, theta = 500000, inv_freq_i =
    theta^(-2i/d), angle = pos * inv_freq_i, applied to q and the new k before
    the Hadamard rotation.  Cached keys are stored post-RoPE.
  * Hadamard: Sylvester order, orthonormal (1/sqrt(n) on every rotation), block
    diagonal along head_dim in blocks of n.  Keys, values and the query are
    rotated; the attention output is rotated back with the same matrix.
  * GQA: query head h reads kv-head h // (n_q_heads / n_kv_heads).
  * pos[b] is the number of tokens already cached; the new token goes to slot
    pos[b] and attention spans positions 0..pos[b].
  * Full decode step (embedding, the blocks, final RMSNorm, LM head): the LM
    head stays bf16 (no INT4 projection follows the final norm, so its gain
    cannot be folded into INT4 codes).  The final gain multiplies the last
    block's output in fp32 and the product is rounded once to bf16, the LM
    head's activation; the RMSNorm factor r (float64 here) scales the logits.
  * GPTQ in the same INT4 format ([ABS]): the same INT4 codes and one fp16
    scale per (output row, 128 inputs), chosen by the published GPTQ column sweep
    (natural column order, 1 % dampening, upper Cholesky factor of the inverse
    Hessian).  Each group's scale follows the rule of the round-to-nearest
    quantizer, applied to the group's error-compensated weights when the sweep
    reaches the group's first column.  The Hessian is that of the normalized
    input the gain-folded weight multiplies.  The sweep's working weights are
    float64; every code and scale decision is taken on their fp32 rounding.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

# ----------------------------------------------------------------------------
# narrow-type rounding (own implementations)
# ----------------------------------------------------------------------------


def round_bf16(x) -> np.ndarray:
    """Round real values to the nearest bf16 value (ties to even), returned as
    float64.  bf16 keeps 8 significant bits and fp32's exponent range."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)                  # subnormal spacing 2^-133
    ulp = np.ldexp(1.0, e - 8)
    return np.rint(x / ulp) * ulp


def round_fp16(x) -> np.ndarray:
    """Round to the nearest IEEE binary16 value (ties to even), as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def bf16_bits_to_float(u) -> np.ndarray:
    """Decode bf16 bit patterns (uint16) to float64."""
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Hadamard rotation  [EN] Hadamard paragraph; [ABS] (a block-diagonal Hadamard
# rotation lowers the cache's quantization error from outlier channels)
# ----------------------------------------------------------------------------


def hadamard(n: int) -> np.ndarray:
    """Sylvester Hadamard matrix: H_1 = [1], H_2m = [[H_m, H_m], [H_m, -H_m]]."""
    assert n >= 1 and (n & (n - 1)) == 0, "Hadamard order must be a power of two"
    h = np.ones((1, 1), dtype=np.int64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def rotate(v: np.ndarray, n: int) -> np.ndarray:
    """Block-diagonal orthonormal rotation along the last axis, float64:
    each contiguous block of n entries x becomes H_n x / sqrt(n)."""
    v = np.asarray(v, dtype=np.float64)
    d = v.shape[-1]
    assert d % n == 0
    blocks = v.reshape(v.shape[:-1] + (d // n, n))
    out = blocks @ hadamard(n).T.astype(np.float64) / math.sqrt(n)
    return out.reshape(v.shape)


def fwht_f32(v: np.ndarray, n: int) -> np.ndarray:
    """The rotation computed in fp32 as the KV quantizer's input.

    Fast Walsh-Hadamard transform on each block of n entries: stages
    s = 0 .. log2(n)-1, stage s pairs entry i (bit s of i clear) with entry
    i + 2^s and replaces them by (a + b, a - b), every sum rounded to fp32.
    The transformed block is multiplied once by float32(1/sqrt(n)).
    """
    v = np.array(v, dtype=np.float32, copy=True)
    d = v.shape[-1]
    assert d % n == 0 and (n & (n - 1)) == 0
    lead = v.shape[:-1]
    w = v.reshape(lead + (d // n, n))
    h = 1
    while h < n:
        w = w.reshape(lead + (d // n, n // (2 * h), 2, h))
        a = w[..., 0, :]
        b = w[..., 1, :]
        w = np.stack([a + b, a - b], axis=-2)
        h *= 2
    w = w.reshape(lead + (d,))
    return w * np.float32(1.0 / math.sqrt(n))


# ----------------------------------------------------------------------------
# INT4 round-to-nearest quantizer  [ABS] (INT4 projection weights rounded to
# nearest; the INT4 cache copy); [EN] INT4 Decode section
# ----------------------------------------------------------------------------

FP16_MAX = 65504.0


def rtn_scale(v32: np.ndarray) -> np.ndarray:
    """The scale of each vector along the last axis: a = max |v| (exact),
    s = fp16(a / 7) with the division in fp32 (a quotient above the fp16 range
    saturates to 65504).  Returns float16 [...]."""
    v = np.asarray(v32, dtype=np.float32)
    a = np.max(np.abs(v), axis=-1)
    q7 = (a / np.float32(7.0)).astype(np.float32)
    return np.minimum(q7, np.float32(FP16_MAX)).astype(np.float16)


def rtn_codes(v32: np.ndarray, s16: np.ndarray) -> np.ndarray:
    """Codes of each vector along the last axis under its scale s:
    clamp(rint(v / s), -8, 7) with v / s an fp32 division and rint
    ties-to-even; s == 0 gives all-zero codes.  Returns int8 [..., n]."""
    v = np.asarray(v32, dtype=np.float32)
    s32 = np.asarray(s16, dtype=np.float16).astype(np.float32)[..., None]
    safe = np.where(s32 > 0, s32, np.float32(1.0))
    q = (v / safe).astype(np.float32)
    return np.where(s32 > 0, np.clip(np.rint(q), -8, 7), 0).astype(np.int8)


def quant_rtn(v32: np.ndarray):
    """Quantize each vector along the last axis to signed INT4 with one fp16
    scale: s = ``rtn_scale(v)``, codes = ``rtn_codes(v, s)``.  Returns
    (codes int8, scales float16)."""
    s16 = rtn_scale(v32)
    return rtn_codes(v32, s16), s16


def dequant(codes: np.ndarray, scales: np.ndarray, group: int) -> np.ndarray:
    """float64 value of INT4 codes [.., K] with one scale per `group` entries."""
    c = np.asarray(codes, dtype=np.float64)
    s = np.asarray(scales, dtype=np.float64)
    k = c.shape[-1]
    cg = c.reshape(c.shape[:-1] + (k // group, group))
    return (cg * s[..., None]).reshape(c.shape)


# ----------------------------------------------------------------------------
# offline weight packing  [ABS] (the fixed RMSNorm gain folded into the
# weights; INT4 projection weights rounded to nearest)
# ----------------------------------------------------------------------------


def fold_gain(w: np.ndarray, g: Optional[np.ndarray]) -> np.ndarray:
    """W' = W diag(g): column j of the [out, in] weight times g_j, one fp32 rounding."""
    w = np.asarray(w, dtype=np.float32)
    if g is None:
        return w.copy()
    return (w * np.asarray(g, dtype=np.float32)[None, :]).astype(np.float32)


def quantize_weight(w: np.ndarray, g: Optional[np.ndarray], group: int = 128):
    """Fold the gain, then INT4-RTN per (output row, `group` inputs).
    Returns codes int8 [out, in] and fp16 scales [out, in/group]."""
    wf = fold_gain(w, g)
    n, k = wf.shape
    assert k % group == 0
    c, s = quant_rtn(wf.reshape(n, k // group, group))
    return c.reshape(n, k), s


def pack_block(weights: Dict[str, np.ndarray], group: int = 128) -> Dict[str, tuple]:
    """Quantize the seven projections of one block.

    Canonical result: 'qkv' (rows Wq; Wk; Wv, gain g_attn), 'o' (no gain),
    'gate', 'up' (gain g_mlp), 'down' (no gain): each (codes, scales).
    """
    ga, gm = weights["g_attn"], weights["g_mlp"]
    wqkv = np.concatenate([weights["wq"], weights["wk"], weights["wv"]], axis=0)
    return {
        "qkv": quantize_weight(wqkv, ga, group),
        "o": quantize_weight(weights["wo"], None, group),
        "gate": quantize_weight(weights["wgate"], gm, group),
        "up": quantize_weight(weights["wup"], gm, group),
        "down": quantize_weight(weights["wdown"], None, group),
    }


def dequant_block(packed: Dict[str, tuple], group: int = 128) -> Dict[str, np.ndarray]:
    return {k: dequant(c, s, group) for k, (c, s) in packed.items()}


# ----------------------------------------------------------------------------
# GPTQ in the same INT4 format  [ABS] (GPTQ codes in the round-to-nearest
# format); [EN] accuracy section, paragraph on GPTQ (calibration data,
# approximate second-order information).
# The pages name the method only; its steps here are those of the published
# GPTQ algorithm (Frantar et al., "GPTQ: Accurate Post-Training Quantization
# for Generative Pre-trained Transformers", 2022), without activation reordering.
# ----------------------------------------------------------------------------


def gptq_hessian(xcal: np.ndarray) -> np.ndarray:
    """H = (2/n) X^T X for n calibration inputs X [n, K] (float64): the Hessian,
    with respect to each row of the quantized weight, of the mean squared
    output error (1/n) sum_i ||(W - Q) x_i||^2."""
    x = np.asarray(xcal, dtype=np.float64)
    return (2.0 / x.shape[0]) * (x.T @ x)


def gptq_quantize(w32: np.ndarray, h: np.ndarray, group: int = 128, damp: float = 0.01):
    """Quantize W [N, K] (fp32) to the format of ``quantize_weight``, choosing
    the codes by GPTQ under the input Hessian h [K, K].

    1. An input that is zero in all calibration data (H_jj = 0) gets H_jj = 1,
       and its weight column is set to 0.
    2. Dampening: H += damp * mean(diag H) * I.
    3. U = the upper Cholesky factor of H^-1 (H^-1 = U^T U).
    4. Columns j = 0 .. K-1 in order, on a float64 working copy of W:
       at the first column of each group of `group` inputs the group's scales
       are ``rtn_scale`` of the group's current weights (in fp32);
       column j's codes are ``rtn_codes`` of its current weights (in fp32)
       under those scales; its error e = (w_j - c_j s) / U_jj is spread over
       the columns not yet quantized, W[:, j+1:] -= e U[j, j+1:].
    With a diagonal H no error is spread and the result is the round-to-nearest
    quantizer's.  Returns codes int8 [N, K] and fp16 scales [N, K/group]."""
    w = np.array(w32, dtype=np.float32).astype(np.float64)
    n, k = w.shape
    assert k % group == 0 and h.shape == (k, k)
    hh = np.array(h, dtype=np.float64, copy=True)
    dead = np.diag(hh) == 0
    hh[dead, dead] = 1.0
    w[:, dead] = 0.0
    hh[np.diag_indices(k)] += damp * np.mean(np.diag(hh))
    u = np.linalg.cholesky(np.linalg.inv(hh)).T
    codes = np.zeros((n, k), dtype=np.int8)
    scales = np.zeros((n, k // group), dtype=np.float16)
    for j in range(k):
        gi = j // group
        if j % group == 0:
            scales[:, gi] = rtn_scale(w[:, j:j + group].astype(np.float32))
        c = rtn_codes(w[:, j:j + 1].astype(np.float32), scales[:, gi])[:, 0]
        codes[:, j] = c
        e = (w[:, j] - c * scales[:, gi].astype(np.float64)) / u[j, j]
        w[:, j + 1:] -= np.outer(e, u[j, j + 1:])
    return codes, scales


def gptq_quantize_weight(w: np.ndarray, g: Optional[np.ndarray], h: np.ndarray, group: int = 128,
                         damp: float = 0.01):
    """Fold the gain (W' = W diag(g), one fp32 rounding), then ``gptq_quantize``
    with the Hessian of the normalized input the folded weight multiplies."""
    return gptq_quantize(fold_gain(w, g), h, group, damp)


def pack_block_gptq(weights: Dict[str, np.ndarray], hessians: Dict[str, np.ndarray], group: int = 128,
                    damp: float = 0.01) -> Dict[str, tuple]:
    """``pack_block`` with GPTQ codes.  hessians: 'attn' [H, H] of the normalized
    block input (QKV), 'o' [Hq*d, Hq*d] of the attention output, 'mlp' [H, H] of
    the normalized residual (gate and up), 'down' [I, I] of the SwiGLU output."""
    ga, gm = weights["g_attn"], weights["g_mlp"]
    wqkv = np.concatenate([weights["wq"], weights["wk"], weights["wv"]], axis=0)
    return {
        "qkv": gptq_quantize_weight(wqkv, ga, hessians["attn"], group, damp),
        "o": gptq_quantize_weight(weights["wo"], None, hessians["o"], group, damp),
        "gate": gptq_quantize_weight(weights["wgate"], gm, hessians["mlp"], group, damp),
        "up": gptq_quantize_weight(weights["wup"], gm, hessians["mlp"], group, damp),
        "down": gptq_quantize_weight(weights["wdown"], None, hessians["down"], group, damp),
    }


# ----------------------------------------------------------------------------
# KV cache copy  [ABS] (the INT4 cache copy and its block-diagonal Hadamard
# rotation)
# ----------------------------------------------------------------------------


def kv_quantize(kv32: np.ndarray, had_block: int):
    """Rotate each head vector (last axis, fp32 FWHT) and INT4-quantize it with
    one fp16 scale per vector (per token, per kv-head)."""
    return quant_rtn(fwht_f32(kv32, had_block))


# ----------------------------------------------------------------------------
# rotary position embedding (Llama convention; not described on the pages)
# ----------------------------------------------------------------------------


def rope(v: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE.  v: [b, heads, d] float64; pos: [b] integer positions."""
    v = np.asarray(v, dtype=np.float64)
    d = v.shape[-1]
    half = d // 2
    inv = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / d)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = v[..., :half], v[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------


def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Single-query attention by the definition: q [d], k, v [L, d] (float64)."""
    s = (k @ q) * scale
    p = np.exp(s - np.max(s))
    return (p @ v) / np.sum(p)


def online_softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                             chunk: int) -> np.ndarray:
    """The same attention computed chunk by chunk with a running max m, running
    normalizer l and unnormalized output o, merged by the log-sum-exp rule
    (the split-context form a decode kernel uses)."""
    parts = []
    for c0 in range(0, k.shape[0], chunk):
        kc, vc = k[c0:c0 + chunk], v[c0:c0 + chunk]
        m, l, o = -np.inf, 0.0, np.zeros(v.shape[1])
        for j in range(kc.shape[0]):
            sj = float(kc[j] @ q) * scale
            mn = max(m, sj)
            corr = math.exp(m - mn) if m != -np.inf else 0.0
            pj = math.exp(sj - mn)
            l = l * corr + pj
            o = o * corr + pj * vc[j]
            m = mn
        parts.append((m, l, o))
    M = max(p[0] for p in parts)
    L = sum(p[1] * math.exp(p[0] - M) for p in parts)
    O = sum(p[2] * math.exp(p[0] - M) for p in parts)
    return O / L


# ----------------------------------------------------------------------------
# the decode block, stage by stage  [ABS] (decode on INT4 projection weights
# and the INT4 cache copy; the kernels are checked against a reference that
# computes on the quantized values) -- evaluated here on the identical
# dequantized values.
# ----------------------------------------------------------------------------


def rms_factor(x: np.ndarray, eps: float) -> np.ndarray:
    """r_b = 1/sqrt(mean_j x_bj^2 + eps) for each row b."""
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / np.sqrt(np.mean(x * x, axis=-1) + eps)


def stage_qkv(x: np.ndarray, wqkv: np.ndarray, pos: np.ndarray, shape) -> Dict[str, np.ndarray]:
    """RMSNorm (gain already folded), fused QKV projection, RoPE, query rotation.

    x: [b, H] float64 (bf16 values); wqkv: dequantized [q_rows + 2 kv_rows, H].
    Returns q_rot [b, Hq, d], k_new, v_new [b, Hkv, d] (float64, k post-RoPE,
    both before rotation)."""
    b = x.shape[0]
    Hq, Hkv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    r = rms_factor(x, shape.rms_eps)
    qkv = r[:, None] * (x @ wqkv.T)
    q = qkv[:, :Hq * d].reshape(b, Hq, d)
    k = qkv[:, Hq * d:(Hq + Hkv) * d].reshape(b, Hkv, d)
    v = qkv[:, (Hq + Hkv) * d:].reshape(b, Hkv, d)
    q = rope(q, pos, shape.rope_theta)
    k = rope(k, pos, shape.rope_theta)
    q_rot = rotate(q, shape.had_block)
    return {"q_rot": q_rot, "k_new": k, "v_new": v}


def stage_attention(q_rot: np.ndarray, k_cache: Sequence[np.ndarray], v_cache: Sequence[np.ndarray],
                    shape, rnd=None) -> np.ndarray:
    """Single-query GQA attention over the rotated, dequantized cache.

    q_rot [b, Hq, d]; k_cache[b], v_cache[b]: [Hkv, L_b, d] (rotated, dequantized,
    the new token included).  The output of every head is rotated back and
    rounded to bf16: o [b, Hq * d].  `rnd` replaces the bf16 rounding
    (default round_bf16) for callers that choose among tied roundings."""
    b = q_rot.shape[0]
    Hq, Hkv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    rep = Hq // Hkv
    o = np.zeros((b, Hq, d))
    for i in range(b):
        for h in range(Hq):
            kv = h // rep
            o[i, h] = softmax_attention(q_rot[i, h], k_cache[i][kv], v_cache[i][kv], 1.0 / math.sqrt(d))
    o = rotate(o, shape.had_block)
    return (rnd or round_bf16)(o.reshape(b, Hq * d))


def stage_o(x: np.ndarray, o: np.ndarray, wo: np.ndarray, rnd=None) -> np.ndarray:
    """h = bf16(x + Wo o)."""
    return (rnd or round_bf16)(x + o @ wo.T)


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def stage_mlp_in(h: np.ndarray, wgate: np.ndarray, wup: np.ndarray, eps: float, rnd=None) -> np.ndarray:
    """RMSNorm (gain folded), gate/up projections, SwiGLU: a = bf16(silu(g) * u)."""
    r = rms_factor(h, eps)[:, None]
    g = r * (h @ wgate.T)
    u = r * (h @ wup.T)
    return (rnd or round_bf16)(silu(g) * u)


def stage_down(h: np.ndarray, a: np.ndarray, wdown: np.ndarray, rnd=None) -> np.ndarray:
    """y = bf16(h + Wdown a)."""
    return (rnd or round_bf16)(h + a @ wdown.T)


def new_kv_codes(k_new: np.ndarray, v_new: np.ndarray, shape):
    """INT4 cache entries of the new token: fp32 input to the rotation+quantizer."""
    kc, ks = kv_quantize(k_new.astype(np.float32), shape.had_block)
    vc, vs = kv_quantize(v_new.astype(np.float32), shape.had_block)
    return kc, ks, vc, vs


def decode_block(x_bits: np.ndarray, wdq: Dict[str, np.ndarray], cache: Sequence[dict], pos: np.ndarray,
                 shape, new_kv: Optional[tuple] = None) -> Dict[str, np.ndarray]:
    """One decode step of the block for every sequence of the batch.

    x_bits: bf16 bits [b, H].  wdq: dequantized projections (``dequant_block``).
    cache[b]: dict with INT4 'k_codes', 'v_codes' [Hkv, >=pos_b, d] and fp16
    'k_scales', 'v_scales' [Hkv, >=pos_b] for the tokens already cached.
    new_kv: optional (k_codes, k_scales, v_codes, v_scales) [b, Hkv, (d)] to use
    for the new token instead of this oracle's own quantization of it.
    Returns every stage's output."""
    x = bf16_bits_to_float(x_bits)
    b = x.shape[0]
    Hkv, d = shape.n_kv_heads, shape.head_dim
    qkv = stage_qkv(x, wdq["qkv"], pos, shape)
    own = new_kv_codes(qkv["k_new"], qkv["v_new"], shape)
    kc, ks, vc, vs = own if new_kv is None else new_kv
    kfull, vfull = [], []
    for i in range(b):
        L = int(pos[i])
        kcodes = np.concatenate([np.asarray(cache[i]["k_codes"])[:, :L], np.asarray(kc)[i][:, None]], axis=1)
        kscal = np.concatenate([np.asarray(cache[i]["k_scales"])[:, :L], np.asarray(ks)[i][:, None]], axis=1)
        vcodes = np.concatenate([np.asarray(cache[i]["v_codes"])[:, :L], np.asarray(vc)[i][:, None]], axis=1)
        vscal = np.concatenate([np.asarray(cache[i]["v_scales"])[:, :L], np.asarray(vs)[i][:, None]], axis=1)
        kfull.append(kcodes.astype(np.float64) * kscal.astype(np.float64)[..., None])
        vfull.append(vcodes.astype(np.float64) * vscal.astype(np.float64)[..., None])
    o = stage_attention(qkv["q_rot"], kfull, vfull, shape)
    h = stage_o(x, o, wdq["o"])
    a = stage_mlp_in(h, wdq["gate"], wdq["up"], shape.rms_eps)
    y = stage_down(h, a, wdq["down"])
    return {"q_rot": qkv["q_rot"], "k_new": qkv["k_new"], "v_new": qkv["v_new"],
            "k_codes": own[0], "k_scales": own[1], "v_codes": own[2], "v_scales": own[3],
            "o": o, "h": h, "a": a, "y": y}


def build_cache(kv_hist: Sequence[tuple], shape) -> List[dict]:
    """Quantize bf16 K/V histories ([Hkv, L, d] bits each) into INT4 cache entries."""
    out = []
    for kb, vb in kv_hist:
        k32 = bf16_bits_to_float(kb).astype(np.float32)
        v32 = bf16_bits_to_float(vb).astype(np.float32)
        kc, ks = kv_quantize(k32, shape.had_block)
        vc, vs = kv_quantize(v32, shape.had_block)
        out.append({"k_codes": kc, "k_scales": ks, "v_codes": vc, "v_scales": vs})
    return out


# ----------------------------------------------------------- full decode step

def float_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of values that are already exactly bf16."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    assert np.array_equal(f.astype(np.float64), np.asarray(x, dtype=np.float64)), "not bf16-exact"
    u = f.view(np.uint32)
    assert not np.any(u & 0xFFFF), "not bf16-exact"
    return (u >> 16).astype(np.uint16)


def embed(tokens: np.ndarray, table_bits: np.ndarray) -> np.ndarray:
    """x_b = row tokens[b] of the bf16 embedding table (bits [vocab, H]); bits."""
    return np.asarray(table_bits)[np.asarray(tokens, dtype=np.int64)]


def final_logits(y: np.ndarray, g_final: np.ndarray, w_lm_bits: np.ndarray, eps: float) -> np.ndarray:
    """Final RMSNorm + bf16 LM head: logits[b, v] = r_b * sum_k W[v, k] xg[b, k],
    r_b = 1/sqrt(mean_k y_bk^2 + eps), xg = bf16(fp32(g_k * y_bk)) (reading: the
    gain is applied in fp32 to the block output and rounded once to bf16)."""
    y = np.asarray(y, dtype=np.float64)
    r = rms_factor(y, eps)
    xg = round_bf16((y.astype(np.float32) * np.asarray(g_final, dtype=np.float32)).astype(np.float64))
    w = bf16_bits_to_float(w_lm_bits)
    return r[:, None] * (xg @ w.T)


def decode_step(tokens: np.ndarray, table_bits: np.ndarray, layers: Sequence[Dict[str, np.ndarray]],
                caches: Sequence[Sequence[dict]], pos: np.ndarray, g_final: np.ndarray, w_lm_bits: np.ndarray,
                shape, new_kv: Optional[Sequence[tuple]] = None) -> Dict[str, object]:
    """Embedding, then every block (``decode_block`` with layers[l], caches[l]),
    then ``final_logits``.  new_kv[l]: optional new-token cache entries per layer
    (as in ``decode_block``).  Returns the per-layer outputs and the logits."""
    x_bits = embed(tokens, table_bits)
    ys = []
    for l, wdq in enumerate(layers):
        out = decode_block(x_bits, wdq, caches[l], pos, shape, None if new_kv is None else new_kv[l])
        ys.append(out["y"])
        x_bits = float_to_bf16_bits(out["y"])
    return {"y": ys, "logits": final_logits(ys[-1], g_final, w_lm_bits, shape.rms_eps)}
