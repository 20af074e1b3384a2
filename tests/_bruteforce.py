"""Independent brute-force restatement of the decode block for tiny shapes.

Pure Python loops, written from the definitions with formulas that differ from
the oracle's vectorised ones: Hadamard entries from (-1)^popcount(i & j), RoPE
as multiplication by a unit complex number, exact rational bf16 rounding,
struct-based fp32/fp16 rounding, explicit softmax sums.  Used only to pin the
oracle; never compared with the CUDA path directly.
"""
from __future__ import annotations

import cmath
import math
import struct
from fractions import Fraction


def f32(x: float) -> float:
    return struct.unpack("f", struct.pack("f", x))[0]


def f16(x: float) -> float:
    return struct.unpack("e", struct.pack("e", x))[0]


def bf16(x: float) -> float:
    """Exact round-half-even to 8 significant bits."""
    if x == 0:
        return 0.0
    fx = Fraction(x)
    e = math.floor(math.log2(abs(x)))
    while Fraction(2) ** e > abs(fx):
        e -= 1
    while Fraction(2) ** (e + 1) <= abs(fx):
        e += 1
    q = Fraction(2) ** (max(e, -126) - 7)
    return float(round(fx / q) * q)


def had(i: int, j: int) -> int:
    return -1 if bin(i & j).count("1") % 2 else 1


def rotate(v, n):
    d = len(v)
    out = []
    for blk in range(d // n):
        for i in range(n):
            acc = 0.0
            for j in range(n):
                acc += had(i, j) * v[blk * n + j]
            out.append(acc / math.sqrt(n))
    return out


def fwht_f32(v, n):
    """fp32 butterflies, stage s pairs i (bit s clear) with i + 2^s."""
    w = [f32(a) for a in v]
    d = len(w)
    for blk in range(d // n):
        h = 1
        while h < n:
            for i in range(n):
                if i & h == 0:
                    a, b = w[blk * n + i], w[blk * n + i + h]
                    w[blk * n + i], w[blk * n + i + h] = f32(a + b), f32(a - b)
            h *= 2
    c = f32(1.0 / math.sqrt(n))
    return [f32(a * c) for a in w]


def quant(v):
    a = max(abs(f32(x)) for x in v)
    q7 = f32(a / 7.0)
    s = f16(min(q7, 65504.0))
    if s == 0:
        return [0] * len(v), 0.0
    return [max(-8, min(7, round(f32(f32(x) / s)))) for x in v], s


def rope(v, pos, theta):
    d = len(v)
    half = d // 2
    out = [0.0] * d
    for i in range(half):
        z = complex(v[i], v[i + half]) * cmath.exp(1j * pos * theta ** (-2.0 * i / d))
        out[i], out[i + half] = z.real, z.imag
    return out


def matvec(w, x):
    return [sum(w[r][c] * x[c] for c in range(len(x))) for r in range(len(w))]


def rms(x, eps):
    return 1.0 / math.sqrt(sum(a * a for a in x) / len(x) + eps)


def block(x, w, cache, pos, sh):
    """x: list of floats (one sequence); w: dict of dequantized matrices as
    lists of rows; cache: dict 'k','v' -> [Hkv][L][d] dequantized floats (old
    tokens only); pos: int.  Returns dict of stage outputs."""
    Hq, Hkv, d, n = sh.n_q_heads, sh.n_kv_heads, sh.head_dim, sh.had_block
    r = rms(x, sh.rms_eps)
    qkv = [r * a for a in matvec(w["qkv"], x)]
    q = [qkv[h * d:(h + 1) * d] for h in range(Hq)]
    k = [qkv[(Hq + h) * d:(Hq + h + 1) * d] for h in range(Hkv)]
    v = [qkv[(Hq + Hkv + h) * d:(Hq + Hkv + h + 1) * d] for h in range(Hkv)]
    q = [rope(a, pos, sh.rope_theta) for a in q]
    k = [rope(a, pos, sh.rope_theta) for a in k]
    q_rot = [rotate(qh, n) for qh in q]
    k_new = [quant(fwht_f32(kh, n)) for kh in k]
    v_new = [quant(fwht_f32(vh, n)) for vh in v]
    o = []
    for h in range(Hq):
        kv = h * Hkv // Hq
        keys = [list(t) for t in cache["k"][kv]] + [[c * k_new[kv][1] for c in k_new[kv][0]]]
        vals = [list(t) for t in cache["v"][kv]] + [[c * v_new[kv][1] for c in v_new[kv][0]]]
        sc = [sum(q_rot[h][i] * key[i] for i in range(d)) / math.sqrt(d) for key in keys]
        mx = max(sc)
        e = [math.exp(s - mx) for s in sc]
        z = sum(e)
        oh = [sum(e[j] * vals[j][i] for j in range(len(vals))) / z for i in range(d)]
        o.extend(bf16(a) for a in rotate(oh, n))
    hres = [bf16(a + b) for a, b in zip(x, matvec(w["o"], o))]
    r2 = rms(hres, sh.rms_eps)
    g = [r2 * a for a in matvec(w["gate"], hres)]
    u = [r2 * a for a in matvec(w["up"], hres)]
    act = [bf16(gg / (1.0 + math.exp(-gg)) * uu) for gg, uu in zip(g, u)]
    y = [bf16(a + b) for a, b in zip(hres, matvec(w["down"], act))]
    return {"q_rot": q_rot, "k_new": k_new, "v_new": v_new, "o": o, "h": hres, "a": act, "y": y}


def code(x: float, s: float) -> int:
    """The INT4 code of x under scale s (0 when s == 0)."""
    if s == 0:
        return 0
    return max(-8, min(7, round(f32(f32(x) / s))))


def gptq_row(w, h, group, damp):
    """GPTQ of one weight row by its least-squares definition: after columns
    0..j-1 are fixed to their quantized values, the remaining weights are the
    minimizers of (w - v) H (w - v)^T over v with the fixed part held, i.e.
    v_R = w_R + H_RR^-1 H_RF (w_F - q_F), solved afresh at every column; column
    j is then quantized from v_j.  Same dead-input and dampening rules as the
    published algorithm.  numpy is used for the linear solves only."""
    import numpy as np
    k = len(w)
    hh = np.array(h, dtype=np.float64, copy=True)
    w = np.array([f32(a) for a in w], dtype=np.float64)
    for j in range(k):
        if hh[j, j] == 0:
            hh[j, j] = 1.0
            w[j] = 0.0
    mean_diag = sum(hh[j, j] for j in range(k)) / k
    for j in range(k):
        hh[j, j] += damp * mean_diag
    q = []
    codes, scales = [], []
    s = 0.0
    for j in range(k):
        fixed, rest = list(range(j)), list(range(j, k))
        v = w[rest].copy()
        if fixed:
            delta = w[fixed] - np.array(q)
            v += np.linalg.solve(hh[np.ix_(rest, rest)], hh[np.ix_(rest, fixed)] @ delta)
        if j % group == 0:
            s = quant(list(v[:group]))[1]
            scales.append(s)
        c = code(float(v[0]), s)
        codes.append(c)
        q.append(c * s)
    return codes, scales
