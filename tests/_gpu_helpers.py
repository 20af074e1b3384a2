"""Shared set-up for the GPU parity tests: seeded inputs -> the CUDA path
through the C ABI, and the same inputs -> the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from int4_weight_kv_w4a16_gb300 import build, futr, inputs

# Block-output tolerance (relative L2 and max-abs relative to rms(reference)).
REL_L2 = 1e-3
MAX_ABS_RMS = 2e-2


def ensure_lib():
    build.build()
    return futr.lib()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits_to_f64(t: torch.Tensor) -> np.ndarray:
    return oracle.bf16_bits_to_float(t.cpu().numpy().view(np.uint16))


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """The spacing of bf16 values at |v| (8 significant bits): 2^(e - 7) for
    |v| in [2^e, 2^(e+1)); 0 for v = 0."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 7), 0.0)


def assert_close(got: np.ndarray, ref: np.ndarray, name: str, rel=REL_L2, mx=MAX_ABS_RMS, flip=False):
    """rel L2 <= rel and |got - ref| <= mx * rms(ref) elementwise.  flip=True
    (stage checks of bf16 outputs) also allows each element one bf16 step at
    the larger of |got| and |ref|: a value that lands within the kernel's fp32
    error of a rounding boundary may round the other way.  Such a flip of one
    large element can exceed the L2 bound of a small output by itself (one
    flip in 512 values: ~3.5e-4), so with flip=True the L2 bound may instead
    hold over the other elements while the one-step differences number at
    most max(4, n / 2000), the end-to-end check's allowance for ties."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), name
    nrm = np.linalg.norm(ref)
    err = np.linalg.norm(got - ref)
    rms = np.sqrt(np.mean(ref * ref))
    if nrm == 0:
        assert np.abs(got).max() == 0, name
        return {"rel_l2": 0.0, "max_abs_rms": 0.0}
    if flip and err / nrm > rel:
        step = bf16_ulp(np.maximum(np.abs(ref), np.abs(got))) * (1 + 1e-12)
        one = (got != ref) & (np.abs(got - ref) <= step)
        n_one = int(one.sum())
        rest = np.linalg.norm(np.where(one, 0.0, got - ref))
        assert n_one <= max(4, got.size // 2000) and rest / nrm <= rel, \
            f"{name}: rel L2 {err / nrm:.3e} > {rel} ({n_one} one-step differences, rest {rest / nrm:.3e})"
    else:
        assert err / nrm <= rel, f"{name}: rel L2 {err / nrm:.3e} > {rel}"
    allowed = mx * rms
    if flip:
        allowed = np.maximum(allowed, bf16_ulp(np.maximum(np.abs(ref), np.abs(got))) * (1 + 1e-12))
    bad = np.abs(got - ref) > allowed
    assert not np.any(bad), f"{name}: max abs {np.abs(got - ref).max():.3e} > allowed ({int(bad.sum())} elements)"
    return {"rel_l2": float(err / nrm), "max_abs_rms": float(np.abs(got - ref).max() / rms)}


def _bf16_key(v: np.ndarray) -> np.ndarray:
    """Order-preserving integer key of bf16 values (adjacent values differ by 1)."""
    bits = (np.asarray(v, dtype=np.float32).view(np.uint32) >> 16).astype(np.int64)
    mag = bits & 0x7FFF
    return np.where(bits & 0x8000, -mag, mag)


def assert_rounded(got: np.ndarray, exact: np.ndarray, name: str, tol: float = 2e-5, max_tie_frac: float = 1e-3):
    """Every bf16 value `got` is a bf16 rounding of a value within
    tol * max(|exact|, rms(exact)) of the float64 result `exact`: the kernel
    computes exact with that fp32 error and rounds it to nearest, so
    |got - exact| <= half a bf16 step + tol * scale.  For values well above
    tol * rms this admits only the nearest rounding, or its neighbour where
    exact lies that close to a midpoint; for values near zero it admits the
    kernel's absolute error.  Values other than the nearest rounding may make
    up at most max_tie_frac of the values (at least 4)."""
    import oracle
    got = np.asarray(got, dtype=np.float64)
    exact = np.asarray(exact, dtype=np.float64)
    assert got.shape == exact.shape, (name, got.shape, exact.shape)
    assert np.all(np.isfinite(got)), name
    r = oracle.round_bf16(exact)
    diff = got != r
    if not diff.any():
        return 0
    scale = np.maximum(np.abs(exact), np.sqrt(np.mean(exact * exact)))
    half_step = 0.5 * bf16_ulp(np.maximum(np.abs(got), np.abs(exact)))
    bad = diff & (np.abs(got - exact) > half_step + tol * scale)
    if bad.any():
        i = np.flatnonzero(bad)[0]
        raise AssertionError(f"{name}: {int(bad.sum())} values are not the rounding of the exact result "
                             f"(first at flat index {i}: got {got.flat[i]!r}, exact {exact.flat[i]!r}, "
                             f"nearest {r.flat[i]!r})")
    ties = int(diff.sum())
    assert ties <= max(4, int(max_tie_frac * got.size)), f"{name}: {ties} near-tie roundings of {got.size}"
    return ties


def errors(got, ref) -> dict:
    """rel L2 and max abs / rms(ref), without asserting."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nrm = np.linalg.norm(ref)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    if nrm == 0:
        return {"rel_l2": float(np.linalg.norm(got)), "max_abs_rms": float(np.abs(got).max(initial=0))}
    return {"rel_l2": float(np.linalg.norm(got - ref) / nrm), "max_abs_rms": float(np.abs(got - ref).max() / rms)}


class TieRounding:
    """bf16 rounding for the oracle chain that accepts the GPU's choice where
    both roundings are correct: the exact value lies within `tol` (relative to
    max(|value|, rms of the vector)) of the midpoint between two adjacent bf16
    values, i.e. inside the fp32 error of the fast path.  Everywhere else the
    oracle's own rounding stands."""

    def __init__(self, gpu_vals: np.ndarray, tol: float = 2e-5):
        self.gpu = np.asarray(gpu_vals, dtype=np.float64)
        self.tol = tol
        self.ties = 0

    def __call__(self, exact: np.ndarray) -> np.ndarray:
        exact = np.asarray(exact, dtype=np.float64)
        r = oracle.round_bf16(exact)
        g = self.gpu.reshape(r.shape)
        diff = g != r
        if not diff.any():
            return r
        scale = np.maximum(np.abs(exact), np.sqrt(np.mean(exact * exact)))
        near = np.abs(exact - (r + g) / 2) <= self.tol * scale
        adjacent = np.abs(_bf16_key(g) - _bf16_key(r)) == 1
        take = diff & near & adjacent
        self.ties += int(take.sum())
        return np.where(take, g, r)


def guided_chain(xf, wdq, kfull, vfull, pos, shape, inter, y_gpu):
    """The oracle's block from x on the identical dequantized weights and cache,
    where each bf16 storage point takes the GPU's rounding only at ties."""
    q = oracle.stage_qkv(xf, wdq["qkv"], pos, shape)["q_rot"]
    tr = {k: TieRounding(v) for k, v in (("o", inter["o"]), ("h", inter["h"]), ("a", inter["a"]), ("y", y_gpu))}
    o = oracle.stage_attention(q, kfull, vfull, shape, rnd=tr["o"])
    h = oracle.stage_o(xf, o, wdq["o"], rnd=tr["h"])
    a = oracle.stage_mlp_in(h, wdq["gate"], wdq["up"], shape.rms_eps, rnd=tr["a"])
    y = oracle.stage_down(h, a, wdq["down"], rnd=tr["y"])
    return y, {k: v.ties for k, v in tr.items()}


class GpuBlock:
    """One packed block + an INT4 KV cache + a workspace, on cuda:0."""

    def __init__(self, shape, weights, max_batch: int, capacity: int, n_layers: int = 1):
        ensure_lib()
        self.shape = shape
        self.cs = futr.make_shape(shape)
        self.blob = futr.alloc_bytes(futr.futr_weights_size(self.cs))
        w = {k: dev(v) for k, v in weights.items()}
        futr.futr_pack_weights(self.cs, w["wq"], w["wk"], w["wv"], w["wo"], w["wgate"], w["wup"], w["wdown"],
                               w["g_attn"], w["g_mlp"], self.blob)
        del w
        self.kv = futr.futr_kv_init(self.cs, n_layers, max_batch, capacity,
                                    futr.alloc_bytes(futr.futr_kv_size(self.cs, n_layers, max_batch, capacity)))
        self.ws = futr.futr_workspace_init(self.cs, max_batch, capacity,
                                           futr.alloc_bytes(futr.futr_workspace_size(self.cs, max_batch, capacity)))
        torch.cuda.synchronize()

    def unpack(self, which):
        sec_rows = {futr.FUTR_PROJ_QKV: (self.shape.qkv_rows, self.shape.hidden),
                    futr.FUTR_PROJ_O: (self.shape.hidden, self.shape.q_rows),
                    futr.FUTR_PROJ_GATE: (self.shape.inter, self.shape.hidden),
                    futr.FUTR_PROJ_UP: (self.shape.inter, self.shape.hidden),
                    futr.FUTR_PROJ_DOWN: (self.shape.hidden, self.shape.inter)}[which]
        r, c = sec_rows
        codes = torch.empty((r, c), dtype=torch.int8, device="cuda")
        scales = torch.empty((r, c // 128), dtype=torch.int16, device="cuda")
        futr.futr_unpack_weights(self.cs, self.blob, which, codes, scales)
        return codes.cpu().numpy(), scales.cpu().numpy().view(np.float16)

    def append(self, layer: int, seq: int, k_bits: np.ndarray, v_bits: np.ndarray, start: int):
        """Append tokens [start, start + n) of one sequence: k, v bits [Hkv, n, d]."""
        n = k_bits.shape[1]
        pos = torch.tensor([start], dtype=torch.int32, device="cuda")
        futr.futr_kv_append(self.kv, layer, seq, 1, pos, n, dev(k_bits), dev(v_bits))

    def append_history(self, layer: int, hist, chunks=None):
        for b, (kb, vb) in enumerate(hist):
            L = kb.shape[1]
            if L == 0:
                continue
            if chunks is None:
                self.append(layer, b, kb, vb, 0)
            else:
                s = 0
                for c in chunks:
                    e = min(L, s + c)
                    if e > s:
                        self.append(layer, b, np.ascontiguousarray(kb[:, s:e]), np.ascontiguousarray(vb[:, s:e]), s)
                    s = e
                if s < L:
                    self.append(layer, b, np.ascontiguousarray(kb[:, s:]), np.ascontiguousarray(vb[:, s:]), s)

    def read_cache(self, layer: int, seq: int, n: int) -> dict:
        Hkv, d = self.shape.n_kv_heads, self.shape.head_dim
        kc = torch.empty((Hkv, n, d), dtype=torch.int8, device="cuda")
        vc = torch.empty_like(kc)
        ks = torch.empty((Hkv, n), dtype=torch.int16, device="cuda")
        vs = torch.empty_like(ks)
        futr.futr_kv_read(self.kv, layer, seq, n, kc, ks, vc, vs)
        return {"k_codes": kc.cpu().numpy(), "k_scales": ks.cpu().numpy().view(np.float16),
                "v_codes": vc.cpu().numpy(), "v_scales": vs.cpu().numpy().view(np.float16)}

    def decode(self, x_bits: np.ndarray, pos: np.ndarray, layer: int = 0):
        b = x_bits.shape[0]
        x = dev(x_bits.view(np.int16))
        p = dev(pos.astype(np.int32))
        y = torch.empty_like(x)
        futr.futr_decode_block(x, self.blob, self.kv, layer, b, p, y, self.ws)
        st = futr.futr_check(self.ws, self.kv)
        assert st == 0, futr.futr_status_string(st)
        return y

    def intermediates(self, b: int) -> dict:
        s = self.shape
        return {
            "q_rot": futr.ws_view(self.ws, "qrot", (b, s.n_q_heads, s.head_dim), torch.float32)
            .cpu().numpy().astype(np.float64),
            "o": bits_to_f64(futr.ws_view(self.ws, "o", (b, s.q_rows), torch.int16)),
            "h": bits_to_f64(futr.ws_view(self.ws, "h", (b, s.hidden), torch.int16)),
            "a": bits_to_f64(futr.ws_view(self.ws, "a", (b, s.inter), torch.int16)),
        }


def oracle_case(shape, weights, x_bits, hist, pos, gpu: GpuBlock, layer: int = 0):
    """Run the oracle on the same inputs, using the GPU's cache entries for the
    new token (the fused append depends on fp32 accumulation order)."""
    packed = oracle.pack_block(weights)
    wdq = oracle.dequant_block(packed)
    cache = oracle.build_cache(hist, shape)
    b = x_bits.shape[0]
    Hkv, d = shape.n_kv_heads, shape.head_dim
    new = [np.zeros((b, Hkv, d), np.int8), np.zeros((b, Hkv), np.float16),
           np.zeros((b, Hkv, d), np.int8), np.zeros((b, Hkv), np.float16)]
    gcache = []
    for i in range(b):
        L = int(pos[i])
        g = gpu.read_cache(layer, i, L + 1)
        gcache.append(g)
        new[0][i] = g["k_codes"][:, L]
        new[1][i] = g["k_scales"][:, L]
        new[2][i] = g["v_codes"][:, L]
        new[3][i] = g["v_scales"][:, L]
    ref = oracle.decode_block(x_bits, wdq, cache, pos, shape, new_kv=tuple(new))
    return ref, packed, cache, gcache
