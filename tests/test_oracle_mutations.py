"""Planted mistakes in the oracle must fail its pins.

Each case below replaces one function of the float64 oracle, in the module and
in the package namespace and only for the duration of the case, by a version
carrying one plausible mistake (a dropped term, a wrong sign, index or operand
order, a wrong rounding or constant), runs every pin of ``test_oracle_pins``
and requires at least one to fail on an assertion (an error raised by a pin
does not count).  The same rewrites built
without their mistake, and the unmodified oracle, must pass every pin: so a
failure is due to the planted mistake, not to the rewrite.  Everything here
runs on the CPU.
"""
import inspect
import math

import numpy as np
import pytest

import oracle
from oracle import futr_oracle as O
from tests import test_oracle_pins as P

ORIG = {name: getattr(O, name) for name in (
    "rope", "stage_attention", "fwht_f32", "hadamard", "rotate", "quant_rtn", "dequant", "fold_gain",
    "pack_block", "rms_factor", "stage_qkv", "stage_o", "stage_mlp_in", "stage_down", "silu", "final_logits",
    "embed", "decode_step", "round_bf16", "online_softmax_attention", "softmax_attention", "build_cache",
    "new_kv_codes", "gptq_quantize", "gptq_hessian", "pack_block_gptq")}


def _pins():
    """(id, function, kwargs) for every pin, parametrized ones expanded."""
    out = []
    for name, fn in inspect.getmembers(P, inspect.isfunction):
        if not name.startswith("test_") or fn.__module__ != P.__name__:
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            out.append((name, fn, {}))
            continue
        assert len(marks) == 1
        names = [a.strip() for a in marks[0].args[0].split(",")]
        for i, v in enumerate(marks[0].args[1]):
            out.append((f"{name}[{i}]", fn, dict(zip(names, v)) if len(names) > 1 else {names[0]: v}))
    return out


PINS = _pins()


def failing_pins(monkeypatch, name, fn):
    """Pins that fail on an assertion, and pins that raise anything else, with
    `fn` in place of the oracle's function `name`."""
    monkeypatch.setattr(O, name, fn)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, fn)
    failed, raised = [], []
    with np.errstate(all="ignore"):
        for pin_id, pin, kw in PINS:
            try:
                pin(**kw)
            except AssertionError:
                failed.append(pin_id)
            except Exception as e:  # a shape or type error is not a pin's verdict
                raised.append(f"{pin_id}: {type(e).__name__}")
    return failed, raised


# ----------------------------------------------- rewrites with a mistake switch

def _rope(sign=1.0, freq_factor=2.0, interleaved=False):
    def rope(v, pos, theta):
        v = np.asarray(v, dtype=np.float64)
        d = v.shape[-1]
        half = d // 2
        inv = theta ** (-(freq_factor * np.arange(half)) / d)
        ang = sign * np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]
        c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
        x1, x2 = (v[..., 0::2], v[..., 1::2]) if interleaved else (v[..., :half], v[..., half:])
        a, b = x1 * c - x2 * s, x2 * c + x1 * s
        out = np.empty_like(v)
        if interleaved:
            out[..., 0::2], out[..., 1::2] = a, b
        else:
            out[..., :half], out[..., half:] = a, b
        return out
    return rope


def _attention(gqa_modulo=False, scaled=True, rotate_back=True, drop_new=False):
    def stage_attention(q_rot, k_cache, v_cache, shape, rnd=None):
        b = q_rot.shape[0]
        Hq, Hkv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
        o = np.zeros((b, Hq, d))
        for i in range(b):
            for h in range(Hq):
                kv = h % Hkv if gqa_modulo else h // (Hq // Hkv)
                k, v = k_cache[i][kv], v_cache[i][kv]
                if drop_new:
                    k, v = k[:-1], v[:-1]
                o[i, h] = O.softmax_attention(q_rot[i, h], k, v, 1.0 / math.sqrt(d) if scaled else 1.0)
        if rotate_back:
            o = O.rotate(o, shape.had_block)
        return (rnd or O.round_bf16)(o.reshape(b, Hq * d))
    return stage_attention


def _fwht(swap_sign=False, normalise=True):
    def fwht_f32(v, n):
        v = np.array(v, dtype=np.float32, copy=True)
        d = v.shape[-1]
        lead = v.shape[:-1]
        w = v.reshape(lead + (d // n, n))
        h = 1
        while h < n:
            w = w.reshape(lead + (d // n, n // (2 * h), 2, h))
            a, b = w[..., 0, :], w[..., 1, :]
            w = np.stack([a - b, a + b] if swap_sign else [a + b, a - b], axis=-2)
            h *= 2
        w = w.reshape(lead + (d,))
        return w * np.float32(1.0 / math.sqrt(n)) if normalise else w
    return fwht_f32


def _hadamard(sylvester=True):
    def hadamard(n):
        h = np.ones((1, 1), dtype=np.int64)
        while h.shape[0] < n:
            h = np.block([[h, h], [h, -h]]) if sylvester else np.block([[h, h], [-h, h]])
        return h
    return hadamard


def _rotate(normalise=True):
    def rotate(v, n):
        v = np.asarray(v, dtype=np.float64)
        d = v.shape[-1]
        blocks = v.reshape(v.shape[:-1] + (d // n, n))
        out = blocks @ O.hadamard(n).T.astype(np.float64)
        return (out / math.sqrt(n) if normalise else out).reshape(v.shape)
    return rotate


def _quant(divisor=7.0, rnd=np.rint, lo=-8, fp16_scale=True):
    def quant_rtn(v32):
        v = np.asarray(v32, dtype=np.float32)
        a = np.max(np.abs(v), axis=-1)
        q7 = np.minimum((a / np.float32(divisor)).astype(np.float32), np.float32(O.FP16_MAX))
        s16 = q7.astype(np.float16)
        s32 = (s16.astype(np.float32) if fp16_scale else q7)[..., None]
        q = (v / np.where(s32 > 0, s32, np.float32(1.0))).astype(np.float32)
        return np.where(s32 > 0, np.clip(rnd(q), lo, 7), 0).astype(np.int8), s16
    return quant_rtn


def _dequant(tiled=False):
    def dequant(codes, scales, group):
        c = np.asarray(codes, dtype=np.float64)
        s = np.asarray(scales, dtype=np.float64)
        if tiled:  # element j takes scale j mod (number of groups)
            return c * np.tile(s, (1,) * (s.ndim - 1) + (group,))
        return c * np.repeat(s, group, axis=-1)
    return dequant


def _fold(divide=False):
    def fold_gain(w, g):
        w = np.asarray(w, dtype=np.float32)
        if g is None:
            return w.copy()
        g = np.asarray(g, dtype=np.float32)[None, :]
        return (w / g if divide else w * g).astype(np.float32)
    return fold_gain


def _pack(attn_gain_on="qkv", mlp_gain_on=("gate", "up")):
    def pack_block(weights, group=128):
        wqkv = np.concatenate([weights["wq"], weights["wk"], weights["wv"]], axis=0)
        mats = {"qkv": wqkv, "o": weights["wo"], "gate": weights["wgate"], "up": weights["wup"],
                "down": weights["wdown"]}
        gains = {k: None for k in mats}
        gains[attn_gain_on] = weights["g_attn"]
        for k in mlp_gain_on:
            gains[k] = weights["g_mlp"]
        return {k: O.quantize_weight(m, gains[k], group) for k, m in mats.items()}
    return pack_block


def _rms(mean=True, eps_inside=True):
    def rms_factor(x, eps):
        x = np.asarray(x, dtype=np.float64)
        ss = np.mean(x * x, axis=-1) if mean else np.sum(x * x, axis=-1)
        return 1.0 / np.sqrt(ss + eps) if eps_inside else 1.0 / (np.sqrt(ss) + eps)
    return rms_factor


def _qkv(rope_k=True, rotate_q=True, swap_kv=False):
    def stage_qkv(x, wqkv, pos, shape):
        b = x.shape[0]
        Hq, Hkv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
        qkv = O.rms_factor(x, shape.rms_eps)[:, None] * (x @ wqkv.T)
        q = qkv[:, :Hq * d].reshape(b, Hq, d)
        k = qkv[:, Hq * d:(Hq + Hkv) * d].reshape(b, Hkv, d)
        v = qkv[:, (Hq + Hkv) * d:].reshape(b, Hkv, d)
        if swap_kv:
            k, v = v, k
        q = O.rope(q, pos, shape.rope_theta)
        if rope_k:
            k = O.rope(k, pos, shape.rope_theta)
        return {"q_rot": O.rotate(q, shape.had_block) if rotate_q else q, "k_new": k, "v_new": v}
    return stage_qkv


def _residual(keep=True):
    def stage(x, inp, w, rnd=None):
        return (rnd or O.round_bf16)((x if keep else 0.0) + inp @ w.T)
    return stage


def _mlp_in(swap=False, normalise=True):
    def stage_mlp_in(h, wgate, wup, eps, rnd=None):
        r = O.rms_factor(h, eps)[:, None] if normalise else 1.0
        g, u = r * (h @ wgate.T), r * (h @ wup.T)
        if swap:
            g, u = u, g
        return (rnd or O.round_bf16)(O.silu(g) * u)
    return stage_mlp_in


def _silu(sign=-1.0):
    return lambda z: z / (1.0 + np.exp(sign * z))


def _final(gain_before_rounding=True, normalise=True):
    def final_logits(y, g_final, w_lm_bits, eps):
        y = np.asarray(y, dtype=np.float64)
        g = np.asarray(g_final, dtype=np.float32)
        if gain_before_rounding:
            xg = O.round_bf16((y.astype(np.float32) * g).astype(np.float64))
        else:
            xg = O.round_bf16(y) * g.astype(np.float64)
        r = O.rms_factor(y, eps) if normalise else np.ones(y.shape[0])
        return r[:, None] * (xg @ O.bf16_bits_to_float(w_lm_bits).T)
    return final_logits


def _embed(offset=0):
    def embed(tokens, table_bits):
        t = np.asarray(table_bits)
        return t[(np.asarray(tokens, dtype=np.int64) + offset) % t.shape[0]]
    return embed


def _step(chain=True):
    def decode_step(tokens, table_bits, layers, caches, pos, g_final, w_lm_bits, shape, new_kv=None):
        x0 = x_bits = O.embed(tokens, table_bits)
        ys = []
        for l, wdq in enumerate(layers):
            out = O.decode_block(x_bits, wdq, caches[l], pos, shape, None if new_kv is None else new_kv[l])
            ys.append(out["y"])
            x_bits = O.float_to_bf16_bits(out["y"]) if chain else x0
        return {"y": ys, "logits": O.final_logits(ys[-1], g_final, w_lm_bits, shape.rms_eps)}
    return decode_step


def _round_bf16(rnd=np.rint, bits=8):
    def round_bf16(x):
        x = np.asarray(x, dtype=np.float64)
        m, e = np.frexp(x)
        ulp = np.ldexp(1.0, np.maximum(e, -125) - bits)
        return rnd(x / ulp) * ulp
    return round_bf16


def _online(correct=True, rescale=True):
    def online_softmax_attention(q, k, v, scale, chunk):
        parts = []
        for c0 in range(0, k.shape[0], chunk):
            m, l, o = -np.inf, 0.0, np.zeros(v.shape[1])
            for kj, vj in zip(k[c0:c0 + chunk], v[c0:c0 + chunk]):
                sj = float(kj @ q) * scale
                mn = max(m, sj)
                corr = (math.exp(m - mn) if m != -np.inf else 0.0) if correct else 1.0
                pj = math.exp(sj - mn)
                l, o, m = l * corr + pj, o * corr + pj * vj, mn
            parts.append((m, l, o))
        M = max(p[0] for p in parts)
        f = [math.exp(p[0] - M) if rescale else 1.0 for p in parts]
        return sum(fi * p[2] for fi, p in zip(f, parts)) / sum(fi * p[1] for fi, p in zip(f, parts))
    return online_softmax_attention


def _softmax(shift=True, sum_normalise=True):
    def softmax_attention(q, k, v, scale):
        s = (k @ q) * scale
        p = np.exp(s - np.max(s)) if shift else np.exp(s)
        return (p @ v) / (np.sum(p) if sum_normalise else np.max(p))
    return softmax_attention


def _build_cache(swap_kv=False, rotate=True):
    def build_cache(kv_hist, shape):
        out = []
        for kb, vb in kv_hist:
            if swap_kv:
                kb, vb = vb, kb
            k32 = O.bf16_bits_to_float(kb).astype(np.float32)
            v32 = O.bf16_bits_to_float(vb).astype(np.float32)
            q = (lambda a: O.kv_quantize(a, shape.had_block)) if rotate else O.quant_rtn
            (kc, ks), (vc, vs) = q(k32), q(v32)
            out.append({"k_codes": kc, "k_scales": ks, "v_codes": vc, "v_scales": vs})
        return out
    return build_cache


def _new_kv(rotate=True):
    def new_kv_codes(k_new, v_new, shape):
        q = (lambda a: O.kv_quantize(a, shape.had_block)) if rotate else O.quant_rtn
        (kc, ks), (vc, vs) = q(k_new.astype(np.float32)), q(v_new.astype(np.float32))
        return kc, ks, vc, vs
    return new_kv_codes


def _gptq(divide=True, spread_sign=1.0, scale_from_current=True, dampen=True, zero_dead=True, upper=True):
    def gptq_quantize(w32, h, group=128, damp=0.01):
        w = np.array(w32, dtype=np.float32).astype(np.float64)
        n, k = w.shape
        hh = np.array(h, dtype=np.float64, copy=True)
        dead = np.diag(hh) == 0
        hh[dead, dead] = 1.0
        if zero_dead:
            w[:, dead] = 0.0
        w0 = w.copy()
        if dampen:
            hh[np.diag_indices(k)] += damp * np.mean(np.diag(hh))
        low = np.linalg.cholesky(np.linalg.inv(hh))
        u = low.T if upper else low
        codes = np.zeros((n, k), dtype=np.int8)
        scales = np.zeros((n, k // group), dtype=np.float16)
        for j in range(k):
            gi = j // group
            if j % group == 0:
                src = w if scale_from_current else w0
                scales[:, gi] = O.rtn_scale(src[:, j:j + group].astype(np.float32))
            c = O.rtn_codes(w[:, j:j + 1].astype(np.float32), scales[:, gi])[:, 0]
            codes[:, j] = c
            e = (w[:, j] - c * scales[:, gi].astype(np.float64)) / (u[j, j] if divide else 1.0)
            w[:, j + 1:] -= spread_sign * np.outer(e, u[j, j + 1:])
        return codes, scales
    return gptq_quantize


def _hessian(factor=2.0):
    def gptq_hessian(xcal):
        x = np.asarray(xcal, dtype=np.float64)
        return (factor / x.shape[0]) * (x.T @ x)
    return gptq_hessian


def _pack_gptq(down_key="down", o_key="o"):
    def pack_block_gptq(weights, hessians, group=128, damp=0.01):
        wqkv = np.concatenate([weights["wq"], weights["wk"], weights["wv"]], axis=0)
        q = lambda m, g, hk: O.gptq_quantize_weight(m, g, hessians[hk], group, damp)
        return {"qkv": q(wqkv, weights["g_attn"], "attn"), "o": q(weights["wo"], None, o_key),
                "gate": q(weights["wgate"], weights["g_mlp"], "mlp"), "up": q(weights["wup"], weights["g_mlp"], "mlp"),
                "down": q(weights["wdown"], None, down_key)}
    return pack_block_gptq


# (oracle function, factory, mistake-free arguments, planted mistake)
CASES = {
    "rope_reversed_rotation": ("rope", _rope, {}, dict(sign=-1.0)),
    "rope_frequency_exponent": ("rope", _rope, {}, dict(freq_factor=1.0)),
    "rope_interleaved_pairs": ("rope", _rope, {}, dict(interleaved=True)),
    "gqa_head_modulo": ("stage_attention", _attention, {}, dict(gqa_modulo=True)),
    "attention_unscaled": ("stage_attention", _attention, {}, dict(scaled=False)),
    "no_inverse_rotation": ("stage_attention", _attention, {}, dict(rotate_back=False)),
    "new_token_not_attended": ("stage_attention", _attention, {}, dict(drop_new=True)),
    "butterfly_sign": ("fwht_f32", _fwht, {}, dict(swap_sign=True)),
    "butterfly_unnormalised": ("fwht_f32", _fwht, {}, dict(normalise=False)),
    "hadamard_not_sylvester": ("hadamard", _hadamard, {}, dict(sylvester=False)),
    "rotation_unnormalised": ("rotate", _rotate, {}, dict(normalise=False)),
    "scale_divisor_8": ("quant_rtn", _quant, {}, dict(divisor=8.0)),
    "round_half_up": ("quant_rtn", _quant, {}, dict(rnd=lambda q: np.floor(q + np.float32(0.5)))),
    "round_toward_zero": ("quant_rtn", _quant, {}, dict(rnd=np.trunc)),
    "clamp_symmetric": ("quant_rtn", _quant, {}, dict(lo=-7)),
    "codes_from_unrounded_scale": ("quant_rtn", _quant, {}, dict(fp16_scale=False)),
    "dequant_scale_of_wrong_group": ("dequant", _dequant, {}, dict(tiled=True)),
    "gain_divided": ("fold_gain", _fold, {}, dict(divide=True)),
    "attn_gain_on_o": ("pack_block", _pack, {}, dict(attn_gain_on="o")),
    "mlp_gain_on_down": ("pack_block", _pack, {}, dict(mlp_gain_on=("gate", "down"))),
    "rms_sum_not_mean": ("rms_factor", _rms, {}, dict(mean=False)),
    "rms_eps_outside_sqrt": ("rms_factor", _rms, {}, dict(eps_inside=False)),
    "k_without_rope": ("stage_qkv", _qkv, {}, dict(rope_k=False)),
    "query_not_rotated": ("stage_qkv", _qkv, {}, dict(rotate_q=False)),
    "k_v_rows_swapped": ("stage_qkv", _qkv, {}, dict(swap_kv=True)),
    "o_residual_dropped": ("stage_o", _residual, {}, dict(keep=False)),
    "down_residual_dropped": ("stage_down", _residual, {}, dict(keep=False)),
    "swiglu_gate_up_swapped": ("stage_mlp_in", _mlp_in, {}, dict(swap=True)),
    "mlp_rmsnorm_dropped": ("stage_mlp_in", _mlp_in, {}, dict(normalise=False)),
    "silu_sign": ("silu", _silu, {}, dict(sign=1.0)),
    "lm_gain_after_rounding": ("final_logits", _final, {}, dict(gain_before_rounding=False)),
    "lm_rmsnorm_dropped": ("final_logits", _final, {}, dict(normalise=False)),
    "embedding_row_off_by_one": ("embed", _embed, {}, dict(offset=1)),
    "blocks_not_chained": ("decode_step", _step, {}, dict(chain=False)),
    "bf16_truncates": ("round_bf16", _round_bf16, {}, dict(rnd=np.trunc)),
    "bf16_seven_bits": ("round_bf16", _round_bf16, {}, dict(bits=7)),
    "online_softmax_no_correction": ("online_softmax_attention", _online, {}, dict(correct=False)),
    "online_merge_not_rescaled": ("online_softmax_attention", _online, {}, dict(rescale=False)),
    "softmax_normalised_by_max": ("softmax_attention", _softmax, {}, dict(sum_normalise=False)),
    "cache_k_v_swapped": ("build_cache", _build_cache, {}, dict(swap_kv=True)),
    "cache_not_rotated": ("build_cache", _build_cache, {}, dict(rotate=False)),
    "new_token_not_rotated": ("new_kv_codes", _new_kv, {}, dict(rotate=False)),
    "gptq_error_not_divided": ("gptq_quantize", _gptq, {}, dict(divide=False)),
    "gptq_error_spread_sign": ("gptq_quantize", _gptq, {}, dict(spread_sign=-1.0)),
    "gptq_scale_from_original_weights": ("gptq_quantize", _gptq, {}, dict(scale_from_current=False)),
    "gptq_undampened": ("gptq_quantize", _gptq, {}, dict(dampen=False)),
    "gptq_dead_inputs_kept": ("gptq_quantize", _gptq, {}, dict(zero_dead=False)),
    "gptq_lower_cholesky_factor": ("gptq_quantize", _gptq, {}, dict(upper=False)),
    "gptq_hessian_unscaled": ("gptq_hessian", _hessian, {}, dict(factor=1.0)),
    "gptq_down_with_mlp_hessian": ("pack_block_gptq", _pack_gptq, {}, dict(down_key="mlp")),
}


def test_unmodified_oracle_passes_every_pin(monkeypatch):
    assert len(PINS) > 40
    assert failing_pins(monkeypatch, "rope", ORIG["rope"]) == ([], [])


@pytest.mark.parametrize("factory", sorted({(c[0], c[1]) for c in CASES.values()}, key=lambda t: t[0]),
                         ids=lambda t: t[0])
def test_rewrite_without_mistake_passes_every_pin(monkeypatch, factory):
    name, make = factory
    assert failing_pins(monkeypatch, name, make()) == ([], [])


@pytest.mark.parametrize("case", sorted(CASES))
def test_planted_mistake_fails_a_pin(monkeypatch, case):
    name, make, _, mistake = CASES[case]
    failed, _ = failing_pins(monkeypatch, name, make(**mistake))
    assert failed, f"no pin fails on an assertion for {case}"
