"""Seeded synthetic inputs for the INT4 decode block.

This module is the one piece shared by the CUDA path and the float64 oracle.
It draws random numbers and nothing else: no folding, quantization, rotation
or any other step of the method lives here.  bf16 tensors are represented as
``uint16`` bit patterns (numpy has no bfloat16); the single fp32 -> bf16 cast
used to make bf16 inputs is torch's CPU cast.

Workloads follow the shapes of the INT4 decode experiments described in
"FuTransformer: FP8 prefill and INT4 decode for Llama-style inference on
Hopper" (abstract: 8B and 70B Llama shapes, batch 1-32).  Every component is
drawn from its own PCG64 stream, ``SeedSequence(seed, spawn_key=(k,))`` with a
fixed k per component, so that large pieces can be generated independently.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np

# component -> spawn key (fixed; changing one changes every seeded input)
_STREAM = {
    "wq": 1, "wk": 2, "wv": 3, "wo": 4, "wgate": 5, "wup": 6, "wdown": 7,
    "g_attn": 8, "g_mlp": 9, "x": 10, "lengths": 11, "outliers": 12, "kv": 13, "calib": 14,
}


@dataclasses.dataclass(frozen=True)
class BlockShape:
    """Shape of one Llama-style decoder block."""
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    inter: int
    had_block: int
    group: int = 128
    rms_eps: float = 1e-5
    rope_theta: float = 500000.0

    @property
    def q_rows(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_rows(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def qkv_rows(self) -> int:
        return self.q_rows + 2 * self.kv_rows


@dataclasses.dataclass(frozen=True)
class Workload:
    """A named decode workload: block shape, batch, cached lengths recipe."""
    name: str
    shape: BlockShape
    batch: int
    ctx: int                       # cached positions per sequence (fixed)
    ragged: Optional[tuple] = None  # (lo, hi) inclusive uniform range, if ragged
    n_outlier: int = 4              # outlier key channels per kv-head (x20)
    outlier_gain: float = 20.0
    n_layers: int = 1
    vocab: int = 0                  # > 0: the full decode step (embedding, n_layers blocks, LM head)


TOY = BlockShape(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, inter=768, had_block=64)
LLAMA8B = BlockShape(hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128, inter=14336, had_block=128)
LLAMA70B = BlockShape(hidden=8192, n_q_heads=64, n_kv_heads=8, head_dim=128, inter=28672, had_block=128)

# 3% of 128 key channels rounds to 4 outlier channels per kv-head.
WORKLOADS: Dict[str, Workload] = {
    "toy_b1_ctx128": Workload("toy_b1_ctx128", TOY, 1, 128, n_outlier=4),
    "llama8b_b1_ctx1024": Workload("llama8b_b1_ctx1024", LLAMA8B, 1, 1024),
    "llama8b_b8_ctx1024": Workload("llama8b_b8_ctx1024", LLAMA8B, 8, 1024),
    "llama8b_b32_ragged512-4096": Workload("llama8b_b32_ragged512-4096", LLAMA8B, 32, 4096,
                                           ragged=(512, 4096)),
    "llama70b_b1_ctx2048": Workload("llama70b_b1_ctx2048", LLAMA70B, 1, 2048),
    "llama70b_b8_ctx2048": Workload("llama70b_b8_ctx2048", LLAMA70B, 8, 2048),
    "llama70b_b32_ctx2048": Workload("llama70b_b32_ctx2048", LLAMA70B, 32, 2048),
    # complete 8B model step: 32 blocks + embedding + final norm + bf16 LM head
    "llama8b_x32_b1_ctx2048": Workload("llama8b_x32_b1_ctx2048", LLAMA8B, 1, 2048, n_layers=32, vocab=128256),
    "llama8b_x32_b16_ctx2048": Workload("llama8b_x32_b16_ctx2048", LLAMA8B, 16, 2048, n_layers=32, vocab=128256),
    # two layers + the full head: a few GB on the device, for kernel profiles
    "llama8b_x2_b1_ctx2048": Workload("llama8b_x2_b1_ctx2048", LLAMA8B, 1, 2048, n_layers=2, vocab=128256),
}


def rng_for(seed: int, component: str) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(seed, spawn_key=(_STREAM[component],)))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), round-to-nearest-even (torch CPU cast)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> the fp32 values they encode (exact widening)."""
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal(seed: int, comp: str, shape, std: float) -> np.ndarray:
    a = rng_for(seed, comp).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def block_weights(shape: BlockShape, seed: int = 0, std: float = 0.02) -> Dict[str, np.ndarray]:
    """fp32 projection weights [out, in] (nn.Linear layout), N(0, std^2), and
    RMSNorm gains U[0.5, 1.5]."""
    H, I = shape.hidden, shape.inter
    w = {
        "wq": _normal(seed, "wq", (shape.q_rows, H), std),
        "wk": _normal(seed, "wk", (shape.kv_rows, H), std),
        "wv": _normal(seed, "wv", (shape.kv_rows, H), std),
        "wo": _normal(seed, "wo", (H, shape.q_rows), std),
        "wgate": _normal(seed, "wgate", (I, H), std),
        "wup": _normal(seed, "wup", (I, H), std),
        "wdown": _normal(seed, "wdown", (H, I), std),
        "g_attn": rng_for(seed, "g_attn").uniform(0.5, 1.5, H).astype(np.float32),
        "g_mlp": rng_for(seed, "g_mlp").uniform(0.5, 1.5, H).astype(np.float32),
    }
    return w


def activations(shape: BlockShape, batch: int, seed: int = 0) -> np.ndarray:
    """Block input x ~ N(0, 1), as bf16 bits [batch, hidden]."""
    return to_bf16_bits(_normal(seed, "x", (batch, shape.hidden), 1.0))


def context_lengths(wl: Workload, seed: int = 0) -> np.ndarray:
    """Cached positions per sequence (int32 [batch])."""
    if wl.ragged is None:
        return np.full(wl.batch, wl.ctx, dtype=np.int32)
    lo, hi = wl.ragged
    return rng_for(seed, "lengths").integers(lo, hi + 1, size=wl.batch).astype(np.int32)


def outlier_channels(shape: BlockShape, n_outlier: int, seed: int = 0) -> np.ndarray:
    """Per kv-head set of key channels (without replacement) that carry outliers."""
    r = rng_for(seed, "outliers")
    return np.stack([r.choice(shape.head_dim, size=n_outlier, replace=False)
                     for _ in range(shape.n_kv_heads)]).astype(np.int64)


def kv_history(shape: BlockShape, lengths: Sequence[int], n_outlier: int = 4,
               gain: float = 20.0, seed: int = 0) -> List[tuple]:
    """Cached keys/values for each sequence: K, V ~ N(0, 1) of shape
    [n_kv_heads, L_b, head_dim]; in every kv-head a fixed set of key channels
    is multiplied by ``gain`` (values untouched).  Returned as bf16 bits."""
    chans = outlier_channels(shape, n_outlier, seed)
    r = rng_for(seed, "kv")
    out = []
    for L in lengths:
        k = r.standard_normal((shape.n_kv_heads, int(L), shape.head_dim), dtype=np.float32)
        v = r.standard_normal((shape.n_kv_heads, int(L), shape.head_dim), dtype=np.float32)
        for h in range(shape.n_kv_heads):
            k[h][:, chans[h]] *= np.float32(gain)
        out.append((to_bf16_bits(k), to_bf16_bits(v)))
    return out


def calibration_inputs(k: int, n: int, seed: int = 0, rank: int = 8, spread: float = 4.0) -> np.ndarray:
    """Synthetic calibration inputs of one projection, fp32 [n, k]: a rank-`rank`
    shared part plus independent noise, each channel then scaled by a factor
    drawn log-uniformly from [1/spread, spread].  The channels are correlated and
    unevenly scaled, as the inputs of a trained model's projections are; there
    is no trained model here to take them from."""
    r = rng_for(seed, "calib")
    z = r.standard_normal((n, rank), dtype=np.float32)
    mix = r.standard_normal((rank, k), dtype=np.float32)
    noise = r.standard_normal((n, k), dtype=np.float32)
    scale = np.exp(r.uniform(-np.log(spread), np.log(spread), k)).astype(np.float32)
    return ((z @ mix + noise) * scale).astype(np.float32)


# Device-side generators for the complete-model workloads (32 layers of fp32
# weights would not fit a host array comfortably): torch's counter-based
# generator on the GPU, one seed per layer and component.

def block_weights_device(shape: BlockShape, seed: int, std: float = 0.02):
    """As ``block_weights``, generated on cuda:0 (dict of fp32 tensors)."""
    import torch
    H, I = shape.hidden, shape.inter
    g = torch.Generator(device="cuda").manual_seed(1_000_003 * (seed + 1))
    n = lambda *sz: torch.randn(sz, generator=g, device="cuda", dtype=torch.float32) * std
    return {"wq": n(shape.q_rows, H), "wk": n(shape.kv_rows, H), "wv": n(shape.kv_rows, H),
            "wo": n(H, shape.q_rows), "wgate": n(I, H), "wup": n(I, H), "wdown": n(H, I),
            "g_attn": torch.rand(H, generator=g, device="cuda") + 0.5,
            "g_mlp": torch.rand(H, generator=g, device="cuda") + 0.5}


def kv_history_device(shape: BlockShape, length: int, seed: int, n_outlier: int = 4, gain: float = 20.0):
    """One sequence's cached K, V on cuda:0 (bf16 bits [Hkv, length, d] as int16
    tensors), N(0, 1) with ``n_outlier`` key channels per kv-head times ``gain``."""
    import torch
    g = torch.Generator(device="cuda").manual_seed(7_000_003 * (seed + 1))
    k = torch.randn((shape.n_kv_heads, length, shape.head_dim), generator=g, device="cuda")
    v = torch.randn((shape.n_kv_heads, length, shape.head_dim), generator=g, device="cuda")
    chans = torch.from_numpy(outlier_channels(shape, n_outlier, seed)).cuda()
    k.scatter_(2, chans[:, None, :].expand(-1, length, -1), k.gather(2, chans[:, None, :].expand(-1, length, -1)) * gain)
    return k.to(torch.bfloat16).view(torch.int16), v.to(torch.bfloat16).view(torch.int16)
