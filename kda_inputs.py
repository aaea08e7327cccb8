"""Seeded synthetic inputs for the KDA mixer core.

This module only draws random numbers and rounds them to the storage type; it
holds none of the mixer's arithmetic. Both the CUDA library's tests/benchmark
and the FP64 oracle consume the arrays it returns, so the two sides always see
identical inputs.

Distributions (shaped like the Kimi K3 KDA layer: 96 heads x 128, conv kernel
4; kimi_k3.c header, "KDA per-head recurrence"). A pair N(m, s2) means mean m
and VARIANCE s2:
  q, k, v, z, b, g pre-activations  ~ N(0, 1)
  conv taps                          ~ N(0, 0.25)  (std 0.5)
  dt_bias                            ~ N(0, 0.5)   (std sqrt(0.5))
  A_log                              ~ U(0, ln 16)
  RMSNorm weight                     1 + N(0, 0.1)
BF16 inputs are drawn in FP32 and rounded to nearest-even BF16; the rounded
values (held in float32 arrays) are what both sides consume.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

_STREAMS = {"conv_w": 1, "dt_bias": 2, "A_log": 3, "norm_w": 4,
            "q": 11, "k": 12, "v": 13, "z": 14, "b": 15, "g": 16,
            "state": 21, "tail": 22, "lengths": 31, "slots": 32,
            "x": 41, "w_fa": 42, "w_fb": 43, "w_b": 44}


def _rng(seed: int, stream: str, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _STREAMS[stream], sub])))


_BF16_HALF = np.array([0x7FFF], dtype=np.uint32)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    u = np.array(x, dtype=np.float32, copy=True).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    u += lsb
    u += _BF16_HALF  # finite inputs never wrap
    u &= np.uint32(0xFFFF0000)
    return u.view(np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array holding bf16-representable values -> uint16 bit patterns."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def from_bf16_bits(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class LayerParams:
    conv_w: np.ndarray   # [3, D, K] float32, taps oldest first, for q, k, v
    dt_bias: np.ndarray  # [D] float32
    A_log: np.ndarray    # [H] float32
    norm_w: np.ndarray   # [d] float32


def make_params(H: int, d: int, K: int = 4, seed: int = 0) -> LayerParams:
    D = H * d
    conv_w = (_rng(seed, "conv_w").standard_normal((3, D, K)) * 0.5).astype(np.float32)
    dt_bias = (_rng(seed, "dt_bias").standard_normal(D) * math.sqrt(0.5)).astype(np.float32)
    A_log = _rng(seed, "A_log").uniform(0.0, math.log(16.0), H).astype(np.float32)
    norm_w = (1.0 + _rng(seed, "norm_w").standard_normal(d) * math.sqrt(0.1)).astype(np.float32)
    return LayerParams(conv_w, dt_bias, A_log, norm_w)


def make_tokens(T: int, H: int, d: int, seed: int, bf16: bool, sub: int = 0) -> dict:
    """Per-token pre-activations: q,k,v,z,g [T, H*d] and b [T, H] (float32 arrays)."""
    D = H * d
    out = {}
    for name in ("q", "k", "v", "z", "g"):
        x = _rng(seed, name, sub).standard_normal((T, D), dtype=np.float32)
        out[name] = bf16_round(x) if bf16 else x
    x = _rng(seed, "b", sub).standard_normal((T, H), dtype=np.float32)
    out["b"] = bf16_round(x) if bf16 else x
    return out


def make_tokens_torch(T: int, H: int, d: int, seed: int, sub: int = 0, device="cuda") -> dict:
    """The same distributions drawn on a device by torch's seeded generator, rounded to
    BF16 (nearest-even): q,k,v,z,g [T, H*d] and b [T, H] as BF16 tensors. For workloads too
    large to draw on the host; callers copy the slices they check to the host."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1_000_003 + sub)
    D = H * d
    return {name: torch.randn(T, H if name == "b" else D, generator=gen, device=device).to(torch.bfloat16)
            for name in ("q", "k", "v", "z", "b", "g")}


def make_state(n: int, H: int, d: int, seed: int, std: float = 0.05) -> np.ndarray:
    """A filled recurrent state [n, H, d, d] float32 (entries ~ N(0, std^2))."""
    return (_rng(seed, "state").standard_normal((n, H, d, d), dtype=np.float32) * np.float32(std))


def make_tail(n: int, H: int, d: int, K: int, seed: int, bf16: bool) -> np.ndarray:
    """A filled conv history [n, 3, K-1, H*d] float32 (raw inputs, ~ N(0, 1))."""
    x = _rng(seed, "tail").standard_normal((n, 3, K - 1, H * d), dtype=np.float32)
    return bf16_round(x) if bf16 else x


def make_gate_proj(T: int, hidden: int, H: int, d: int, seed: int, sub: int = 0) -> dict:
    """Inputs of the gate/beta input projections, rounded to BF16 (float32 arrays):
    hidden states x [T, hidden] ~ N(0, 1) and random-init weights scaled by their fan-in,
    W_fa [d, hidden] ~ N(0, 1/hidden), W_fb [H*d, d] ~ N(0, 1/d), W_b [H, hidden] ~
    N(0, 1/hidden), so that f, z and b come out ~ N(0, 1) like the mixer's inputs."""
    x = _rng(seed, "x", sub).standard_normal((T, hidden), dtype=np.float32)
    fa = _rng(seed, "w_fa").standard_normal((d, hidden), dtype=np.float32) * np.float32(hidden ** -0.5)
    fb = _rng(seed, "w_fb").standard_normal((H * d, d), dtype=np.float32) * np.float32(d ** -0.5)
    bp = _rng(seed, "w_b").standard_normal((H, hidden), dtype=np.float32) * np.float32(hidden ** -0.5)
    return {"x": bf16_round(x), "w_fa": bf16_round(fa), "w_fb": bf16_round(fb), "w_b": bf16_round(bp)}


def varlen_lengths(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """n sequence lengths ~ U[lo, hi] (integers, inclusive)."""
    return _rng(seed, "lengths").integers(lo, hi + 1, size=n).astype(np.int64)


# The five workloads (sizes and distributions as the configs state them).
CONFIGS = {
    "tiny": dict(H=2, d=128, K=4, T=64, T_prefill=32, bf16=False, seed=0),
    "decode_b1": dict(H=96, d=128, K=4, B=1, prefill_steps=256, bf16=True, seed=1),
    "decode_b256": dict(H=96, d=128, K=4, B=256, steps=1000, bf16=True, seed=2),
    "prefill_8192": dict(H=96, d=128, K=4, T=8192, C=64, check_tokens=1024, bf16=True, seed=3),
    "varlen": dict(H=96, d=128, K=4, n_seq=16, len_lo=512, len_hi=16384, decode_steps=128,
                   bf16=True, seed=4),
}
