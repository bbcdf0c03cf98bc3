"""Seeded synthetic inputs for causal kernelized linear attention.

This module is shared by the tests, the benchmark and the smoke check, on
both sides of every parity comparison (the CUDA library and the fp64 oracle).
It holds shapes and random draws only — none of the method's arithmetic.

Every draw uses a torch CPU ``Generator`` so that the values do not depend on
the device.  Draw order per forward workload: q, k, v, a, ω.  Values that the
workload stores in bf16 are rounded with round-to-nearest-even by the dtype
cast.  The workloads mirror the shapes and value distributions of the method
description ("Efficient Transformers II" §2.2 eq (6)–(11); "Linear Attention
Research 2026", Performer and elu+1 sections); no public dataset is involved.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional, Tuple

import torch


@dataclass(frozen=True)
class ForwardWorkload:
    name: str
    B: int
    H: int
    n: int
    d: int
    dtype: str                 # "bf16" or "f32"
    feature_map: str           # "elu1" or "performer"
    m: int = 0                 # Performer feature count (d' = m)
    decay: Optional[Tuple[float, float]] = None  # a_h ~ U[lo, hi], None => a = 1
    seed: int = 0
    qk_scale: float = 1.0      # multiplies q and k before rounding
    omega_std: Optional[float] = None  # ω ~ N(0, omega_std²); None => d^-1/2
    modes: Tuple[str, ...] = ("causal",)

    @property
    def dprime(self) -> int:
        return self.d if self.feature_map == "elu1" else self.m

    @property
    def tokens(self) -> int:
        return self.B * self.n


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    H: int
    d: int
    prefill: int
    steps: int
    decay: Tuple[float, float]
    seed: int
    feature_map: str = "elu1"
    m: int = 0
    qk_scale: float = 1.0


# The five workloads of the method's evaluation plan.
TINY_FP32 = ForwardWorkload("tiny_fp32_B1_H1_n256_d32", 1, 1, 256, 32, "f32", "elu1",
                            seed=0, modes=("causal", "noncausal"))
ELU1_DECAY = ForwardWorkload("elu1_decay_B4_H8_n2048_d64", 4, 8, 2048, 64, "bf16", "elu1",
                             decay=(0.9, 0.999), seed=1)
PERFORMER = ForwardWorkload("performer_B2_H8_n4096_d64_m256", 2, 8, 4096, 64, "bf16",
                            "performer", m=256, seed=2, qk_scale=64 ** -0.25,
                            modes=("noncausal", "causal"))
LONG = ForwardWorkload("long_B1_H16_n65536_d128", 1, 16, 65536, 128, "bf16", "elu1",
                       decay=(0.95, 0.9999), seed=3)
DECODE = DecodeWorkload("decode_B256_H32_d128", 256, 32, 128, prefill=512, steps=1024,
                        decay=(0.9, 0.999), seed=4)
# Decode with the Performer map (the recurrent counterpart of the Performer
# workload: d = 64, m = 256, q and k scaled by d^{-1/4}; decay and state size
# as in the decode workload: 8192 heads × 64 KiB of μ).
PERFORMER_DECODE = DecodeWorkload("performer_decode_B256_H32_d64_m256", 256, 32, 64, prefill=512,
                                  steps=1024, decay=(0.9, 0.999), seed=5, feature_map="performer",
                                  m=256, qk_scale=64 ** -0.25)

# Non-causal elu+1 (eq (6) has no decay): the shapes of the elu+1 decay
# workload and of the long workload, each head reading out its totals.
ELU1_NONCAUSAL = ForwardWorkload("elu1_noncausal_B4_H8_n2048_d64", 4, 8, 2048, 64, "bf16", "elu1",
                                 seed=8, modes=("noncausal",))
LONG_NONCAUSAL = ForwardWorkload("long_noncausal_B1_H16_n65536_d128", 1, 16, 65536, 128, "bf16",
                                 "elu1", seed=9, modes=("noncausal",))

FORWARD_WORKLOADS = {w.name: w for w in (TINY_FP32, ELU1_DECAY, PERFORMER, LONG)}


@dataclass(frozen=True)
class TokenDecayWorkload:
    """A forward workload whose decay varies by token (and carries an input
    weight per token), drawn as in the selective state update of the Mamba
    section of "Linear Attention Research 2026": a step Δ_t = softplus(z_t +
    bias) from the input, a_t = exp(−A_h·Δ_t) with a per-head rate A_h, and the
    input weight b_t = Δ_t."""
    base: ForwardWorkload
    rate: Tuple[float, float] = (1.0, 16.0)   # A_h log-uniform in this range
    bias: float = -4.0
    weight: bool = True                       # b_t = Δ_t; False: b_t = 1 − a_t
    resets: float = 0.0                       # fraction of tokens with a_t = 0

    @property
    def name(self) -> str:
        return "token_decay_" + self.base.name.split("_", 1)[1]


# The long-sequence shape with a per-token decay and weight.
TOKEN_DECAY_LONG = TokenDecayWorkload(ForwardWorkload("long_B1_H16_n65536_d128", 1, 16, 65536,
                                                      128, "bf16", "elu1", seed=6))

_TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPE[name]


def make_forward_inputs(B, H, n, d, dtype="bf16", feature_map="elu1", m=0,
                        decay=None, seed=0, qk_scale=1.0, omega_std=None):
    """Return a dict of CPU tensors: q, k, v [B,H,n,d] in ``dtype``,
    a [H] fp32 or None, omega [d,m] in ``dtype`` or None."""
    g = torch.Generator().manual_seed(int(seed))
    dt = _TORCH_DTYPE[dtype]
    q = torch.randn(B, H, n, d, generator=g)
    k = torch.randn(B, H, n, d, generator=g)
    v = torch.randn(B, H, n, d, generator=g)
    if qk_scale != 1.0:
        q = q * qk_scale
        k = k * qk_scale
    a = None
    if decay is not None:
        lo, hi = decay
        a = (torch.rand(H, generator=g, dtype=torch.float64) * (hi - lo) + lo).float()
    omega = None
    if feature_map == "performer":
        std = (d ** -0.5) if omega_std is None else omega_std
        omega = (torch.randn(d, m, generator=g) * std).to(dt)
    return {"q": q.to(dt), "k": k.to(dt), "v": v.to(dt), "a": a, "omega": omega}


def forward_inputs(w: ForwardWorkload, n: Optional[int] = None, B: Optional[int] = None,
                   H: Optional[int] = None):
    """Inputs of a named workload (optionally with fewer tokens/heads for a
    quick case drawn the same way)."""
    return make_forward_inputs(B or w.B, H or w.H, n or w.n, w.d, w.dtype, w.feature_map,
                               w.m, w.decay, w.seed, w.qk_scale, w.omega_std)


def decode_prefill_inputs(w: DecodeWorkload, B: Optional[int] = None, H: Optional[int] = None):
    """Prefill q, k, v [B,H,prefill,d] bf16, the per-head decay a [H] fp32 and
    (Performer) ω [d, m]."""
    return make_forward_inputs(B or w.B, H or w.H, w.prefill, w.d, "bf16", w.feature_map, w.m,
                               decay=w.decay, seed=w.seed, qk_scale=w.qk_scale)


def decode_step_inputs(w: DecodeWorkload, step: int, B: Optional[int] = None,
                       H: Optional[int] = None):
    """Fresh bf16 q, k, v [B,H,d] for one decode step; each step has its own
    seed so that any step can be regenerated on its own."""
    g = torch.Generator().manual_seed(int(w.seed) * 1_000_003 + 7919 * (int(step) + 1))
    B = B or w.B
    H = H or w.H
    q = torch.randn(B, H, w.d, generator=g) * w.qk_scale
    k = torch.randn(B, H, w.d, generator=g) * w.qk_scale
    v = torch.randn(B, H, w.d, generator=g)
    return {"q": q.bfloat16(), "k": k.bfloat16(), "v": v.bfloat16()}


def make_token_decay(B, H, n, seed, rate=(1.0, 16.0), bias=-4.0, weight=True, resets=0.0):
    """Per-token decay a [B,H,n] fp32 and input weight b [B,H,n] fp32 (None
    when ``weight`` is False): Δ = softplus(z + bias), z ~ N(0, 1); a = exp(−A_h·Δ)
    with A_h log-uniform in ``rate``; b = Δ; a fraction ``resets`` of the
    tokens (chosen uniformly) get a = 0.  Drawn in fp64 from their own
    generator, then rounded to fp32."""
    g = torch.Generator().manual_seed(int(seed) * 7919 + 104729)
    lo, hi = rate
    A = torch.exp(torch.rand(H, generator=g, dtype=torch.float64) * (math.log(hi) - math.log(lo))
                  + math.log(lo))
    z = torch.randn(B, H, n, generator=g, dtype=torch.float64)
    delta = torch.nn.functional.softplus(z + bias)
    a = torch.exp(-A[None, :, None] * delta)
    if resets > 0.0:
        a = torch.where(torch.rand(B, H, n, generator=g, dtype=torch.float64) < resets,
                        torch.zeros_like(a), a)
    return a.float(), (delta.float() if weight else None)


def token_decay_inputs(w: TokenDecayWorkload, n: Optional[int] = None, B: Optional[int] = None,
                       H: Optional[int] = None):
    """q, k, v (as the base workload) plus the per-token a and b."""
    x = forward_inputs(w.base, n=n, B=B, H=H)
    a, b = make_token_decay(B or w.base.B, H or w.base.H, n or w.base.n, w.base.seed, w.rate,
                            w.bias, w.weight, w.resets)
    x["a"] = None
    x["a_tok"] = a
    x["b_tok"] = b
    return x
