"""Seeded synthetic inputs for the mLSTM forward pass and the recurrent step.

This module only draws random numbers and lays them out; it holds none of the
mLSTM arithmetic, so both the CUDA path and the fp64 oracle can consume its
output without sharing any computation.

Every tensor is drawn on the host in fp32 from a ``torch.Generator`` seeded
with the given seed, in a fixed order, then cast to the requested dtype.  A
consumer that wants fp64 values widens the *cast* tensor, so both sides see
bit-identical inputs.  ``N(mu, sd)`` below means mean ``mu`` and standard
deviation ``sd``.

The named workloads are synthetic stand-ins for the layer shapes of the xLSTM
language models ("xLSTM: Extended Long Short-Term Memory", section 2.4 "xLSTM
Blocks": mLSTM sits in a pre-up-projection block, so the head dimension is
twice the embedding width divided by the number of heads).  No dataset or
trained weight is involved.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class ParallelWorkload:
    name: str
    B: int
    H: int
    T: int
    d_qk: int
    d_v: int
    dtype: torch.dtype          # dtype of q, k, v (and of the output)
    qkv_std: float = 1.0
    ig_mean: float = 0.0
    ig_std: float = 1.0
    fg_mean: float = 3.0
    fg_std: float = 1.0

    @property
    def causal_flops(self) -> float:
        """T^2*(d_qk+d_v) per head: Q K^T and C'V over the T^2/2 causal pairs, 2 flops per MAC."""
        return float(self.B * self.H) * self.T * self.T * (self.d_qk + self.d_v)

    @property
    def tokens(self) -> int:
        return self.B * self.T


@dataclasses.dataclass(frozen=True)
class StepWorkload:
    name: str
    B: int
    H: int
    d_qk: int
    d_v: int
    dtype: torch.dtype          # dtype of q, k, v, o and of h
    state_std: float = 0.1
    ig_mean: float = 0.0
    ig_std: float = 1.0
    fg_mean: float = 3.0
    fg_std: float = 1.0

    @property
    def state_bytes(self) -> int:
        return self.B * self.H * self.d_v * self.d_qk * 4


# The five workloads: a tiny fp32 check, two T=2048 layer shapes, a long
# context with slow forgetting, and one generation step over a large batch.
TINY = ParallelWorkload("tiny_B1_H1_T64_d16_f32", 1, 1, 64, 16, 16, torch.float32)
L125M = ParallelWorkload("mlstm125m_B8_H4_T2048_d384_bf16", 8, 4, 2048, 384, 384, torch.bfloat16)
L350M = ParallelWorkload("mlstm350m_B4_H4_T2048_d512_bf16", 4, 4, 2048, 512, 512, torch.bfloat16)
LONG = ParallelWorkload("long_B1_H4_T16384_d512_bf16", 1, 4, 16384, 512, 512, torch.bfloat16,
                        ig_mean=0.0, ig_std=2.0, fg_mean=5.0, fg_std=1.0)
STEP = StepWorkload("step_B256_H4_d512_bf16", 256, 4, 512, 512, torch.bfloat16)

PARALLEL_WORKLOADS: Dict[str, ParallelWorkload] = {w.name: w for w in (TINY, L125M, L350M, LONG)}


def _normal(g: torch.Generator, shape, mean: float, std: float) -> torch.Tensor:
    t = torch.empty(shape, dtype=torch.float32)
    t.normal_(mean=mean, std=std, generator=g)
    return t


def parallel_inputs(w: ParallelWorkload, seed: int = 0, *, B: Optional[int] = None,
                    H: Optional[int] = None, T: Optional[int] = None,
                    with_ogate: bool = False) -> Dict[str, torch.Tensor]:
    """q, k [B,H,T,d_qk], v [B,H,T,d_v] in ``w.dtype``; igate_pre, fgate_pre [B,H,T] fp32.

    ``B``/``H``/``T`` override the workload's sizes (same distributions).  With
    ``with_ogate`` an output-gate pre-activation ``ogate_pre`` [B,H,T,d_v] ~
    N(0,1) is drawn last, in ``w.dtype``.
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    T = w.T if T is None else T
    g = torch.Generator().manual_seed(seed)
    q = _normal(g, (B, H, T, w.d_qk), 0.0, w.qkv_std).to(w.dtype)
    k = _normal(g, (B, H, T, w.d_qk), 0.0, w.qkv_std).to(w.dtype)
    v = _normal(g, (B, H, T, w.d_v), 0.0, w.qkv_std).to(w.dtype)
    ig = _normal(g, (B, H, T), w.ig_mean, w.ig_std)
    fg = _normal(g, (B, H, T), w.fg_mean, w.fg_std)
    out = dict(q=q, k=k, v=v, igate_pre=ig, fgate_pre=fg)
    if with_ogate:
        out["ogate_pre"] = _normal(g, (B, H, T, w.d_v), 0.0, 1.0).to(w.dtype)
    return out


def step_inputs(w: StepWorkload, seed: int = 0, *, B: Optional[int] = None,
                H: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """State C [B,H,d_v,d_qk], n [B,H,d_qk], m [B,H] fp32 ~ N(0, state_std);
    q, k [B,H,d_qk], v, o [B,H,d_v] in ``w.dtype`` ~ N(0,1); igate_pre,
    fgate_pre [B,H] fp32."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    g = torch.Generator().manual_seed(seed)
    C = _normal(g, (B, H, w.d_v, w.d_qk), 0.0, w.state_std)
    n = _normal(g, (B, H, w.d_qk), 0.0, w.state_std)
    m = _normal(g, (B, H), 0.0, w.state_std)
    q = _normal(g, (B, H, w.d_qk), 0.0, 1.0).to(w.dtype)
    k = _normal(g, (B, H, w.d_qk), 0.0, 1.0).to(w.dtype)
    v = _normal(g, (B, H, w.d_v), 0.0, 1.0).to(w.dtype)
    o = _normal(g, (B, H, w.d_v), 0.0, 1.0).to(w.dtype)
    ig = _normal(g, (B, H), w.ig_mean, w.ig_std)
    fg = _normal(g, (B, H), w.fg_mean, w.fg_std)
    return dict(C=C, n=n, m=m, q=q, k=k, v=v, o=o, igate_pre=ig, fgate_pre=fg)


def step_seq_inputs(w: StepWorkload, L: int, seed: int = 0, *, B: Optional[int] = None,
                    H: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Like ``step_inputs`` with a token axis of length L: state C, n, m as
    there; q, k [B,H,L,d_qk], v, o [B,H,L,d_v] in ``w.dtype`` ~ N(0,1);
    igate_pre, fgate_pre [B,H,L] fp32."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    g = torch.Generator().manual_seed(seed)
    C = _normal(g, (B, H, w.d_v, w.d_qk), 0.0, w.state_std)
    n = _normal(g, (B, H, w.d_qk), 0.0, w.state_std)
    m = _normal(g, (B, H), 0.0, w.state_std)
    q = _normal(g, (B, H, L, w.d_qk), 0.0, 1.0).to(w.dtype)
    k = _normal(g, (B, H, L, w.d_qk), 0.0, 1.0).to(w.dtype)
    v = _normal(g, (B, H, L, w.d_v), 0.0, 1.0).to(w.dtype)
    o = _normal(g, (B, H, L, w.d_v), 0.0, 1.0).to(w.dtype)
    ig = _normal(g, (B, H, L), w.ig_mean, w.ig_std)
    fg = _normal(g, (B, H, L), w.fg_mean, w.fg_std)
    return dict(C=C, n=n, m=m, q=q, k=k, v=v, o=o, igate_pre=ig, fgate_pre=fg)


def sequence_inputs(B: int, H: int, T: int, d_qk: int, d_v: int, dtype: torch.dtype,
                    seed: int = 0, ig=(0.0, 1.0), fg=(3.0, 1.0), qkv_std: float = 1.0,
                    with_ogate: bool = False) -> Dict[str, torch.Tensor]:
    """Free-form sizes and gate distributions (for tests)."""
    w = ParallelWorkload("custom", B, H, T, d_qk, d_v, dtype, qkv_std=qkv_std,
                         ig_mean=ig[0], ig_std=ig[1], fg_mean=fg[0], fg_std=fg[1])
    return parallel_inputs(w, seed, with_ogate=with_ogate)
