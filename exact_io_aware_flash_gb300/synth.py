"""Seeded synthetic inputs for attention workloads.

This module holds no attention arithmetic: it only draws tensors.  Both the
CUDA path's callers and the fp64 oracle's callers take their inputs from here,
so the two always see the same rounded values.

Recipe (the pages' workloads are synthetic shapes with iid N(0,1) entries; the
sm75 README's usage example draws Q, K, V with ``torch.randn`` of shape
(B, H, N, d), "flash-attention-sm75", section "Usage"):

* one CPU ``torch.Generator`` seeded with ``seed``;
* fp32 standard-normal draws in the order Q, K, V, dO, each of shape
  [B, H, N, d] (H = Hq for Q and dO, Hkv for K and V), multiplied by
  ``q_scale`` for Q only (``q_scale`` > 1 widens the score range so that the
  running row maximum moves often and the rescaling path is exercised);
* cast to the requested 16-bit dtype.  Everyone consumes the rounded values.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Shape:
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv


def make_inputs(shape: Shape, dtype: str, seed: int, with_dO: bool = True,
                q_scale: float = 1.0):
    """Return a dict of CPU tensors q, k, v (and dO) in ``dtype`` ("fp16" or "bf16")."""
    if dtype not in DTYPES:
        raise ValueError(f"dtype must be one of {sorted(DTYPES)}")
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    s = shape
    out = {}
    out["q"] = torch.randn(s.B, s.Hq, s.N, s.d, generator=g, dtype=torch.float32) * q_scale
    out["k"] = torch.randn(s.B, s.Hkv, s.N, s.d, generator=g, dtype=torch.float32)
    out["v"] = torch.randn(s.B, s.Hkv, s.N, s.d, generator=g, dtype=torch.float32)
    if with_dO:
        out["dO"] = torch.randn(s.B, s.Hq, s.N, s.d, generator=g, dtype=torch.float32)
    return {name: t.to(DTYPES[dtype]).contiguous() for name, t in out.items()}


# The five workloads of the method's evaluation, by what they are.
WORKLOADS = {
    "single_head_fwd_n128_d64_fp16": dict(shape=Shape(1, 1, 1, 128, 64), dtype="fp16",
                                          causal=(False,), seed=1001),
    "fwd_b1_h8_n1024_d64_fp16": dict(shape=Shape(1, 8, 8, 1024, 64), dtype="fp16",
                                     causal=(False, True), seed=1002),
    "fwd_b4_h16_n4096_d128_bf16_causal": dict(shape=Shape(4, 16, 16, 4096, 128), dtype="bf16",
                                              causal=(True,), seed=1003),
    "gqa_fwd_b2_hq32_hkv8_n8192_d128_bf16_causal": dict(shape=Shape(2, 32, 8, 8192, 128),
                                                        dtype="bf16", causal=(True,), seed=1004),
}


def backward_sweep_shape(N: int) -> Shape:
    """Backward sweep: H=16, d=128, bf16, causal, with B*N held at 32768."""
    if 32768 % N:
        raise ValueError("N must divide 32768")
    return Shape(32768 // N, 16, 16, N, 128)


BACKWARD_SWEEP_N = (512, 2048, 4096, 8192, 16384)
