"""Per-tensor FP8 attention, the comparison baseline of the FP8 claim -- TEST
INFRASTRUCTURE ONLY (imported by tests, never by the CUDA library).

"FlashAttention Primer", section "FlashAttention-3: Hopper asynchrony and FP8",
and "Flash Attention" (aiwiki.ai), section "FlashAttention-3": the block-scaled,
rotated FP8 forward is reported at 2.6x lower numerical error than a baseline
FP8 attention that uses one scale per tensor.  This module is that baseline,
in the plainest form the pages allow: Q, K and V each quantized to e4m3 with a
single scale (largest magnitude -> 448, no rotation), scores and softmax in
fp64, and the probabilities rounded to e4m3 before the P V product (as an FP8
attention kernel feeds P to its second FP8 matrix product).
"""
from __future__ import annotations

import numpy as np

from . import _as_f32, e4m3_decode, e4m3_encode


def _per_tensor(x: np.ndarray) -> np.ndarray:
    amax = np.float32(np.abs(x).max())
    if amax == 0:
        return np.zeros(x.shape)
    f = np.float32(448.0) / amax
    return e4m3_decode(e4m3_encode(x * f)) * (float(amax) / 448.0)


def forward(q, k, v, causal: bool, scale: float) -> np.ndarray:
    """O of the per-tensor FP8 baseline for q [B,Hq,N,d], k, v [B,Hkv,N,d]."""
    q, k, v = (np.ascontiguousarray(_as_f32(t)) for t in (q, k, v))
    qh, kh, vh = _per_tensor(q), _per_tensor(k), _per_tensor(v)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    o = np.empty((B, Hq, N, d))
    mask = np.tril(np.ones((N, N), dtype=bool)) if causal else np.ones((N, N), dtype=bool)
    for b in range(B):
        for h in range(Hq):
            g = h * Hkv // Hq
            s = scale * (qh[b, h] @ kh[b, g].T)
            s = np.where(mask, s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            l = p.sum(axis=1, keepdims=True)
            p8 = e4m3_decode(e4m3_encode(p.astype(np.float32)))
            o[b, h] = (p8 @ vh[b, g]) / l
    return o
