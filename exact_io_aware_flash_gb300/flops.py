"""Algorithmic FLOP and byte counts of one attention call (host-side bookkeeping).

Forward: two N x N x d matrix products per head (S = Q K^T and O = P V), i.e.
4 * B * H * N^2 * d FLOPs, halved for causal attention.  This is the count the
sm75 README's throughput tables use ("flash-attention-sm75", section
"Performance": e.g. d=64, N=1024, B*H=8 in 1.586 ms is 1.35 TFLOPS); the tests
pin it against those printed tables.

Backward: five N x N x d matrix products per head (recomputed S, dV = P^T dO,
dP = dO V^T, dQ = dS K, dK = dS^T Q), i.e. 2.5 x the forward count.

Bytes: each tensor read or written once -- the IO-optimal traffic the tiled
schedule aims at ("FlashAttention Primer", Figure 2: Q, K, V stream in, O is
written, no N x N matrix reaches HBM).
"""
from __future__ import annotations


def forward_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    f = 4.0 * B * H * N * N * d
    return f / 2.0 if causal else f


def backward_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    return 2.5 * forward_flops(B, H, N, d, causal)


def window_pairs(N: int, window: int) -> int:
    """Visible (query, key) pairs of a causal sliding window of ``window`` keys
    over N positions (query i sees keys i - window < k <= i): sum_i min(i + 1, window)."""
    w = min(window, N)
    return w * (w + 1) // 2 + (N - w) * w


def forward_flops_window(B: int, H: int, N: int, d: int, window: int) -> float:
    """Two products of 2*d FLOPs per visible pair (the work a block-sparse
    schedule that skips empty blocks needs, "Flash Attention" (aiwiki.ai),
    section "Block-sparse FlashAttention")."""
    return 4.0 * d * B * H * window_pairs(N, window)


def backward_flops_window(B: int, H: int, N: int, d: int, window: int) -> float:
    return 2.5 * forward_flops_window(B, H, N, d, window)


def forward_bytes(B: int, Hq: int, Hkv: int, N: int, d: int, elt: int = 2) -> int:
    """Q, K, V read + O written (16-bit) + LSE written (fp32)."""
    return elt * N * d * B * (2 * Hq + 2 * Hkv) + 4 * B * Hq * N


def backward_bytes(B: int, Hq: int, Hkv: int, N: int, d: int, elt: int = 2) -> int:
    """Q, K, V, O, dO read + dQ, dK, dV written (16-bit) + LSE read, D written and read (fp32)."""
    return elt * N * d * B * (4 * Hq + 4 * Hkv) + 4 * B * Hq * N * 3


def materialised_score_bytes(N: int, heads: int = 1, elt: int = 2) -> int:
    """Bytes a standard schedule needs to hold S and P for ``heads`` heads.

    "FlashAttention Primer", section "Why attention is quadratic": two N x N
    matrices of ``elt``-byte entries per head.
    """
    return 2 * N * N * elt * heads
