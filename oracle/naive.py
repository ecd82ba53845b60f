"""Materialising fp64 attention in numpy -- TEST INFRASTRUCTURE ONLY (see ``oracle``).

This is the "standard attention" schedule the pages contrast FlashAttention
with: the full N x N score matrix S and probability matrix P are formed, then
O = P V ("FlashAttention Primer", Figure 2, left column; "Flash Attention"
(aiwiki.ai), section "Forward pass", the unfused three-line expression).  It is
an independent implementation of the same definition as ``oracle.c`` and is
used to cross-check it on tiny inputs.

The backward is written in matrix form from the chain rule of the definition:
  dV = P^T dO, dP = dO V^T, dS = P o (dP - rowsum(P o dP)),
  dQ = scale dS K, dK = scale dS^T Q.
Note rowsum(P o dP) is computed here directly from P and dP, not as
rowsum(dO o O): the two agree in exact arithmetic, and the tests check that.
"""
from __future__ import annotations

import numpy as np


def _expand_kv(x: np.ndarray, Hq: int) -> np.ndarray:
    """Repeat each KV head for its contiguous group of query heads: head h -> floor(h*Hkv/Hq)."""
    Hkv = x.shape[1]
    idx = (np.arange(Hq) * Hkv) // Hq
    return x[:, idx]


def scores(q, k, scale, causal, window=None):
    """Scores with future keys (causal) and, with a window W, keys more than
    W - 1 positions in the past set to -inf."""
    q = np.asarray(q, dtype=np.float64)
    k = _expand_kv(np.asarray(k, dtype=np.float64), q.shape[1])
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    if causal or window is not None:
        n = q.shape[2]
        i = np.arange(n)[:, None]
        j = np.arange(n)[None, :]
        mask = j > i
        if window is not None:
            mask |= j <= i - window
        s = np.where(mask, -np.inf, s)
    return s


def softmax(s):
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


def forward(q, k, v, causal, scale, window=None):
    s = scores(q, k, scale, causal, window)
    p = softmax(s)
    vv = _expand_kv(np.asarray(v, dtype=np.float64), p.shape[1])
    o = np.einsum("bhij,bhjd->bhid", p, vv)
    m = s.max(axis=-1)
    lse = m + np.log(np.exp(s - m[..., None]).sum(axis=-1))
    return o, lse, p


def backward(q, k, v, dO, causal, scale, window=None):
    q = np.asarray(q, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    B, Hq, N, d = q.shape
    Hkv = np.asarray(k).shape[1]
    kk = _expand_kv(np.asarray(k, dtype=np.float64), Hq)
    vv = _expand_kv(np.asarray(v, dtype=np.float64), Hq)
    _, _, p = forward(q, k, v, causal, scale, window)
    dv_e = np.einsum("bhij,bhid->bhjd", p, dO)
    dp = np.einsum("bhid,bhjd->bhij", dO, vv)
    rs = (p * dp).sum(axis=-1, keepdims=True)
    ds = p * (dp - rs)
    dq = scale * np.einsum("bhij,bhjd->bhid", ds, kk)
    dk_e = scale * np.einsum("bhij,bhid->bhjd", ds, q)
    g = Hq // Hkv
    dk = dk_e.reshape(B, Hkv, g, N, d).sum(axis=2)
    dv = dv_e.reshape(B, Hkv, g, N, d).sum(axis=2)
    return dq, dk, dv, rs[..., 0]
