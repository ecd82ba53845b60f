"""The pages' tiled online-softmax recurrences in numpy fp64 -- TEST INFRASTRUCTURE ONLY.

Two forms, each written from its page's description for one head (q [N,d],
k, v [N,d]), with key/value blocks of caller-chosen sizes:

* ``fa1_form``: "FlashAttention Primer", section "FlashAttention-1", the
  online-softmax equation and Figure 4.  The state (m, l, O) is kept
  unnormalised; a new block contributes P~ = exp(S_blk - rowmax S_blk) with its
  own row sum l_blk, the old state is scaled by alpha = exp(m - m') and the block
  by beta = exp(rowmax S_blk - m'), where m' = max(m, rowmax S_blk).  The output
  is O / l at the end.

* ``fa2_form``: "Flash Attention" (aiwiki.ai), section "Online softmax", and the
  concept-page forward loop ("FlashAttention", praveentn.live, section "The fix:
  tiling + online softmax"): P = exp(S_blk - m_new) directly against the new
  running max, l and O are scaled by exp(m_old - m_new), and O is divided by l
  once after the last block.

Both also return the per-row log-sum-exp m + ln l.  Causal masking sets future
scores to -inf before the exponentials ("Flash Attention", section "Online
softmax", last paragraph).  Query rows are processed all at once (one query
block), which is allowed because rows are independent.
"""
from __future__ import annotations

import numpy as np


def _blocks(n, sizes):
    start = 0
    for s in sizes:
        if start >= n:
            break
        yield start, min(n, start + s)
        start += s
    if start < n:
        yield start, n


def _block_scores(q, k, lo, hi, scale, causal):
    s = scale * (q @ k[lo:hi].T)
    if causal:
        rows = np.arange(q.shape[0])[:, None]
        cols = np.arange(lo, hi)[None, :]
        s = np.where(cols > rows, -np.inf, s)
    return s


def fa1_form(q, k, v, scale, causal=False, block_sizes=(64,)):
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    n, d = q.shape
    m = np.full(n, -np.inf)
    l = np.zeros(n)
    o = np.zeros((n, d))
    sizes = list(block_sizes) * (k.shape[0] // max(1, min(block_sizes)) + 1)
    for lo, hi in _blocks(k.shape[0], sizes):
        s = _block_scores(q, k, lo, hi, scale, causal)
        m_blk = s.max(axis=1)
        m_new = np.maximum(m, m_blk)
        # rows whose block is fully masked contribute nothing
        valid = np.isfinite(m_blk)
        p_t = np.where(valid[:, None], np.exp(s - np.where(valid, m_blk, 0.0)[:, None]), 0.0)
        l_blk = p_t.sum(axis=1)
        alpha = np.where(np.isfinite(m), np.exp(m - m_new), 0.0)
        beta = np.where(valid, np.exp(np.where(valid, m_blk, 0.0) - m_new), 0.0)
        l = alpha * l + beta * l_blk
        o = alpha[:, None] * o + beta[:, None] * (p_t @ v[lo:hi])
        m = m_new
    return o / l[:, None], m + np.log(l)


def fa2_form(q, k, v, scale, causal=False, block_sizes=(64,)):
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    n, d = q.shape
    m = np.full(n, -np.inf)
    l = np.zeros(n)
    o = np.zeros((n, d))
    sizes = list(block_sizes) * (k.shape[0] // max(1, min(block_sizes)) + 1)
    for lo, hi in _blocks(k.shape[0], sizes):
        s = _block_scores(q, k, lo, hi, scale, causal)
        m_new = np.maximum(m, s.max(axis=1))
        p = np.exp(s - m_new[:, None])
        corr = np.where(np.isfinite(m), np.exp(m - m_new), 0.0)
        l = corr * l + p.sum(axis=1)
        o = corr[:, None] * o + p @ v[lo:hi]
        m = m_new
    return o / l[:, None], m + np.log(l)
