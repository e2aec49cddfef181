"""The method's softmax and tiling algorithm in fp64 numpy, in the pages' order and notation.

TEST INFRASTRUCTURE (part of the oracle package; see ``oracle/__init__.py``).

These functions restate, step by step, what the pages describe, so that tests can show the
tiled algorithm reaches the plain definition that ``attn_oracle.c`` computes:

* ``softmax_three_pass``: "FlashAttention 优化原理与实现要点解析" §4.1 -- the softmax
  definition and its three passes (maximum, sum of shifted exponentials, normalisation).
* ``online_softmax_stream``: "FlashAttention V2 核心原理与架构设计" §2.1 -- one element at a
  time, keep the running maximum m and running sum l; on each element the old l is rescaled
  by e^{m - m_new} and e^{x_i - m_new} is added; the result is e^{x - m} / l. (The page's
  printed update is garbled; this is the reading that makes it a softmax.)
* ``online_softmax``: "FlashAttention 优化原理与实现要点解析" §4.2 -- blocks of the vector:
  each block gives a local maximum m_new and local sum l_new; the global values merge as
  m = max(m_old, m_new), l = l_old e^{m_old - m} + l_new e^{m_new - m}.
* ``blockwise_attention``: same page §4.3 and §5 -- for each Q block, for each K/V block:
  local scores, local max and sum, update the global m and l, rescale the old O by
  e^{m_old - m} and add P_block V_block (P_block taken relative to the updated m), and after
  the last K/V block divide O by l (§6: numerator and denominator kept apart until the end).
  Causal (§7): a query attends to keys at positions <= its own; K/V blocks that lie
  entirely above the diagonal are skipped. §8's padding and sliding-window masks take the
  same form: a per-row key interval, and blocks with no allowed key are skipped.
"""
from __future__ import annotations

import math

import numpy as np


def softmax_three_pass(x) -> np.ndarray:
    """Softmax of a 1-D vector by the three passes: max, shifted sum, normalise."""
    x = np.asarray(x, dtype=np.float64)
    m = -math.inf
    for xi in x:                       # pass 1
        m = max(m, float(xi))
    l = 0.0
    for xi in x:                       # pass 2
        l += math.exp(float(xi) - m)
    return np.array([math.exp(float(xi) - m) / l for xi in x])   # pass 3


def online_softmax_stream(x) -> np.ndarray:
    """Softmax with one running (m, l) pair updated element by element."""
    x = np.asarray(x, dtype=np.float64)
    m, l = -math.inf, 0.0
    for xi in x:
        m_new = max(m, float(xi))
        l = l * math.exp(m - m_new) + math.exp(float(xi) - m_new)
        m = m_new
    return np.exp(x - m) / l


def online_softmax(x, block_sizes) -> tuple[np.ndarray, float, float]:
    """Softmax of ``x`` from per-block statistics merged block by block.

    ``block_sizes`` lists the lengths of consecutive blocks (they must add up to len(x)).
    Returns (softmax(x), m, l) with m the global maximum and l = sum_j e^{x_j - m}.
    """
    x = np.asarray(x, dtype=np.float64)
    if sum(block_sizes) != x.size or any(bs <= 0 for bs in block_sizes):
        raise ValueError("block sizes must be positive and cover x")
    m, l = -math.inf, 0.0
    start = 0
    for bs in block_sizes:
        blk = x[start:start + bs]
        start += bs
        m_blk = float(blk.max())                      # local maximum of the new block
        l_blk = float(np.exp(blk - m_blk).sum())      # local sum w.r.t. the local maximum
        m_new = max(m, m_blk)
        l = l * math.exp(m - m_new) + l_blk * math.exp(m_blk - m_new)
        m = m_new
    return np.exp(x - m) / l, m, l


def blockwise_attention(q, k, v, Br: int, Bc: int, causal: bool, scale: float,
                        window=(-1, -1), kv_len=None):
    """Tiled attention with online softmax, fp64, for one head.

    q: [Nq, d], k, v: [Nk, d] float arrays with Nk >= Nq; query i sits at position
    i + Nk - Nq. ``window`` = (left, right) bounds the keys a query at position p sees
    (j >= p - left, j <= p + right; -1 = no bound); ``kv_len`` (default Nk): keys at or past it
    do not exist. K/V blocks with no allowed key for any row of the Q block are skipped.
    Returns (O [Nq, d], LSE [Nq]) with LSE = m + ln l; rows with no allowed key get O = 0 and
    LSE = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Nq, d = q.shape
    N = k.shape[0]
    offset = N - Nq
    kv_len = N if kv_len is None else kv_len
    left, right = window
    O = np.zeros((Nq, d))
    LSE = np.zeros(Nq)
    for i0 in range(0, Nq, Br):                       # outer loop: Q blocks
        rows = np.arange(i0, min(i0 + Br, Nq))
        Qi = q[rows]
        pos = rows + offset                           # positions of these queries
        m = np.full(rows.size, -math.inf)
        l = np.zeros(rows.size)
        Oi = np.zeros((rows.size, d))
        for j0 in range(0, N, Bc):                    # inner loop: K/V blocks
            cols = np.arange(j0, min(j0 + Bc, N))
            allowed = cols[None, :] < kv_len
            if causal:
                allowed = allowed & (cols[None, :] <= pos[:, None])
            if left >= 0:
                allowed = allowed & (cols[None, :] >= pos[:, None] - left)
            if right >= 0:
                allowed = allowed & (cols[None, :] <= pos[:, None] + right)
            if not allowed.any():
                continue                              # block fully masked: skipped
            S = np.where(allowed, scale * (Qi @ k[cols].T), -math.inf)   # local scores
            m_blk = S.max(axis=1)                     # local maximum
            m_new = np.maximum(m, m_blk)
            # rows whose keys so far are all masked keep m = -inf; shift by 0 instead
            shift = np.where(np.isfinite(m_new), m_new, 0.0)
            P = np.exp(S - shift[:, None])            # block probabilities w.r.t. new max
            alpha = np.exp(m - shift)                 # e^{m_old - m}
            l = l * alpha + P.sum(axis=1)
            Oi = Oi * alpha[:, None] + P @ v[cols]
            m = m_new
        with np.errstate(divide="ignore", invalid="ignore"):
            O[rows] = np.where(l[:, None] > 0, Oi / np.where(l > 0, l, 1.0)[:, None], 0.0)
            LSE[rows] = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -math.inf)
    return O, LSE
