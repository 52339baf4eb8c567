"""Tiled evaluation of attention by the online-softmax merge -- TEST INFRASTRUCTURE.

This is a second, independent fp64 evaluator used only to pin the naive oracle: it walks the
keys in column blocks of arbitrary widths and merges per-block statistics (m, l, U) with the
recurrence of "FlashAttention · InkStack", section 1.1.2 "Online Softmax":

    m_new = max(m_old, m~)
    l_new = e^(m_old - m_new) l_old + e^(m~ - m_new) l~
    U_new = e^(m_old - m_new) U_old + e^(m~ - m_new) U~,      o = U / l

and the stored statistic L = m + log l of section 2.1 of the same page.  Equality with the
two-pass safe softmax of the naive oracle is the identity the method rests on
(e^(x - m_new) = e^(x - m_old) e^(m_old - m_new), "FlashAttention 深度解析", section 2.2), and
it fixes the direction of the rescale factor alpha = e^(m_old - m_new) <= 1.

Also here: the FlashAttention-2 form that keeps the unnormalised numerator and divides once at
the end ("FlashAttention · InkStack", section 2.1), used by the same pins.
"""
from __future__ import annotations

import numpy as np


def block_stats(x: np.ndarray, v: np.ndarray):
    """Statistics of one column block: local max, local sum of exps, local unnormalised PV."""
    m = np.max(x)
    e = np.exp(x - m)
    return m, np.sum(e), e @ v


def merge(state, block):
    """Associative merge of (m, l, U) for the block recurrence."""
    m_old, l_old, u_old = state
    m_blk, l_blk, u_blk = block
    m_new = max(m_old, m_blk)
    a_old = np.exp(m_old - m_new) if np.isfinite(m_old) else 0.0
    a_blk = np.exp(m_blk - m_new)
    return m_new, a_old * l_old + a_blk * l_blk, a_old * u_old + a_blk * u_blk


def row_online(x: np.ndarray, v: np.ndarray, splits):
    """Attention output and LSE of one row of logits ``x`` over values ``v`` [n, d]."""
    state = (-np.inf, 0.0, np.zeros(v.shape[1]))
    edges = [0] + list(splits) + [x.size]
    for a, b in zip(edges[:-1], edges[1:]):
        if b > a:
            state = merge(state, block_stats(x[a:b], v[a:b]))
    m, l, u = state
    return u / l, m + np.log(l)


def row_deferred(x: np.ndarray, v: np.ndarray, block: int):
    """FlashAttention-2 form: O~' = alpha O~ + P~ V per block, normalised once at the end."""
    m = -np.inf
    l = 0.0
    acc = np.zeros(v.shape[1])
    for a in range(0, x.size, block):
        xb = x[a:a + block]
        m_new = max(m, np.max(xb))
        alpha = np.exp(m - m_new) if np.isfinite(m) else 0.0
        p = np.exp(xb - m_new)
        l = alpha * l + np.sum(p)
        acc = alpha * acc + p @ v[a:a + block]
        m = m_new
    return acc / l, m + np.log(l)


def attention_online(q, k, v, scale: float, causal: bool, block_edges_fn):
    """Whole-tensor tiled evaluation; ``block_edges_fn(n_keys)`` picks the column splits."""
    B, H, N, d = q.shape
    o = np.empty((B, H, N, d))
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            logits = scale * (q[b, h] @ k[b, h].T)
            for i in range(N):
                n = i + 1 if causal else N
                o[b, h, i], lse[b, h, i] = row_online(logits[i, :n], v[b, h, :n],
                                                      block_edges_fn(n))
    return o, lse
