"""Blockwise online-softmax recurrence in fp64 -- TEST INFRASTRUCTURE ONLY.

This restates, for one score row at a time, the statistics the pages fix:

* auturnal.com "From attention to IO-aware execution", §8: keep only the
  running max m, the denominator l and the not-yet-divided weighted sum u;
  when a new block arrives, align old and new to m' = max(m, m_block),
  rescale the old l and u by exp(m - m'), and emit u / l at the end.
* marketmaker.cc "Flash Attention and sequence length", "The Flash Attention
  algorithm": the same update written with the output kept normalised after
  every block (O <- O * l e^{m-m'} / l' + P V * e^{m_blk-m'} / l').
* The split combine (several partial (m, l, u) states over disjoint key
  ranges merged into one) is the same alignment applied to partial states.

Used only to pin the invariant "blockwise recurrence == full softmax" and the
combine formula; the GPU kernels are checked against ``oracle.sdpa``.
"""
from __future__ import annotations

import numpy as np


def full_softmax_row(s: np.ndarray, V: np.ndarray):
    """Two-pass reference for one row: returns (o, lse)."""
    m = np.max(s)
    p = np.exp(s - m)
    l = p.sum()
    return (p[:, None] * V).sum(0) / l, m + np.log(l)


def deferred(s: np.ndarray, V: np.ndarray, cuts):
    """(m, l, u) over the key blocks delimited by ``cuts`` (sorted interior
    split points); normalisation deferred to the end.  Returns (o, lse)."""
    edges = [0] + list(cuts) + [len(s)]
    m, l, u = -np.inf, 0.0, np.zeros(V.shape[1])
    for a, b in zip(edges[:-1], edges[1:]):
        if b <= a:
            continue
        sb = s[a:b]
        m_new = max(m, float(np.max(sb)))
        if m_new == -np.inf:  # nothing visible yet
            continue
        alpha = 0.0 if m == -np.inf else np.exp(m - m_new)
        p = np.exp(sb - m_new)
        l = l * alpha + p.sum()
        u = u * alpha + (p[:, None] * V[a:b]).sum(0)
        m = m_new
    return u / l, m + np.log(l)


def normalised(s: np.ndarray, V: np.ndarray, cuts):
    """The per-block-normalised form: O stays a convex combination after
    every block.  Returns (o, lse)."""
    edges = [0] + list(cuts) + [len(s)]
    m, l, O = -np.inf, 0.0, np.zeros(V.shape[1])
    for a, b in zip(edges[:-1], edges[1:]):
        if b <= a:
            continue
        sb = s[a:b]
        m_blk = float(np.max(sb))
        if m_blk == -np.inf:
            continue
        P = np.exp(sb - m_blk)
        l_blk = P.sum()
        m_new = max(m, m_blk)
        a_old = 0.0 if m == -np.inf else np.exp(m - m_new)
        a_blk = np.exp(m_blk - m_new)
        l_new = l * a_old + l_blk * a_blk
        O = O * (l * a_old / l_new) + (P[:, None] * V[a:b]).sum(0) * (a_blk / l_new)
        m, l = m_new, l_new
    return O, m + np.log(l)


def partial_state(s: np.ndarray, V: np.ndarray):
    """(m, l, u) of one key range, as one split of a split-KV decode."""
    if len(s) == 0 or np.max(s) == -np.inf:
        return -np.inf, 0.0, np.zeros(V.shape[1])
    m = float(np.max(s))
    p = np.exp(s - m)
    return m, float(p.sum()), (p[:, None] * V).sum(0)


def combine(states):
    """Merge partial states: M = max m_s, o = sum e^{m_s-M} u_s / sum
    e^{m_s-M} l_s, lse = M + ln sum e^{m_s-M} l_s."""
    M = max(st[0] for st in states)
    if M == -np.inf:
        d = states[0][2].shape[0]
        return np.zeros(d), -np.inf
    L = 0.0
    U = np.zeros_like(states[0][2])
    for m, l, u in states:
        if m == -np.inf:
            continue
        w = np.exp(m - M)
        L += w * l
        U += w * u
    return U / L, M + np.log(L)
