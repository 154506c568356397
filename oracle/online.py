"""Tile-merge algorithms behind the fast method, for one query row, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

``online_merge`` follows the FlashAttention explainer (wq-win.github.io),
section 2: a row's scores arrive block by block; the state is the running
maximum m, the running sum of exponentials l and the unnormalised output u. A
new block (s_new, V_new) updates them as

    m' = max(m, max s_new)
    l' = e^(m - m') l + sum_j e^(s_new_j - m')
    u' = e^(m - m') u + sum_j e^(s_new_j - m') V_new_j

and the output is u / l. The same recurrence is the one of the FlashAttention-4
summary (papercache.org), section 3.1.4, with O in place of u.

``online_merge_lazy`` is the conditional-rescaling variant of that same section:
the old state is rescaled only when the maximum grows by more than tau, with tau
measured in powers of two (tau = log2(256) = 8 means a factor of 256); otherwise
the stale maximum is kept and the block's exponentials are taken against it. The
final division by l gives the same output.

``blockwise_average_merge`` is the incorrect merge the explainer warns about
(softmax each block on its own, then average the block outputs). It exists only
so the tests can show that it differs from the definition.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = ["online_merge", "online_merge_lazy", "blockwise_average_merge"]


def online_merge(s_blocks, v_blocks):
    """Returns (o, m, l) after merging the blocks in order."""
    m = -math.inf
    l = 0.0
    u = None
    for s, vb in zip(s_blocks, v_blocks):
        s = np.asarray(s, dtype=np.float64)
        vb = np.asarray(vb, dtype=np.float64)
        if u is None:
            u = np.zeros(vb.shape[1:], dtype=np.float64)
        m_new = max(m, float(np.max(s))) if s.size else m
        if m_new == -math.inf:
            continue  # nothing visible yet
        c = math.exp(m - m_new)  # e^(m - m'); zero on the first visible block
        e = np.exp(s - m_new)
        l = c * l + float(np.sum(e))
        u = c * u + e @ vb
        m = m_new
    o = u / l if l > 0 else np.zeros_like(u)
    return o, m, l


def online_merge_lazy(s_blocks, v_blocks, tau=8.0):
    """Conditional rescaling. Returns (o, m_used, l, n_rescales); l is relative
    to m_used, the maximum actually used for the exponentials."""
    m_used = -math.inf
    l = 0.0
    u = None
    n_rescales = 0
    log2e = 1.0 / math.log(2.0)
    for s, vb in zip(s_blocks, v_blocks):
        s = np.asarray(s, dtype=np.float64)
        vb = np.asarray(vb, dtype=np.float64)
        if u is None:
            u = np.zeros(vb.shape[1:], dtype=np.float64)
        m_blk = float(np.max(s)) if s.size else -math.inf
        m_new = max(m_used, m_blk)
        if m_new == -math.inf:
            continue
        if (m_new - m_used) * log2e > tau:  # the maximum moved by more than 2^tau
            c = math.exp(m_used - m_new)
            l *= c
            u = u * c
            m_used = m_new
            n_rescales += 1
        e = np.exp(s - m_used)  # may exceed 1, by at most 2^tau
        l += float(np.sum(e))
        u = u + e @ vb
    o = u / l if l > 0 else np.zeros_like(u)
    return o, m_used, l, n_rescales


def blockwise_average_merge(s_blocks, v_blocks):
    """The wrong merge: independent softmax per block, outputs averaged."""
    outs = []
    for s, vb in zip(s_blocks, v_blocks):
        s = np.asarray(s, dtype=np.float64)
        e = np.exp(s - np.max(s))
        outs.append((e / np.sum(e)) @ np.asarray(vb, dtype=np.float64))
    return np.mean(outs, axis=0)
