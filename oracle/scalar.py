"""Pure-Python scalar attention for tiny inputs (lists of floats).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Written independently of ``attention.py`` so that the two can pin each other:
the forward pass is the textbook softmax with explicit loops, and the score
gradient uses the row form from the FlashAttention explainer
(wq-win.github.io), section 2, "backward needs only blocks and a few row
statistics": for one row with probabilities p, values v_j, output o and upstream
gradient g, dl/ds_j = p_j * g . (v_j - o).  The chain rule through
s_ij = alpha * q_i . k_j then gives dq_i = alpha sum_j ds_ij k_j and
dk_j = alpha sum_i ds_ij q_i, and o_i = sum_j p_ij v_j gives dv_j = sum_i p_ij g_i.
"""

from __future__ import annotations

import math

__all__ = ["forward", "backward"]


def _dot(a, b):
    return sum(x * y for x, y in zip(a, b))


def _row_probs(qi, k, scale, visible):
    s = [scale * _dot(qi, kj) if visible[j] else -math.inf for j, kj in enumerate(k)]
    finite = [x for x in s if x != -math.inf]
    if not finite:
        return [0.0] * len(k), -math.inf
    m = max(finite)
    e = [math.exp(x - m) if x != -math.inf else 0.0 for x in s]
    z = sum(e)
    return [x / z for x in e], m + math.log(z)


def forward(q, k, v, scale, causal=False):
    """q: N_q lists of d floats; k, v: N_k lists. Returns (o, lse)."""
    o, lse = [], []
    for i, qi in enumerate(q):
        visible = [(not causal) or j <= i for j in range(len(k))]
        p, l = _row_probs(qi, k, scale, visible)
        o.append([sum(p[j] * v[j][c] for j in range(len(k))) for c in range(len(v[0]))])
        lse.append(l)
    return o, lse


def backward(q, k, v, do, scale, causal=False):
    """Returns (dq, dk, dv) as lists of lists."""
    n_q, n_k, d, dv_dim = len(q), len(k), len(q[0]), len(v[0])
    dq = [[0.0] * d for _ in range(n_q)]
    dk = [[0.0] * d for _ in range(n_k)]
    dv = [[0.0] * dv_dim for _ in range(n_k)]
    for i, qi in enumerate(q):
        visible = [(not causal) or j <= i for j in range(n_k)]
        p, _ = _row_probs(qi, k, scale, visible)
        oi = [sum(p[j] * v[j][c] for j in range(n_k)) for c in range(dv_dim)]
        g = do[i]
        for j in range(n_k):
            ds = p[j] * sum(g[c] * (v[j][c] - oi[c]) for c in range(dv_dim))
            for c in range(d):
                dq[i][c] += scale * ds * k[j][c]
                dk[j][c] += scale * ds * qi[c]
            for c in range(dv_dim):
                dv[j][c] += p[j] * g[c]
    return dq, dk, dv
