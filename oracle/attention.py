"""Plain float64 definition of exact softmax attention and its gradient.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What is computed, per (batch, query head), following the pages:

* FlashAttention-4 (papercache.org summary), section 2.1 "Multi-head attention":
  O = softmax(alpha * Q K^T) V with the softmax taken row by row, alpha = 1/sqrt(d)
  by default; the row maximum is subtracted for numerical stability. The backward
  pass of the same section: dV = P^T dO, dP = dO V^T, dS = dsoftmax(dP) with
  ds = (diag(p) - p p^T) dp per row, dQ = alpha dS K, dK = alpha dS^T Q.
* FlashAttention explainer (wq-win.github.io), section 2: the row form of the
  softmax gradient, dl/ds_j = p_j g^T (v_j - o), which is the same thing as
  P o (dP - D) with D = rowsum(dO o O).
* FlashAttention notes (xwysyy.cn), "safe softmax": m = max_i x_i,
  f = exp(x - m), l = sum f, softmax = f / l. The log-sum-exp saved for the
  backward pass is m + ln(l) (the pages keep m and l per row).

Masks are additive minus infinity: causal means key j is visible to query i only
when j <= i; variable-length inputs are packed sequences described by cumulative
offsets, and a query only sees keys of its own sequence. A row that sees no key
at all gets O = 0 and LSE = -inf, and contributes no gradient.

Grouped-query attention: query head h reads KV head h // (H_q / H_kv); the
gradients of a KV head are the sums over the query heads that read it.

S and P are materialised in full for every row. For very long sequences the
query rows are processed in groups of at most ``row_block`` rows; every row still
sees all of its keys at once (this is not an online softmax), and only the
order in which the dK / dV sums are added changes.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "visible_mask",
    "head_forward",
    "head_backward",
    "attention_forward",
    "attention_backward",
]


def visible_mask(rows: np.ndarray, n_k: int, causal: bool) -> np.ndarray:
    """Boolean [len(rows), n_k]: True where query ``rows[i]`` may see key j."""
    keys = np.arange(n_k)
    if causal:
        return keys[None, :] <= np.asarray(rows)[:, None]
    return np.ones((len(rows), n_k), dtype=bool)


def _softmax_rows(s: np.ndarray):
    """Safe softmax of each row of s (entries may be -inf). Returns (P, lse)."""
    m = np.max(s, axis=1, keepdims=True)
    dead = ~np.isfinite(m)  # every key masked
    m_safe = np.where(dead, 0.0, m)
    f = np.exp(s - m_safe)
    l = np.sum(f, axis=1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(dead, 0.0, f / np.where(dead, 1.0, l))
        lse = np.where(dead[:, 0], -np.inf, m_safe[:, 0] + np.log(np.where(dead[:, 0], 1.0, l[:, 0])))
    return p, lse


def head_forward(q, k, v, scale, causal=False, rows=None, row_block=2048):
    """One head. q [N_q, d], k [N_k, d], v [N_k, d_v] float64.

    ``rows`` selects which query rows to compute (default: all); the result
    then has one row per selected query. Returns (O, LSE)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if rows is None:
        rows = np.arange(q.shape[0])
    rows = np.asarray(rows)
    o = np.zeros((len(rows), v.shape[1]))
    lse = np.zeros(len(rows))
    for r0 in range(0, len(rows), row_block):
        rr = rows[r0:r0 + row_block]
        s = scale * (q[rr] @ k.T)
        s = np.where(visible_mask(rr, k.shape[0], causal), s, -np.inf)
        p, lse[r0:r0 + len(rr)] = _softmax_rows(s)
        o[r0:r0 + len(rr)] = p @ v
    return o, lse


def head_backward(q, k, v, do, scale, causal=False, row_block=2048, return_ds=False):
    """One head, all rows. Returns dict with dq, dk, dv, o, lse (and ds, dp, p
    when ``return_ds`` and the head fits one row block)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    n_q = q.shape[0]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    o = np.zeros((n_q, v.shape[1]))
    lse = np.zeros(n_q)
    out = {}
    for r0 in range(0, n_q, row_block):
        rr = np.arange(r0, min(n_q, r0 + row_block))
        s = scale * (q[rr] @ k.T)
        s = np.where(visible_mask(rr, k.shape[0], causal), s, -np.inf)
        p, lse[rr] = _softmax_rows(s)
        o[rr] = p @ v
        dp = do[rr] @ v.T                                  # dP = dO V^T
        dvec = np.sum(do[rr] * o[rr], axis=1, keepdims=True)  # D = rowsum(dO o O)
        ds = p * (dp - dvec)                               # (diag(p) - p p^T) dp, row by row
        dq[rr] = scale * (ds @ k)                          # dQ = alpha dS K
        dk += scale * (ds.T @ q[rr])                       # dK = alpha dS^T Q
        dv += p.T @ do[rr]                                 # dV = P^T dO
        if return_ds and n_q <= row_block:
            out.update(ds=ds, dp=dp, p=p)
    out.update(dq=dq, dk=dk, dv=dv, o=o, lse=lse)
    return out


# ---------------------------------------------------------------------------
# Whole-tensor wrappers. Fixed length: q [B, N_q, H_q, d], k/v [B, N_k, H_kv, d],
# lse [B, H_q, N_q]. Packed variable length (cu_seqlens given): q [T, H_q, d],
# k/v [T, H_kv, d], lse [H_q, T], sequence s = rows cu[s]:cu[s+1].
# ``pairs`` restricts the work to a list of (b, h) (query head) pairs; outputs
# for other pairs are left as NaN.


def _segments(q, cu_seqlens):
    if cu_seqlens is None:
        return [(b, None) for b in range(q.shape[0])]
    cu = np.asarray(cu_seqlens)
    return [(s, (int(cu[s]), int(cu[s + 1]))) for s in range(len(cu) - 1)]


def _head_views(x, b, seg, h):
    if seg is None:
        return x[b, :, h, :]
    return x[seg[0]:seg[1], h, :]


def attention_forward(q, k, v, scale, causal=False, cu_seqlens=None, pairs=None):
    h_q, h_kv = q.shape[-2], k.shape[-2]
    assert h_q % h_kv == 0
    group = h_q // h_kv
    o = np.full(q.shape[:-1] + (v.shape[-1],), np.nan)
    if cu_seqlens is None:
        lse = np.full((q.shape[0], h_q, q.shape[1]), np.nan)
    else:
        lse = np.full((h_q, q.shape[0]), np.nan)
    want = None if pairs is None else set(map(tuple, pairs))
    for b, seg in _segments(q, cu_seqlens):
        for h in range(h_q):
            if want is not None and (b, h) not in want:
                continue
            oh, lh = head_forward(_head_views(q, b, seg, h), _head_views(k, b, seg, h // group),
                                  _head_views(v, b, seg, h // group), scale, causal)
            if seg is None:
                o[b, :, h, :] = oh
                lse[b, h, :] = lh
            else:
                o[seg[0]:seg[1], h, :] = oh
                lse[h, seg[0]:seg[1]] = lh
    return o, lse


def attention_backward(q, k, v, do, scale, causal=False, cu_seqlens=None, kv_pairs=None):
    """Returns dict(dq, dk, dv, o, lse). ``kv_pairs`` restricts the work to a
    list of (b, kv_head) groups; each is computed with all of its query heads so
    that dK and dV are complete. Other entries are NaN."""
    h_q, h_kv = q.shape[-2], k.shape[-2]
    assert h_q % h_kv == 0
    group = h_q // h_kv
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    o = np.full(q.shape[:-1] + (v.shape[-1],), np.nan)
    lse = np.full((q.shape[0], h_q, q.shape[1]) if cu_seqlens is None else (h_q, q.shape[0]), np.nan)
    want = None if kv_pairs is None else set(map(tuple, kv_pairs))
    for b, seg in _segments(q, cu_seqlens):
        for g in range(h_kv):
            if want is not None and (b, g) not in want:
                continue
            kh = _head_views(k, b, seg, g)
            vh = _head_views(v, b, seg, g)
            dk_sum = np.zeros(kh.shape)
            dv_sum = np.zeros(vh.shape)
            for h in range(g * group, (g + 1) * group):
                r = head_backward(_head_views(q, b, seg, h), kh, vh, _head_views(do, b, seg, h), scale, causal)
                dk_sum += r["dk"]
                dv_sum += r["dv"]
                if seg is None:
                    dq[b, :, h, :] = r["dq"]
                    o[b, :, h, :] = r["o"]
                    lse[b, h, :] = r["lse"]
                else:
                    dq[seg[0]:seg[1], h, :] = r["dq"]
                    o[seg[0]:seg[1], h, :] = r["o"]
                    lse[h, seg[0]:seg[1]] = r["lse"]
            if seg is None:
                dk[b, :, g, :] = dk_sum
                dv[b, :, g, :] = dv_sum
            else:
                dk[seg[0]:seg[1], g, :] = dk_sum
                dv[seg[0]:seg[1], g, :] = dv_sum
    return dict(dq=dq, dk=dk, dv=dv, o=o, lse=lse)
