"""Pins of the CPU oracle against facts the pages and the mathematics fix.

Each check is a function of the oracle module under test, so that the same check
can be run against a deliberately broken copy (see test_oracle_mutants.py) to
show that it catches the mistake.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import attention as A
from oracle import online as OL
from oracle import scalar as SC

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _num(x):
    return math.log(3.0) if x == "ln3" else float(x)


# ------------------------------------------------------------------ worked example

def check_worked_example_forward(att):
    g = _golden("worked_example.json")
    s = [_num(x) for x in g["scores"]]
    # one query q = [1], keys k_j = [s_j], scale 1: the scores are exactly s
    q = np.array([[1.0]])
    k = np.array([[s[0]], [s[1]]])
    v = np.array([[g["values"][0]], [g["values"][1]]])
    o, lse = att.head_forward(q, k, v, 1.0)
    assert abs(o[0, 0] - g["output"]) < 1e-14
    assert abs(lse[0] - math.log(4.0)) < 1e-14
    r = att.head_backward(q, k, v, np.array([[g["upstream_gradient"]]]), 1.0, return_ds=True)
    np.testing.assert_allclose(r["p"][0], g["weights"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(r["ds"][0], g["score_gradients"], rtol=0, atol=1e-14)
    assert abs(np.sum(r["ds"][0])) < 1e-14
    # the chain rule through s_j = q . k_j with q = 1: dk_j = ds_j, dv_j = p_j, dq = sum ds_j k_j
    np.testing.assert_allclose(r["dk"][:, 0], g["score_gradients"], atol=1e-14)
    np.testing.assert_allclose(r["dv"][:, 0], g["weights"], atol=1e-15)
    assert abs(r["dq"][0, 0] - 1.5 * math.log(3.0)) < 1e-14


def test_worked_example_forward_backward():
    check_worked_example_forward(A)


def test_worked_example_scalar():
    g = _golden("worked_example.json")
    s = [_num(x) for x in g["scores"]]
    o, lse = SC.forward([[1.0]], [[s[0]], [s[1]]], [[2.0], [10.0]], 1.0)
    assert abs(o[0][0] - 8.0) < 1e-14
    dq, dk, dv = SC.backward([[1.0]], [[s[0]], [s[1]]], [[2.0], [10.0]], [[1.0]], 1.0)
    assert abs(dk[0][0] + 1.5) < 1e-14 and abs(dk[1][0] - 1.5) < 1e-14


def check_online_merge(ol):
    g = _golden("worked_example.json")
    s = [_num(x) for x in g["scores"]]
    sb = [np.array([s[0]]), np.array([s[1]])]
    vb = [np.array([[2.0]]), np.array([[10.0]])]
    o, m, l = ol.online_merge(sb, vb)
    assert abs(o[0] - g["output"]) < 1e-14
    # after the max moves 0 -> ln 3, the old sum 1 becomes 1/3, plus the new e^0 = 1
    assert abs(m - math.log(3.0)) < 1e-15
    assert abs(l - (g["rescale_factor_on_max_move"] + 1.0)) < 1e-14
    # both the lazy variant that keeps the stale max and the one that always rescales
    for tau, n_expected in ((8.0, 1), (0.0, 2)):
        o2, m_used, l2, n = ol.online_merge_lazy(sb, vb, tau=tau)
        assert abs(o2[0] - g["output"]) < 1e-14
        assert n == n_expected
    # stale max kept: e^(0-0) + e^(ln3 - 0) = 4 relative to m_used = 0
    o2, m_used, l2, _ = ol.online_merge_lazy(sb, vb, tau=8.0)
    assert m_used == 0.0 and abs(l2 - 4.0) < 1e-14


def test_online_merge_worked_example():
    check_online_merge(OL)


def test_blockwise_average_is_wrong():
    g = _golden("worked_example.json")
    s = [_num(x) for x in g["scores"]]
    wrong = OL.blockwise_average_merge([np.array([s[0]]), np.array([s[1]])],
                                       [np.array([[2.0]]), np.array([[10.0]])])
    assert abs(wrong[0] - g["wrong_blockwise_average"]) < 1e-14
    assert abs(wrong[0] - g["output"]) > 1.0


# ------------------------------------------------------------------ merges vs definition

def check_merges_match_definition(att, ol, seed=3):
    rng = np.random.default_rng(seed)
    for trial in range(20):
        n_k = int(rng.integers(1, 40))
        d = 4
        q = rng.standard_normal((1, d))
        k = rng.standard_normal((n_k, d)) * rng.choice([0.5, 3.0, 12.0])
        v = rng.standard_normal((n_k, 3))
        o, lse = att.head_forward(q, k, v, 0.7)
        s = 0.7 * (k @ q[0])
        cuts = np.sort(rng.choice(np.arange(1, n_k + 1), size=min(n_k, 4), replace=False))
        edges = [0] + [c for c in cuts if c < n_k] + [n_k]
        sb = [s[a:b] for a, b in zip(edges[:-1], edges[1:])]
        vb = [v[a:b] for a, b in zip(edges[:-1], edges[1:])]
        o1, m1, l1 = ol.online_merge(sb, vb)
        np.testing.assert_allclose(o1, o[0], rtol=1e-12, atol=1e-12)
        assert abs(m1 + math.log(l1) - lse[0]) < 1e-11
        for tau in (0.0, 1.0, 8.0):
            o2, mu, l2, _ = ol.online_merge_lazy(sb, vb, tau=tau)
            np.testing.assert_allclose(o2, o[0], rtol=1e-12, atol=1e-12)
            assert abs(mu + math.log(l2) - lse[0]) < 1e-11


def test_merges_match_definition():
    check_merges_match_definition(A, OL)


def test_lazy_rescale_counts_fewer():
    # scores drifting upward slowly: an always-rescale merge rescales every block,
    # tau = 8 only when the max has climbed by more than 2^8
    rng = np.random.default_rng(5)
    s = np.linspace(0.0, 20.0, 64 * 32) + 0.1 * rng.standard_normal(64 * 32)
    v = rng.standard_normal((64 * 32, 2))
    sb = [s[i:i + 64] for i in range(0, len(s), 64)]
    vb = [v[i:i + 64] for i in range(0, len(s), 64)]
    _, _, _, n_always = OL.online_merge_lazy(sb, vb, tau=0.0)
    _, _, _, n_lazy = OL.online_merge_lazy(sb, vb, tau=8.0)
    assert n_always == 32 and n_lazy <= 4


# ------------------------------------------------------------------ brute force

def _rand_head(rng, n_q, n_k, d, dv=None):
    dv = dv or d
    return (rng.standard_normal((n_q, d)), rng.standard_normal((n_k, d)),
            rng.standard_normal((n_k, dv)), rng.standard_normal((n_q, dv)))


def check_brute_force_scalar(att, seed=11):
    rng = np.random.default_rng(seed)
    for causal in (False, True):
        for n in (1, 2, 5, 8):
            q, k, v, do = _rand_head(rng, n, n, 3)
            o, lse = att.head_forward(q, k, v, 0.9, causal)
            o2, lse2 = SC.forward(q.tolist(), k.tolist(), v.tolist(), 0.9, causal)
            np.testing.assert_allclose(o, o2, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(lse, lse2, rtol=1e-13, atol=1e-13)
            r = att.head_backward(q, k, v, do, 0.9, causal)
            dq, dk, dv = SC.backward(q.tolist(), k.tolist(), v.tolist(), do.tolist(), 0.9, causal)
            np.testing.assert_allclose(r["dq"], dq, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(r["dk"], dk, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(r["dv"], dv, rtol=1e-12, atol=1e-12)


def test_brute_force_scalar():
    check_brute_force_scalar(A)


def check_finite_differences(att, seed=13, d_qk=4, d_v=None):
    """Central differences of L = sum(O o dO) in float64, h = 1e-6. With d_v the
    values (and O, dO) have their own width, as in the (192, 128) head
    dimensions of the FlashAttention-4 benchmark."""
    rng = np.random.default_rng(seed)
    h = 1e-6
    for causal in (False, True):
        n = 6
        q, k, v, do = _rand_head(rng, n, n, d_qk, d_v)
        scale = 0.8
        r = att.head_backward(q, k, v, do, scale, causal)

        def loss(qq, kk, vv):
            o, _ = att.head_forward(qq, kk, vv, scale, causal)
            return float(np.sum(o * do))

        for name, x, g in (("q", q, r["dq"]), ("k", k, r["dk"]), ("v", v, r["dv"])):
            num = np.zeros_like(x)
            for idx in np.ndindex(*x.shape):
                xp = x.copy(); xp[idx] += h
                xm = x.copy(); xm[idx] -= h
                args_p = {"q": q, "k": k, "v": v}; args_p[name] = xp
                args_m = {"q": q, "k": k, "v": v}; args_m[name] = xm
                num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"]) -
                            loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
            err = np.linalg.norm(num - g) / max(np.linalg.norm(g), 1e-30)
            assert err < 1e-6, (name, causal, err)


def test_finite_differences():
    check_finite_differences(A)


def test_finite_differences_separate_head_dims():
    """The backward with query/key width 5 and value width 3: dQ, dK have 5
    columns, dV 3, all matching central differences."""
    check_finite_differences(A, seed=31, d_qk=5, d_v=3)


# ------------------------------------------------------------------ invariants and closed forms

def check_invariants(att, seed=17):
    rng = np.random.default_rng(seed)
    for causal in (False, True):
        q, k, v, do = _rand_head(rng, 24, 24, 8)
        scale = 0.5
        r = att.head_backward(q, k, v, do, scale, causal, return_ds=True)
        np.testing.assert_allclose(r["p"].sum(axis=1), 1.0, atol=1e-14)       # rows of P sum to 1
        np.testing.assert_allclose(r["ds"].sum(axis=1), 0.0, atol=1e-12)      # rows of dS sum to 0
        np.testing.assert_allclose(r["dv"].sum(axis=0), do.sum(axis=0), atol=1e-12)  # sum_keys dV = sum_queries dO
        s = scale * q @ k.T
        if causal:
            s = np.where(np.tril(np.ones_like(s, dtype=bool)), s, -np.inf)
        assert np.all(r["lse"] >= s.max(axis=1) - 1e-12)                      # LSE >= max S
        assert np.all(r["lse"] <= s.max(axis=1) + math.log(24) + 1e-12)
        vmin, vmax = v.min(axis=0), v.max(axis=0)                               # O in the hull of V
        assert np.all(r["o"] >= vmin - 1e-12) and np.all(r["o"] <= vmax + 1e-12)
        if causal:
            # row 0 sees key 0 only
            np.testing.assert_allclose(r["o"][0], v[0], atol=1e-14)


def test_invariants():
    check_invariants(A)


def check_closed_forms(att, seed=19):
    rng = np.random.default_rng(seed)
    q, k, v, do = _rand_head(rng, 10, 10, 4)
    # scale 0: uniform attention -> mean of V; causal -> prefix means; LSE = ln(#keys)
    o, lse = att.head_forward(q, k, v, 0.0, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=0), o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, math.log(10), atol=1e-14)
    o, lse = att.head_forward(q, k, v, 0.0, True)
    prefix = np.cumsum(v, axis=0) / np.arange(1, 11)[:, None]
    np.testing.assert_allclose(o, prefix, atol=1e-14)
    np.testing.assert_allclose(lse, np.log(np.arange(1, 11)), atol=1e-14)
    # one key: O = V_0, dQ = dK = 0, dV = sum dO
    r = att.head_backward(q, k[:1], v[:1], do, 0.7, False)
    np.testing.assert_allclose(r["o"], np.broadcast_to(v[0], r["o"].shape), atol=1e-14)
    np.testing.assert_allclose(r["dq"], 0.0, atol=1e-14)
    np.testing.assert_allclose(r["dk"], 0.0, atol=1e-13)
    np.testing.assert_allclose(r["dv"][0], do.sum(axis=0), atol=1e-13)


def test_closed_forms():
    check_closed_forms(A)


def check_asymmetric_head_dims(att, seed=29):
    """Queries/keys and values of different widths (the FlashAttention-4 benchmark
    also runs d_qk = 192, d_v = 128; here 5 and 3): O has d_v columns and equals
    the scalar textbook loop; scale 0 gives the mean of the V rows."""
    rng = np.random.default_rng(seed)
    for causal in (False, True):
        n = 7
        q = rng.standard_normal((n, 5))
        k = rng.standard_normal((n, 5))
        v = rng.standard_normal((n, 3))
        o, lse = att.head_forward(q, k, v, 0.6, causal)
        assert o.shape == (n, 3)
        o2, lse2 = SC.forward(q.tolist(), k.tolist(), v.tolist(), 0.6, causal)
        np.testing.assert_allclose(o, o2, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(lse, lse2, rtol=1e-13, atol=1e-13)
    o, _ = att.head_forward(q, k, v, 0.0, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=0), o.shape), atol=1e-14)


def test_asymmetric_head_dims():
    check_asymmetric_head_dims(A)


def test_fully_masked_row():
    # a query that sees no key: O = 0, LSE = -inf, no gradient
    q = np.ones((1, 2)); k = np.ones((3, 2)); v = np.ones((3, 2))
    s = A._softmax_rows(np.full((1, 3), -np.inf))
    assert np.all(s[0] == 0.0) and s[1][0] == -np.inf


# ------------------------------------------------------------------ GQA and packed layout

def check_gqa_is_repeated_heads(att_mod, seed=23):
    rng = np.random.default_rng(seed)
    B, N, H_q, H_kv, d = 2, 12, 4, 2, 4
    q = rng.standard_normal((B, N, H_q, d))
    k = rng.standard_normal((B, N, H_kv, d))
    v = rng.standard_normal((B, N, H_kv, d))
    do = rng.standard_normal((B, N, H_q, d))
    g = att_mod.attention_backward(q, k, v, do, 0.6, causal=True)
    # the same problem with K/V heads repeated explicitly: query head h reads KV head h // 2
    kr = np.repeat(k, 2, axis=2)
    vr = np.repeat(v, 2, axis=2)
    m = att_mod.attention_backward(q, kr, vr, do, 0.6, causal=True)
    np.testing.assert_allclose(g["o"], m["o"], atol=1e-13)
    np.testing.assert_allclose(g["dq"], m["dq"], atol=1e-12)
    np.testing.assert_allclose(g["dk"], m["dk"][:, :, 0::2] + m["dk"][:, :, 1::2], atol=1e-12)
    np.testing.assert_allclose(g["dv"], m["dv"][:, :, 0::2] + m["dv"][:, :, 1::2], atol=1e-12)
    o_f, lse_f = att_mod.attention_forward(q, k, v, 0.6, causal=True)
    np.testing.assert_allclose(o_f, g["o"], atol=1e-13)
    np.testing.assert_allclose(lse_f, g["lse"], atol=1e-13)
    # head 1 of the repeated problem uses KV head 0 (not 1): check one head by hand
    oh, _ = att_mod.head_forward(q[0, :, 1], k[0, :, 0], v[0, :, 0], 0.6, True)
    np.testing.assert_allclose(g["o"][0, :, 1], oh, atol=1e-14)


def test_gqa_is_repeated_heads():
    check_gqa_is_repeated_heads(A)


def check_packed_is_per_sequence(att_mod, seed=29):
    rng = np.random.default_rng(seed)
    lens = [3, 1, 7, 5]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, H_q, H_kv, d = int(cu[-1]), 2, 1, 4
    q = rng.standard_normal((T, H_q, d)); do = rng.standard_normal((T, H_q, d))
    k = rng.standard_normal((T, H_kv, d)); v = rng.standard_normal((T, H_kv, d))
    r = att_mod.attention_backward(q, k, v, do, 0.5, causal=True, cu_seqlens=cu)
    for s, L in enumerate(lens):
        a, b = cu[s], cu[s + 1]
        one = att_mod.attention_backward(q[None, a:b], k[None, a:b], v[None, a:b], do[None, a:b], 0.5, causal=True)
        np.testing.assert_allclose(r["o"][a:b], one["o"][0], atol=1e-13)
        np.testing.assert_allclose(r["lse"][:, a:b], one["lse"][0], atol=1e-13)
        np.testing.assert_allclose(r["dq"][a:b], one["dq"][0], atol=1e-12)
        np.testing.assert_allclose(r["dk"][a:b], one["dk"][0], atol=1e-12)
        np.testing.assert_allclose(r["dv"][a:b], one["dv"][0], atol=1e-12)
    o, lse = att_mod.attention_forward(q, k, v, 0.5, causal=True, cu_seqlens=cu)
    np.testing.assert_allclose(o, r["o"], atol=1e-13)
    np.testing.assert_allclose(lse, r["lse"], atol=1e-13)


def test_packed_is_per_sequence():
    check_packed_is_per_sequence(A)


def test_row_blocking_does_not_change_results():
    rng = np.random.default_rng(31)
    q, k, v, do = _rand_head(rng, 50, 50, 4)
    a = A.head_backward(q, k, v, do, 0.4, True, row_block=7)
    b = A.head_backward(q, k, v, do, 0.4, True, row_block=4096)
    for key in ("dq", "dk", "dv", "o", "lse"):
        np.testing.assert_allclose(a[key], b[key], atol=1e-13)
    o, _ = A.head_forward(q, k, v, 0.4, True, rows=np.array([3, 17, 49]))
    np.testing.assert_allclose(o, b["o"][[3, 17, 49]], atol=1e-14)
