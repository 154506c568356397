"""GPU parity: the CUDA forward and backward passes against the fp64 oracle on
the same seeded bf16 inputs, through the C ABI (ctypes binding).

Small cases are compared element by element in full; they span several tiles
and a ragged tail. The five named workloads run at full size on the GPU and are
compared on seeded (batch, head) samples (every row of a sampled head, or a
seeded subset of rows for the longest sequences).
"""

import math

import numpy as np
import pytest

import oracle
from exact_attention_15_gb300 import workloads as W
from gpu_common import (GRAD_TOL, LSE_TOL, O_TOL, as_f64, gpu_head, gpu_lse, head_slices,
                        rel_fro, run_backward, run_forward, to_host_f64)

pytestmark = pytest.mark.gpu


def _oracle_fwd_check(inp, o, lse, pairs, rows=None):
    worst_o = worst_l = 0.0
    for b, h in pairs:
        q, k, v, _ = head_slices(inp, b, h)
        if q.shape[0] == 0:
            continue
        r = None
        if rows is not None:
            r = np.unique(np.concatenate([rows[rows < q.shape[0]], [q.shape[0] - 1]]))
        o_ref, lse_ref = oracle.head_forward(q, k, v, inp.scale, inp.causal, rows=r)
        o_gpu = gpu_head(o, inp, b, h)
        l_gpu = gpu_lse(lse, inp, b, h)
        if r is not None:
            o_gpu, l_gpu = o_gpu[r], l_gpu[r]
        fin = np.isfinite(lse_ref)
        assert np.array_equal(fin, np.isfinite(l_gpu)), "masked-row pattern differs"
        worst_o = max(worst_o, float(np.max(np.abs(o_gpu - o_ref))) if o_ref.size else 0.0)
        if fin.any():
            worst_l = max(worst_l, float(np.max(np.abs(l_gpu[fin] - lse_ref[fin]))))
    assert worst_o <= O_TOL, f"O max-abs error {worst_o}"
    assert worst_l <= LSE_TOL, f"LSE abs error {worst_l}"
    return worst_o, worst_l


def _oracle_bwd_check(inp, dq, dk, dv, groups):
    g = inp.H_q // inp.H_kv
    worst = 0.0
    for b, hk in groups:
        dk_ref = dv_ref = None
        for h in range(hk * g, (hk + 1) * g):
            q, k, v, do = head_slices(inp, b, h)
            if q.shape[0] == 0:
                continue
            r = oracle.head_backward(q, k, v, do, inp.scale, inp.causal)
            e = rel_fro(gpu_head(dq, inp, b, h), r["dq"])
            assert e <= GRAD_TOL, f"dQ rel err {e} (b={b}, h={h})"
            worst = max(worst, e)
            dk_ref = r["dk"] if dk_ref is None else dk_ref + r["dk"]
            dv_ref = r["dv"] if dv_ref is None else dv_ref + r["dv"]
        if dk_ref is None:
            continue
        ek = rel_fro(gpu_head(dk, inp, b, hk), dk_ref)
        ev = rel_fro(gpu_head(dv, inp, b, hk), dv_ref)
        assert ek <= GRAD_TOL, f"dK rel err {ek} (b={b}, kv head={hk})"
        assert ev <= GRAD_TOL, f"dV rel err {ev} (b={b}, kv head={hk})"
        worst = max(worst, ek, ev)
    return worst


def _all_pairs(inp):
    return [(b, h) for b in range(inp.B) for h in range(inp.H_q)]


def _all_groups(inp):
    return [(b, g) for b in range(inp.B) for g in range(inp.H_kv)]


SMALL = {
    "tiny_cfg": dict(B=1, H_q=1, H_kv=1, N_q=128, N_k=128, d=64, scale=1 / math.sqrt(8), causal=False),
    "ragged_d64": dict(B=2, H_q=2, H_kv=2, N_q=300, N_k=300, d=64, causal=False),
    "ragged_d128_causal": dict(B=2, H_q=2, H_kv=2, N_q=300, N_k=300, d=128, causal=True),
    "gqa_causal": dict(B=1, H_q=4, H_kv=2, N_q=257, N_k=257, d=128, causal=True),
    "cross_lengths": dict(B=2, H_q=1, H_kv=1, N_q=200, N_k=333, d=64, causal=False),
    "one_query_row": dict(B=1, H_q=2, H_kv=1, N_q=1, N_k=700, d=128, causal=False),
    "varlen_causal": dict(B=0, H_q=4, H_kv=1, N_q=0, N_k=0, d=128, causal=True,
                          seqlens=[1, 127, 129, 300, 513, 64]),
    "varlen_d64": dict(B=0, H_q=2, H_kv=2, N_q=0, N_k=0, d=64, causal=False, seqlens=[5, 256, 255]),
    "boosted_keys": dict(B=1, H_q=2, H_kv=2, N_q=1000, N_k=1000, d=128, causal=True,
                         boost_frac=0.05, boost=3.0),
    "negative_scale": dict(B=1, H_q=1, H_kv=1, N_q=256, N_k=256, d=64, scale=-0.2, causal=False),
    "zero_scale": dict(B=1, H_q=1, H_kv=1, N_q=130, N_k=130, d=64, scale=0.0, causal=True),
    # packed lengths out of order, with empty sequences: the forward's work list
    # visits them longest first
    "varlen_unsorted_empty": dict(B=0, H_q=4, H_kv=2, N_q=0, N_k=0, d=64, causal=True,
                                  seqlens=[0, 700, 3, 0, 256, 1000, 0, 257]),
    # more work tiles (3 x 8 x 8 = 192) than SMs: each persistent CTA takes several
    "more_tiles_than_sms": dict(B=3, H_q=8, H_kv=4, N_q=2000, N_k=2000, d=64, causal=True),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_forward_backward(name):
    kw = dict(SMALL[name])
    inp = W.custom(seed=100 + len(name), **kw)
    o, lse, dev = run_forward(inp)
    _oracle_fwd_check(inp, o, lse, _all_pairs(inp))
    dq, dk, dv = run_backward(inp, o, lse, dev)
    _oracle_bwd_check(inp, dq, dk, dv, _all_groups(inp))


@pytest.mark.parametrize("d", [64, 128])
def test_worked_example_on_gpu(d):
    """One query, 256 keys in two key tiles; only key 0 (score 0) and key 128
    (score ln 3) matter, with values 2 and 10: O = 8 in every column. With scale
    20 the running max jumps by far more than 2^8 across the tiles, which forces
    the rescale branch."""
    import torch
    from exact_attention_15_gb300 import binding
    for scale, expected in ((math.log(3.0), 8.0), (20.0, None)):
        q = torch.zeros(1, 1, 1, d, dtype=torch.bfloat16, device="cuda")
        q[..., 0] = 1.0
        k = torch.zeros(1, 256, 1, d, dtype=torch.bfloat16, device="cuda")
        k[0, :, 0, 0] = -64.0
        k[0, 0, 0, 0] = 0.0
        k[0, 128, 0, 0] = 1.0
        v = torch.zeros(1, 256, 1, d, dtype=torch.bfloat16, device="cuda")
        v[0, 0] = 2.0
        v[0, 128] = 10.0
        o, lse = binding.forward(q, k, v, scale=scale)
        torch.cuda.synchronize()
        o = o.float().cpu().numpy()[0, 0, 0]
        if expected is None:
            # weights e^0 : e^20 -> essentially all on key 128
            w1 = 1.0 / (1.0 + math.exp(-20.0))
            expected = 2.0 * (1 - w1) + 10.0 * w1
        assert np.max(np.abs(o - expected)) < 3e-2, (scale, o[:4])
        ref_lse = math.log(1.0 + math.exp(scale))
        assert abs(float(lse.cpu()[0, 0, 0]) - ref_lse) < 2e-3


# d_qk = 192, d_v = 128. Eight or more key tiles put a V tile across the end of
# the forward's block ring (its column blocks in slots 7 and 0); the backward
# runs its two passes (query/key head columns 0-127 with dV, then 128-191).
ASYM = {
    "asym_ragged_causal": dict(B=2, H_q=2, H_kv=2, N_q=300, N_k=300, causal=True),
    "asym_gqa_ring_wrap": dict(B=1, H_q=4, H_kv=2, N_q=1000, N_k=1000, causal=False),
    "asym_gqa_ring_wrap_causal": dict(B=1, H_q=4, H_kv=2, N_q=1300, N_k=1300, causal=True),
    "asym_cross_lengths": dict(B=2, H_q=1, H_kv=1, N_q=200, N_k=1333, causal=False),
    "asym_varlen": dict(B=0, H_q=4, H_kv=1, N_q=0, N_k=0, causal=True,
                        seqlens=[1, 127, 0, 129, 1100, 300, 64]),
    "asym_no_keys_rows": dict(B=1, H_q=2, H_kv=1, N_q=5, N_k=700, causal=False),
}


@pytest.mark.parametrize("name", list(ASYM))
def test_asymmetric_head_dims_forward(name):
    inp = W.custom(seed=200 + len(name), d=192, d_v=128, parts=("q", "k", "v"), **ASYM[name])
    o, lse, _ = run_forward(inp)
    assert tuple(o.shape[-1:]) == (128,)
    _oracle_fwd_check(inp, o, lse, _all_pairs(inp))


@pytest.mark.parametrize("name", list(ASYM))
def test_asymmetric_head_dims_backward(name):
    inp = W.custom(seed=200 + len(name), d=192, d_v=128, **ASYM[name])
    o, lse, dev = run_forward(inp)
    dq, dk, dv = run_backward(inp, o, lse, dev)
    assert tuple(dq.shape[-1:]) == (192,) and tuple(dk.shape[-1:]) == (192,)
    assert tuple(dv.shape[-1:]) == (128,)
    _oracle_bwd_check(inp, dq, dk, dv, _all_groups(inp))


@pytest.mark.parametrize("B,H,N,d,H_kv", [(2, 16, 8192, 64, 16), (1, 16, 8192, 128, 16),
                                           (1, 16, 4096, 192, 16), (1, 16, 8192, 128, 4),
                                           (1, 12, 6000, 64, 2)])
def test_balanced_schedule_writes_every_tile(B, H, N, d, H_kv):
    """Causal shapes with long, unequal work tiles run on a persistent grid
    that takes its tiles from a host-built balanced list. Every output row must
    be written exactly as the per-tile computation gives it: the outputs start
    as NaN and must end finite everywhere, a second launch (schedule reused from
    its cache) must be bit-identical, and sampled heads and rows match the
    oracle. With an even GQA group a work tile holds the same rows of two query
    heads."""
    from exact_attention_15_gb300 import binding
    import torch
    d_v = 128 if d == 192 else d
    inp = W.custom(B, H, H_kv, N, N, d, causal=True, seed=4242 + d + H_kv, parts=("q", "k", "v"),
                   d_v=d_v)
    from gpu_common import device_inputs
    dev = device_inputs(inp)
    outs = []
    for _ in range(2):
        o = torch.full((B, N, H, d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
        binding.forward(dev["q"], dev["k"], dev["v"], scale=inp.scale, causal=True, out=o, lse=lse)
        torch.cuda.synchronize()
        assert binding.attn_check(None) == 0
        assert not torch.isnan(o).any().item(), "an output tile was not written"
        assert not torch.isnan(lse).any().item(), "an LSE tile was not written"
        outs.append((o, lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    rng = np.random.default_rng(11)
    pairs = _sample(rng, _all_pairs(inp), 2)
    # rows from the first, a middle and the last work tile of the sequence
    rows = np.array([0, 1, 255, 256, N // 2 - 1, N // 2, N - 257, N - 256, N - 2, N - 1])
    _oracle_fwd_check(inp, outs[0][0], outs[0][1], pairs, rows)


@pytest.mark.parametrize("d,causal,H_q,H_kv", [(128, True, 4, 1), (128, False, 2, 2), (64, True, 4, 2),
                                               (192, True, 2, 1)])
def test_claimed_schedule_packed(d, causal, H_q, H_kv):
    """Packed inputs with more work tiles than SMs run on a persistent grid whose
    CTAs claim tiles from a device counter (zeroed by the planning kernel at every
    call). Every row must be written (outputs start as NaN), repeated calls and a
    CUDA-graph replay must give the same bits, and every (sequence, head) matches
    the oracle. The lengths include empty and one-row sequences and several whole
    and ragged tiles."""
    import torch
    from exact_attention_15_gb300 import binding
    from gpu_common import device_inputs
    rng = np.random.default_rng(900 + d)
    lens = [int(x) for x in rng.integers(0, 700, size=56)] + [0, 1, 0, 128, 256, 1500, 2]
    d_v = 128 if d == 192 else d
    inp = W.custom(0, H_q, H_kv, 0, 0, d, causal=causal, seed=901 + d, seqlens=lens,
                   parts=("q", "k", "v"), d_v=d_v)
    T = inp.N_q
    plan = binding.attn_debug_fwd_plan(len(lens), H_q, H_kv, T, T, d, d_v, causal, True, 152)
    assert plan["mode"] == binding.FWD_CLAIMED and plan["tiles"] > 152
    dev = device_inputs(inp)

    def fwd(o, lse):
        binding.forward(dev["q"], dev["k"], dev["v"], scale=inp.scale, causal=causal,
                        cu_seqlens=dev["cu"], out=o, lse=lse)

    outs = []
    for _ in range(3):
        o = torch.full((T, H_q, d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((H_q, T), float("nan"), dtype=torch.float32, device="cuda")
        fwd(o, lse)
        torch.cuda.synchronize()
        assert binding.attn_check(None) == 0
        assert not torch.isnan(o).any().item(), "an output row was not written"
        assert not torch.isnan(lse).any().item(), "an LSE row was not written"
        outs.append((o, lse))
    for o, lse in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(lse, outs[0][1])
    go = torch.full((T, H_q, d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    gl = torch.full((H_q, T), float("nan"), dtype=torch.float32, device="cuda")
    # the first packed call on a stream (which sets up its planning buffer) is
    # made outside capture, as the C ABI asks
    cap = torch.cuda.Stream()
    with torch.cuda.stream(cap):
        fwd(go, gl)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        fwd(go, gl)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert binding.attn_check(None) == 0
        assert torch.equal(go.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(gl, outs[0][1])
    _oracle_fwd_check(inp, outs[0][0], outs[0][1], _all_pairs(inp))


def test_forward_on_concurrent_streams():
    """Forward passes issued on two streams at once give the same bits as the
    same passes run one after the other, launch after launch."""
    import torch
    from exact_attention_15_gb300 import binding
    probs = [W.custom(seed=s, B=2, H_q=8, H_kv=8, N_q=1500, N_k=1500, d=64, causal=c,
                      parts=("q", "k", "v"))
             for s, c in ((11, True), (12, False))]
    devs = [device_inputs_fwd(x) for x in probs]
    ref = []
    for x, dv in zip(probs, devs):
        o, lse = binding.forward(dv["q"], dv["k"], dv["v"], scale=x.scale, causal=x.causal)
        torch.cuda.synchronize()
        ref.append((o.clone(), lse.clone()))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[], []]
    torch.cuda.synchronize()
    for rep in range(4):
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                x, dv = probs[i], devs[i]
                outs[i].append(binding.forward(dv["q"], dv["k"], dv["v"], scale=x.scale,
                                               causal=x.causal))
    torch.cuda.synchronize()
    assert binding.attn_check(None) == 0
    for i in range(2):
        for o, lse in outs[i]:
            assert torch.equal(o.view(torch.int16), ref[i][0].view(torch.int16))
            assert torch.equal(lse, ref[i][1])
    _oracle_fwd_check(probs[0], ref[0][0], ref[0][1], [(0, 0), (1, 7)])


def test_cuda_graph_capture_and_replay():
    """Forward and deterministic backward captured in a CUDA graph and replayed on
    new inputs give the same bits as eager calls. The causal shape is new when the
    first graph is captured, so its balanced forward schedule is not built during
    capture and that graph runs one CTA per work tile; the second graph is captured
    after an eager call built the schedule and uses it. Per-tile results do not
    depend on the schedule, so all three agree bit for bit."""
    import torch
    from exact_attention_15_gb300 import binding
    from gpu_common import device_inputs
    B, H, N, d = 1, 16, 6144, 128
    a = W.custom(B, H, H, N, N, d, causal=True, seed=777)
    b = W.custom(B, H, H, N, N, d, causal=True, seed=778)
    dev_a, dev_b = device_inputs(a), device_inputs(b)
    names = ("q", "k", "v", "do")
    static = {n: dev_a[n].clone() for n in names}

    def step(t):
        o, lse = binding.forward(t["q"], t["k"], t["v"], scale=a.scale, causal=True)
        dq, dk, dv = binding.backward(t["q"], t["k"], t["v"], o, lse, t["do"], scale=a.scale,
                                      causal=True, deterministic=True)
        return o, lse, dq, dk, dv

    def capture():
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            outs = step(static)
        return g, outs

    g1, outs1 = capture()                # shape first seen here: no schedule built
    eager = [step(dev_a), step(dev_b)]   # builds and uses the schedule
    torch.cuda.synchronize()
    g2, outs2 = capture()                # uses the cached schedule
    for src, ref in ((dev_b, eager[1]), (dev_a, eager[0])):
        for n in names:
            static[n].copy_(src[n])
        for g, outs in ((g1, outs1), (g2, outs2)):
            g.replay()
            torch.cuda.synchronize()
            assert binding.attn_check(None) == 0
            for x, y in zip(outs, ref):
                assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                                   y.view(torch.int16) if y.dtype == torch.bfloat16 else y)
    _oracle_fwd_check(a, eager[0][0], eager[0][1], [(0, 3)], np.array([0, 127, 128, 3000, N - 1]))


def device_inputs_fwd(inp):
    from gpu_common import to_dev
    return dict(q=to_dev(inp.q), k=to_dev(inp.k), v=to_dev(inp.v))


def test_no_keys_and_empty_batch():
    import torch
    from exact_attention_15_gb300 import binding
    q = torch.randn(1, 5, 2, 64, device="cuda").bfloat16()
    k = torch.empty(1, 0, 2, 64, device="cuda", dtype=torch.bfloat16)
    o, lse = binding.forward(q, k, k)
    torch.cuda.synchronize()
    assert binding.attn_check(None) == 0
    assert torch.all(o == 0)
    assert torch.all(torch.isinf(lse)) and torch.all(lse < 0)
    q0 = torch.empty(0, 5, 2, 64, device="cuda", dtype=torch.bfloat16)
    binding.forward(q0, q0, q0)
    torch.cuda.synchronize()
    assert binding.attn_check(None) == 0


# ------------------------------------------------------------------ full-size workloads

def _sample(rng, items, n):
    idx = rng.choice(len(items), size=min(n, len(items)), replace=False)
    return [items[i] for i in sorted(idx)]


FULL = [
    ("tiny", None, None),
    ("short", 8, None),
    ("short_causal", 8, None),
    ("mid", 3, 512),
    ("mid_causal", 3, 512),
    ("long", 2, 384),
    ("varlen_gqa", 2, None),
    ("mla", 3, 512),
    ("mla_causal", 3, 512),
]


@pytest.mark.parametrize("name,n_pairs,n_rows", FULL, ids=[f[0] for f in FULL])
def test_workload_forward(name, n_pairs, n_rows):
    inp = W.generate(name, parts=("q", "k", "v"))
    o, lse, _ = run_forward(inp)
    rng = np.random.default_rng(7)
    pairs = _all_pairs(inp) if n_pairs is None else _sample(rng, _all_pairs(inp), n_pairs)
    rows = None if n_rows is None else np.sort(rng.choice(inp.N_q if inp.cu_seqlens is None else 512,
                                                             size=n_rows, replace=False))
    _oracle_fwd_check(inp, o, lse, pairs, rows)


BWD_FULL = [("tiny", None), ("short", 3), ("short_causal", 3), ("mid", 1), ("mid_causal", 1),
            ("long", 1), ("varlen_gqa", 1), ("mla", 1), ("mla_causal", 1)]


@pytest.mark.parametrize("name,n_groups", BWD_FULL, ids=[f[0] for f in BWD_FULL])
def test_workload_backward(name, n_groups):
    inp = W.generate(name)
    o, lse, dev = run_forward(inp)
    dq, dk, dv = run_backward(inp, o, lse, dev)
    rng = np.random.default_rng(11)
    groups = _all_groups(inp) if n_groups is None else _sample(rng, _all_groups(inp), n_groups)
    _oracle_bwd_check(inp, dq, dk, dv, groups)


DET_CUSTOM = {
    # non-causal, equal lengths: key tiles walk their query tiles from their own
    "rotated_gqa": dict(B=2, H_q=4, H_kv=2, N_q=1000, N_k=1000, d=128, causal=False),
    "rotated_packed": dict(B=0, H_q=2, H_kv=1, N_q=0, N_k=0, d=64, causal=False,
                           seqlens=[300, 0, 129, 700, 1]),
    # causal, ragged: shortest-processing-time order from the diagonal
    "spt_ragged": dict(B=1, H_q=4, H_kv=1, N_q=1100, N_k=1100, d=128, causal=True),
    # different query and key lengths: ascending key-tile order
    "ascending_cross": dict(B=2, H_q=2, H_kv=2, N_q=300, N_k=700, d=64, causal=False),
    # separate head dimensions: each of the two passes has its own ordering
    "asym_spt": dict(B=1, H_q=4, H_kv=2, N_q=1100, N_k=1100, d=192, d_v=128, causal=True),
    "asym_rotated_packed": dict(B=0, H_q=2, H_kv=1, N_q=0, N_k=0, d=192, d_v=128, causal=False,
                                seqlens=[300, 700, 129]),
}


@pytest.mark.parametrize("name", ["varlen_gqa", "short_causal", "short"] + list(DET_CUSTOM))
def test_deterministic_backward(name):
    """Deterministic mode: three runs bit-identical, and within tolerance, in each
    order the library picks for the dQ additions."""
    import torch
    if name in DET_CUSTOM:
        inp = W.custom(seed=300 + len(name), **DET_CUSTOM[name])
    else:
        inp = W.generate(name)
    o, lse, dev = run_forward(inp)
    runs = [run_backward(inp, o, lse, dev, deterministic=True) for _ in range(3)]
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), "not bit-identical"
    rng = np.random.default_rng(13)
    groups = _all_groups(inp) if name in DET_CUSTOM else _sample(rng, _all_groups(inp), 1)
    _oracle_bwd_check(inp, *runs[0], groups)
