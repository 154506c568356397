"""The CTA-pair forward (M = 256 tiles over a cluster of two CTAs: the 2-CTA
tensor-core mode of the FlashAttention-4 summary, section 2.2), selected with
attn_set_fwd_variant, against the fp64 oracle: every d = 128 small case, blocks
that end inside either CTA's half, packed sequences, GQA, causal masks, no keys,
and a full-size workload sample."""

import numpy as np
import pytest

from exact_attention_15_gb300 import workloads as W
from gpu_common import run_backward, run_forward
from test_gpu_parity import SMALL, _all_groups, _all_pairs, _oracle_bwd_check, _oracle_fwd_check, _sample

pytestmark = pytest.mark.gpu

D128 = [n for n, kw in SMALL.items() if kw["d"] == 128]


@pytest.fixture()
def pair_variant():
    from exact_attention_15_gb300 import binding
    old = binding.attn_set_fwd_variant(binding.FWD_CTA_PAIR)
    yield
    binding.attn_set_fwd_variant(old)


def test_fwd_variant_hook_rejects_unknown():
    from exact_attention_15_gb300 import binding
    old = binding.attn_set_fwd_variant(binding.FWD_ONE_CTA)
    assert binding.attn_set_fwd_variant(5) == -1
    assert binding.attn_set_fwd_variant(old) == binding.FWD_ONE_CTA


@pytest.mark.parametrize("name", D128)
def test_fwd_pair_small(name, pair_variant):
    inp = W.custom(seed=500 + len(name), **SMALL[name])
    o, lse, _ = run_forward(inp)
    _oracle_fwd_check(inp, o, lse, _all_pairs(inp))


@pytest.mark.parametrize("kw", [
    # 512-row blocks ending in the even CTA's first tile, the odd CTA's second
    # tile, and exactly on a block edge
    dict(B=2, H_q=2, H_kv=1, N_q=1100, N_k=1100, d=128, causal=True),
    dict(B=1, H_q=2, H_kv=2, N_q=1400, N_k=1400, d=128, causal=False),
    dict(B=1, H_q=3, H_kv=1, N_q=1024, N_k=1024, d=128, causal=True),
    dict(B=2, H_q=1, H_kv=1, N_q=333, N_k=900, d=128, causal=False),
    dict(B=0, H_q=4, H_kv=2, N_q=0, N_k=0, d=128, causal=True, seqlens=[300, 0, 129, 1030, 64, 512]),
], ids=["causal_tail_in_even", "noncausal_tail_in_odd", "block_edge_gqa3", "cross_lengths", "varlen"])
def test_fwd_pair_blocks(kw, pair_variant):
    inp = W.custom(seed=47, **kw)
    o, lse, _ = run_forward(inp)
    _oracle_fwd_check(inp, o, lse, _all_pairs(inp))


def test_fwd_pair_no_keys(pair_variant):
    """N_k = 0: every row sees no key, O = 0 and LSE = -inf."""
    import torch
    from exact_attention_15_gb300 import binding
    q = torch.randn(1, 300, 2, 128, device="cuda").to(torch.bfloat16)
    k = torch.empty(1, 0, 2, 128, device="cuda", dtype=torch.bfloat16)
    o, lse = binding.forward(q, k, k)
    torch.cuda.synchronize()
    assert binding.attn_check(None) == 0
    assert torch.count_nonzero(o).item() == 0
    assert bool(torch.isneginf(lse).all())


def test_fwd_pair_then_backward(pair_variant):
    """The backward runs on the pair forward's O and LSE."""
    inp = W.custom(seed=49, B=1, H_q=4, H_kv=2, N_q=700, N_k=700, d=128, causal=True)
    o, lse, dev = run_forward(inp)
    _oracle_fwd_check(inp, o, lse, _all_pairs(inp))
    dq, dk, dv = run_backward(inp, o, lse, dev)
    _oracle_bwd_check(inp, dq, dk, dv, _all_groups(inp))


@pytest.mark.parametrize("name,n_rows", [("mid", 512), ("mid_causal", 512), ("varlen_gqa", None)])
def test_fwd_pair_full_workload_sample(name, n_rows, pair_variant):
    inp = W.generate(name, parts=("q", "k", "v"))
    o, lse, _ = run_forward(inp)
    rng = np.random.default_rng(19)
    rows = None if n_rows is None else np.sort(rng.choice(inp.N_q, size=n_rows, replace=False))
    _oracle_fwd_check(inp, o, lse, _sample(rng, _all_pairs(inp), 2), rows)
