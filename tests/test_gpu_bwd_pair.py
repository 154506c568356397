"""The CTA-pair backward (the 2-CTA backward of the FlashAttention-4 summary,
section 3.2.3), selected with attn_set_bwd_variant, against the fp64 oracle on
the same cases as the default backward: ragged and packed lengths, GQA, causal
masks, deterministic mode, and a full-size workload sample."""

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
    old = binding.attn_set_bwd_variant(binding.BWD_CTA_PAIR)
    yield
    binding.attn_set_bwd_variant(old)


def test_variant_hook_rejects_unknown():
    from exact_attention_15_gb300 import binding
    old = binding.attn_set_bwd_variant(binding.BWD_ONE_CTA)
    assert binding.attn_set_bwd_variant(7) == -1
    assert binding.attn_set_bwd_variant(old) == binding.BWD_ONE_CTA


@pytest.mark.parametrize("name", D128)
def test_pair_small(name, pair_variant):
    inp = W.custom(seed=300 + len(name), **SMALL[name])
    o, lse, dev = run_forward(inp)
    dq, dk, dv = run_backward(inp, o, lse, dev)
    _oracle_bwd_check(inp, dq, dk, dv, _all_groups(inp))


@pytest.mark.parametrize("kw", [
    dict(B=1, H_q=2, H_kv=1, N_q=700, N_k=700, d=128, causal=True),
    dict(B=2, H_q=2, H_kv=2, N_q=600, N_k=600, d=128, causal=False),
    dict(B=0, H_q=4, H_kv=2, N_q=0, N_k=0, d=128, causal=True, seqlens=[300, 0, 129, 520, 64]),
], ids=["causal_odd_pairs", "noncausal", "varlen"])
def test_pair_multi_pair(kw, pair_variant):
    inp = W.custom(seed=41, **kw)
    o, lse, dev = run_forward(inp)
    dq, dk, dv = run_backward(inp, o, lse, dev)
    _oracle_bwd_check(inp, dq, dk, dv, _all_groups(inp))


def test_pair_deterministic(pair_variant):
    import torch
    inp = W.custom(seed=43, B=0, H_q=4, H_kv=2, N_q=0, N_k=0, d=128, causal=True,
                   seqlens=[900, 257, 640])
    o, lse, dev = run_forward(inp)
    runs = [run_backward(inp, o, lse, dev, deterministic=True) for _ in range(3)]
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), "not bit-identical"
    _oracle_bwd_check(inp, *runs[0], _all_groups(inp))


def test_pair_full_workload_sample(pair_variant):
    inp = W.generate("mid_causal")
    o, lse, dev = run_forward(inp)
    dq, dk, dv = run_backward(inp, o, lse, dev)
    rng = np.random.default_rng(17)
    _oracle_bwd_check(inp, dq, dk, dv, _sample(rng, _all_groups(inp), 1))
