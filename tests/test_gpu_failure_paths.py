"""Failure paths, tested without faulting, trapping or hanging the GPU: bounded
device-side waits give up, record ATTN_ERR_TIMEOUT for attn_check(), and the
context stays usable."""

import numpy as np
import pytest

from exact_attention_15_gb300 import workloads as W
from gpu_common import GRAD_TOL, rel_fro, run_backward, run_forward, to_host_f64

pytestmark = pytest.mark.gpu

SHORT_LIMIT = 2_000_000  # cycles, about a millisecond


def test_stalled_wait_reports_timeout():
    import torch
    from exact_attention_15_gb300 import binding
    old = binding.attn_set_wait_limit(SHORT_LIMIT)
    try:
        assert binding.attn_check(None) == 0
        assert binding.attn_debug_stall(None) == 0
        assert binding.attn_check(None) == 9  # ATTN_ERR_TIMEOUT, and the record is cleared
        assert binding.attn_check(None) == 0
    finally:
        binding.attn_set_wait_limit(old)
    # the context is still usable
    inp = W.custom(1, 2, 2, 200, 200, 64, seed=5)
    o, lse, dev = run_forward(inp)
    assert torch.isfinite(o.float()).all()


def test_skipped_semaphore_release_times_out_then_recovers():
    import torch
    from exact_attention_15_gb300 import binding
    inp = W.custom(1, 2, 1, 384, 384, 128, causal=False, seed=6)
    o, lse, dev = run_forward(inp)
    ref = run_backward(inp, o, lse, dev, deterministic=True)
    old = binding.attn_set_wait_limit(SHORT_LIMIT)
    try:
        assert binding.attn_debug_inject(binding.FAULT_SKIP_DQ_RELEASE) == 0
        binding.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], scale=inp.scale,
                         deterministic=True)
        torch.cuda.synchronize()
        assert binding.attn_check(None) == 9
    finally:
        binding.attn_debug_inject(binding.FAULT_NONE)
        binding.attn_set_wait_limit(old)
    assert binding.attn_debug_inject(7) == 4  # unknown fault
    # normal operation again: bit-identical to the run before the fault
    again = run_backward(inp, o, lse, dev, deterministic=True)
    for a, b in zip(ref, again):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    _ = (np, GRAD_TOL, rel_fro, to_host_f64)


def test_rescale_counters_absent_in_shipped_build():
    """The forward's rescale counters exist only in a measurement build
    (ATTN_COUNT_RESCALE=1); the shipped library reports none."""
    from exact_attention_15_gb300 import binding
    assert binding.attn_debug_rescale_stats() is None
