"""attn_bwd_noalloc: the backward pass served from the library's own fixed
scratch buffer, for callers that cannot allocate device memory when they run
it (a plugin whose host program owns all device memory and offers no
allocator, or a latency-critical loop that must not stall on cudaMalloc).

Checked through the C ABI against the regular attn_bwd (which takes a
caller-allocated workspace) on the same inputs, within the gradient tolerance
the parity tests use, on two calls in a row (the second call starts from the
first call's leftovers in the shared buffer). This file is named so that pytest
collects it last.
"""

import numpy as np
import pytest

from exact_attention_15_gb300 import workloads as W
from gpu_common import GRAD_TOL, device_inputs, rel_fro, to_host_f64

pytestmark = pytest.mark.gpu

CASES = {
    "fixed_causal_gqa": dict(B=2, H_q=4, H_kv=2, N_q=700, N_k=700, d=128, causal=True),
    "packed_d64": dict(B=0, H_q=2, H_kv=1, N_q=0, N_k=0, d=64, causal=True, seqlens=[33, 400, 129]),
    "fixed_noncausal_d64": dict(B=1, H_q=2, H_kv=2, N_q=300, N_k=450, d=64, causal=False),
}


def _shape_args(inp):
    if inp.cu_seqlens is not None:
        return len(inp.cu_seqlens) - 1, inp.H_q, inp.H_kv, inp.N_q, inp.N_k, inp.d
    return inp.B, inp.H_q, inp.H_kv, inp.N_q, inp.N_k, inp.d


def _outputs(dev):
    import torch
    return torch.empty_like(dev["q"]), torch.empty_like(dev["k"]), torch.empty_like(dev["v"])


def _call(fn, inp, dev, o, lse, outs, deterministic, workspace=None):
    import torch
    from exact_attention_15_gb300 import binding
    B, H_q, H_kv, N_q, N_k, d = _shape_args(inp)
    dq, dk, dv = outs
    cu = dev["cu"].data_ptr() if dev["cu"] is not None else None
    stream = torch.cuda.current_stream().cuda_stream
    common = (dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(), o.data_ptr(),
              lse.data_ptr(), dev["do"].data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
              B, H_q, H_kv, N_q, N_k, d, inp.causal, cu, inp.scale, deterministic)
    if fn == "noalloc":
        st = binding.attn_bwd_noalloc(*common, stream)
    else:
        st = binding.attn_bwd(*common, workspace.data_ptr(), workspace.numel(), stream)
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("deterministic", [0, 1])
@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_workspace_backward(name, deterministic):
    import torch
    from exact_attention_15_gb300 import binding
    inp = W.custom(seed=300 + len(name), **CASES[name])
    dev = device_inputs(inp)
    o, lse = binding.forward(dev["q"], dev["k"], dev["v"], scale=inp.scale, causal=inp.causal,
                             cu_seqlens=dev["cu"])
    B, H_q, H_kv, N_q, N_k, d = _shape_args(inp)
    nbytes = binding.attn_bwd_workspace_bytes(B, H_q, H_kv, N_q, N_k, d, inp.cu_seqlens is not None,
                                              deterministic)
    assert 0 < nbytes <= binding.NOALLOC_SCRATCH_BYTES
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ref = _outputs(dev)
    assert _call("workspace", inp, dev, o, lse, ref, deterministic, ws) == 0
    ref64 = [to_host_f64(t) for t in ref]
    for call in range(2):
        got = _outputs(dev)
        for t in got:
            t.fill_(float("nan"))
        assert _call("noalloc", inp, dev, o, lse, got, deterministic) == 0, f"call {call}"
        assert binding.attn_check(None) == 0
        for name_g, g, r in zip(("dq", "dk", "dv"), got, ref64):
            e = rel_fro(to_host_f64(g), r)
            assert e <= GRAD_TOL, f"{name_g} differs from attn_bwd by {e} on call {call}"
        if deterministic:
            for g, r in zip(got, ref):
                assert torch.equal(g.view(torch.int16), r.view(torch.int16))


def test_noalloc_rejects_oversize_problem():
    import torch
    from exact_attention_15_gb300 import binding
    B, H, N, d = 1, 16, 16384, 128  # needs ~138 MB of scratch, more than the buffer holds
    assert binding.attn_bwd_workspace_bytes(B, H, H, N, N, d, 0, 0) > binding.NOALLOC_SCRATCH_BYTES
    x = torch.zeros(B, N, H, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, H, N, dtype=torch.float32, device="cuda")
    dq = torch.full_like(x, 7.0)
    st = binding.attn_bwd_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                                  lse.data_ptr(), x.data_ptr(), dq.data_ptr(), dq.data_ptr(),
                                  dq.data_ptr(), B, H, H, N, N, d, 0, None, 0.088, 0,
                                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 7, binding.status_string(st)
    assert torch.all(dq == 7.0), "a rejected call must not write its outputs"
    _ = np
