"""Malformed packed-sequence offsets: every kernel clamps the rows it decodes
into the T packed rows the tensors hold, so a cu_seqlens array that runs past T,
decreases, or does not start at 0 never makes a read or write leave the caller's
buffers. The call reports ATTN_ERR_SEQLENS through attn_check, and the context
stays usable.

Each output tensor is allocated with a guard region after its last element,
filled with a sentinel bit pattern, and the guard must come back unchanged."""

import numpy as np
import pytest

from exact_attention_15_gb300 import workloads as W

pytestmark = pytest.mark.gpu

T = 700          # packed rows every tensor holds
GUARD = 4096     # guard elements after each output tensor
SENTINEL = 0x7FC1  # a bf16 NaN payload no kernel writes
H_Q, H_KV = 4, 2
SEQLENS_ERR = 12   # ATTN_ERR_SEQLENS

BAD_ARRAYS = {
    "past_the_end": [0, 300, 500, 900],
    "decreasing": [0, 400, 150, 700],
    "nonzero_start": [100, 300, 500, 700],
}


def _guarded_bf16(n, torch):
    buf = torch.full((n + GUARD,), SENTINEL, dtype=torch.int16, device="cuda")
    return buf, buf[:n].view(torch.bfloat16)


def _guard_intact(buf, n, torch):
    return bool((buf[n:] == SENTINEL).all())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", sorted(BAD_ARRAYS))
@pytest.mark.parametrize("causal", [False, True])
def test_bad_offsets_stay_inside_buffers(case, causal, d):
    import torch
    from exact_attention_15_gb300 import binding
    assert binding.attn_check(None) == 0
    inp = W.custom(1, H_Q, H_KV, T, T, d, causal=causal, seed=77)
    dev = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)
    q, k, v, do = (dev(x[0]) for x in (inp.q, inp.k, inp.v, inp.do))  # [T, H, d]
    cu = torch.tensor(BAD_ARRAYS[case], dtype=torch.int32, device="cuda")
    B = cu.numel() - 1
    n_q, n_k = T * H_Q * d, T * H_KV * d
    o_buf, o = _guarded_bf16(n_q, torch)
    lse_buf = torch.full((H_Q * T + GUARD,), float("nan"), dtype=torch.float32, device="cuda")
    lse = lse_buf[:H_Q * T]
    st = binding.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          B, H_Q, H_KV, T, T, d, causal, cu.data_ptr(), inp.scale, None)
    assert st == 0
    torch.cuda.synchronize()
    assert binding.attn_check(None) == SEQLENS_ERR
    assert binding.attn_check(None) == 0  # the record is cleared
    assert _guard_intact(o_buf, n_q, torch)
    assert torch.isnan(lse_buf[H_Q * T:]).all()

    dq_buf, dq = _guarded_bf16(n_q, torch)
    dk_buf, dk = _guarded_bf16(n_k, torch)
    dv_buf, dv = _guarded_bf16(n_k, torch)
    for det in (False, True):
        ws_bytes = binding.attn_bwd_workspace_bytes(B, H_Q, H_KV, T, T, d, True, det)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        st = binding.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), B, H_Q, H_KV, T, T, d, causal, cu.data_ptr(),
                              inp.scale, det, ws.data_ptr(), ws_bytes, None)
        assert st == 0
        torch.cuda.synchronize()
        assert binding.attn_check(None) == SEQLENS_ERR
        for buf, n in ((dq_buf, n_q), (dk_buf, n_k), (dv_buf, n_k)):
            assert _guard_intact(buf, n, torch)


def test_bad_offsets_pair_forward():
    """The CTA-pair forward clamps and reports the same way."""
    import torch
    from exact_attention_15_gb300 import binding
    old = binding.attn_set_fwd_variant(binding.FWD_CTA_PAIR)
    try:
        inp = W.custom(1, H_Q, H_KV, T, T, 128, causal=True, seed=78)
        dev = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)
        q, k, v = (dev(x[0]) for x in (inp.q, inp.k, inp.v))
        n_q = T * H_Q * 128
        for case in sorted(BAD_ARRAYS):
            cu = torch.tensor(BAD_ARRAYS[case], dtype=torch.int32, device="cuda")
            o_buf, o = _guarded_bf16(n_q, torch)
            lse_buf = torch.full((H_Q * T + GUARD,), float("nan"), dtype=torch.float32, device="cuda")
            st = binding.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse_buf.data_ptr(), cu.numel() - 1, H_Q, H_KV, T, T, 128, True,
                                  cu.data_ptr(), inp.scale, None)
            assert st == 0
            torch.cuda.synchronize()
            assert binding.attn_check(None) == SEQLENS_ERR, case
            assert _guard_intact(o_buf, n_q, torch), case
            assert torch.isnan(lse_buf[H_Q * T:]).all(), case
    finally:
        binding.attn_set_fwd_variant(old)


def test_valid_offsets_report_nothing_after_bad_ones():
    """A valid array right after a bad one: no error, and the usual parity."""
    import torch
    from gpu_common import O_TOL, run_forward
    import oracle
    from gpu_common import gpu_head, head_slices
    inp = W.custom(3, H_Q, H_KV, 0, 0, 64, causal=True, seed=79, seqlens=[100, 300, 170])
    o, lse, devs = run_forward(inp)
    for s in range(3):
        q, k, v, _ = head_slices(inp, s, 1)
        ref_o, _ = oracle.head_forward(q, k, v, inp.scale, True)
        assert np.max(np.abs(gpu_head(o, inp, s, 1) - ref_o)) <= O_TOL
    _ = torch
