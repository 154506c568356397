"""Helpers shared by the GPU parity tests: moving the seeded bf16 inputs to the
device, running the library through its binding, and comparing with the oracle.

Tolerances (fixed for this operator): O max-abs error <= 1.5e-2, LSE abs error
<= 2e-3, relative Frobenius error <= 2e-2 for each of dQ, dK and dV.
"""

from __future__ import annotations

import numpy as np

O_TOL = 1.5e-2
LSE_TOL = 2e-3
GRAD_TOL = 2e-2


def torch_mod():
    import torch
    return torch


def to_dev(bits):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def to_host_f64(t):
    torch = torch_mod()
    bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def as_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def device_inputs(inp):
    torch = torch_mod()
    dev = dict(q=to_dev(inp.q), k=to_dev(inp.k), v=to_dev(inp.v))
    if inp.do is not None:
        dev["do"] = to_dev(inp.do)
    dev["cu"] = None if inp.cu_seqlens is None else torch.from_numpy(inp.cu_seqlens).cuda()
    return dev


def run_forward(inp, dev=None):
    from exact_attention_15_gb300 import binding
    torch = torch_mod()
    dev = dev or device_inputs(inp)
    o, lse = binding.forward(dev["q"], dev["k"], dev["v"], scale=inp.scale, causal=inp.causal,
                             cu_seqlens=dev["cu"])
    torch.cuda.synchronize()
    assert binding.attn_check(None) == 0
    return o, lse, dev


def run_backward(inp, o, lse, dev, deterministic=False):
    from exact_attention_15_gb300 import binding
    torch = torch_mod()
    dq, dk, dv = binding.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], scale=inp.scale,
                                  causal=inp.causal, cu_seqlens=dev["cu"],
                                  deterministic=deterministic)
    torch.cuda.synchronize()
    assert binding.attn_check(None) == 0
    return dq, dk, dv


def rel_fro(a, b):
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def head_slices(inp, b, h):
    """(q, k, v, do) fp64 arrays of one (batch or sequence, query head)."""
    g = inp.H_q // inp.H_kv
    if inp.cu_seqlens is None:
        sl = lambda x, hh: as_f64(x[b, :, hh, :])
    else:
        a, e = int(inp.cu_seqlens[b]), int(inp.cu_seqlens[b + 1])
        sl = lambda x, hh: as_f64(x[a:e, hh, :])
    do = sl(inp.do, h) if inp.do is not None else None
    return sl(inp.q, h), sl(inp.k, h // g), sl(inp.v, h // g), do


def gpu_head(t, inp, b, h, kv=False):
    """Slice one head out of a device output tensor, as fp64 host array."""
    if inp.cu_seqlens is None:
        return to_host_f64(t[b, :, h, :])
    a, e = int(inp.cu_seqlens[b]), int(inp.cu_seqlens[b + 1])
    return to_host_f64(t[a:e, h, :])


def gpu_lse(lse, inp, b, h):
    if inp.cu_seqlens is None:
        return lse[b, h].double().cpu().numpy()
    a, e = int(inp.cu_seqlens[b]), int(inp.cu_seqlens[b + 1])
    return lse[h, a:e].double().cpu().numpy()
