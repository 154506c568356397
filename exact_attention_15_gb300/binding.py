"""Thin Python binding over the C ABI in ``include/attn.h`` (ctypes).

The functions named like the C entry points take raw device pointers (ints)
and sizes exactly as the C functions do; ``forward`` / ``backward`` are
convenience wrappers that take torch CUDA tensors, allocate the outputs (and
the backward workspace) with torch, and pass pointers and torch's current
stream. Argument marshalling only: every step of the computation runs in the
library's CUDA kernels. There is no fallback: if the library has not been
built, or a call fails, an exception is raised.
"""

from __future__ import annotations

import ctypes
import math
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libattn_gb300.so")
_lib = None

ATTN_STATUS = {
    0: "ATTN_OK", 1: "ATTN_ERR_NULL_PTR", 2: "ATTN_ERR_ALIGNMENT", 3: "ATTN_ERR_UNSUPPORTED_HEADDIM",
    4: "ATTN_ERR_BAD_SHAPE", 5: "ATTN_ERR_GQA_RATIO", 6: "ATTN_ERR_CAUSAL_SHAPE",
    7: "ATTN_ERR_WORKSPACE", 8: "ATTN_ERR_CUDA", 9: "ATTN_ERR_TIMEOUT", 10: "ATTN_ERR_NO_DEVICE",
    11: "ATTN_ERR_UNSUPPORTED_DEVICE", 12: "ATTN_ERR_SEQLENS",
}

# name -> (restype, argtypes)
_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, ctypes.c_float, _P]),
    "attn_fwd_dims": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, ctypes.c_float, _P]),
    "attn_bwd_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P,
                      ctypes.c_float, _I, _P, ctypes.c_size_t, _P]),
    "attn_bwd_dims_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I, _I, _I, _I]),
    "attn_bwd_dims": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P,
                           ctypes.c_float, _I, _P, ctypes.c_size_t, _P]),
    "attn_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P,
                              ctypes.c_float, _I, _P]),
    "attn_check": (_I, [_P]),
    "attn_status_string": (ctypes.c_char_p, [_I]),
    "attn_debug_exp2": (_I, [_P, _P, _I, _I, _P]),
    "attn_set_wait_limit": (ctypes.c_longlong, [ctypes.c_longlong]),
    "attn_set_bwd_variant": (_I, [_I]),
    "attn_set_fwd_variant": (_I, [_I]),
    "attn_debug_inject": (_I, [_I]),
    "attn_debug_stall": (_I, [_P]),
    "attn_debug_rescale_stats": (_I, [_P, _I]),
    "attn_debug_fwd_plan": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, ctypes.c_longlong]),
    "attn_profile_enable": (_I, [_I]),
    "attn_profile_read": (_I, [_P, _I]),
}

KERNEL_NAMES = {1: "attn_fwd_kernel", 2: "attn_bwd_pre_kernel", 3: "attn_bwd_main_kernel",
                4: "attn_bwd_post_kernel", 5: "exp2_probe_kernel", 6: "stall_probe_kernel",
                7: "fwd_plan_kernel", 8: "attn_fwd_pair_kernel", 9: "attn_bwd_main_kernel_pass2",
                10: "bwd_plan_kernel"}
FAULT_NONE = 0
FAULT_SKIP_DQ_RELEASE = 1
BWD_ONE_CTA = 0
BWD_CTA_PAIR = 1
FWD_ONE_CTA = 0
FWD_CTA_PAIR = 1


class ProfileRecord(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("ms", ctypes.c_float)]


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {ATTN_STATUS.get(status, status)} ({status_string(status)})")


def library_path() -> str:
    return _LIB_PATH


def load():
    """Loads the shared library (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                f"CUDA library not built: {_LIB_PATH} is missing "
                "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def exported_symbols():
    return list(_SIGS)


# ------------------------------------------------------------------ raw C entry points

def attn_fwd(q, k, v, o, lse, B, H_q, H_kv, N_q, N_k, d, causal, seqlens, scale, stream) -> int:
    return load().attn_fwd(q, k, v, o, lse, B, H_q, H_kv, N_q, N_k, d, int(causal), seqlens,
                           float(scale), stream)


def attn_fwd_dims(q, k, v, o, lse, B, H_q, H_kv, N_q, N_k, d_qk, d_v, causal, seqlens, scale,
                  stream) -> int:
    return load().attn_fwd_dims(q, k, v, o, lse, B, H_q, H_kv, N_q, N_k, d_qk, d_v, int(causal),
                                seqlens, float(scale), stream)


def attn_bwd_workspace_bytes(B, H_q, H_kv, N_q, N_k, d, varlen, deterministic) -> int:
    return load().attn_bwd_workspace_bytes(B, H_q, H_kv, N_q, N_k, d, int(varlen), int(deterministic))


def attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H_q, H_kv, N_q, N_k, d, causal, seqlens,
             scale, deterministic, workspace, workspace_bytes, stream) -> int:
    return load().attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H_q, H_kv, N_q, N_k, d,
                           int(causal), seqlens, float(scale), int(deterministic), workspace,
                           workspace_bytes, stream)


def attn_bwd_dims_workspace_bytes(B, H_q, H_kv, N_q, N_k, d_qk, d_v, varlen, deterministic) -> int:
    return load().attn_bwd_dims_workspace_bytes(B, H_q, H_kv, N_q, N_k, d_qk, d_v, int(varlen),
                                                int(deterministic))


def attn_bwd_dims(q, k, v, o, lse, dout, dq, dk, dv, B, H_q, H_kv, N_q, N_k, d_qk, d_v, causal,
                  seqlens, scale, deterministic, workspace, workspace_bytes, stream) -> int:
    return load().attn_bwd_dims(q, k, v, o, lse, dout, dq, dk, dv, B, H_q, H_kv, N_q, N_k, d_qk,
                                d_v, int(causal), seqlens, float(scale), int(deterministic),
                                workspace, workspace_bytes, stream)


def attn_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, H_q, H_kv, N_q, N_k, d, causal,
                     seqlens, scale, deterministic, stream) -> int:
    """attn_bwd served from the library's own fixed scratch buffer (no workspace,
    no allocation); for callers that cannot allocate device memory."""
    return load().attn_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, H_q, H_kv, N_q, N_k, d,
                                   int(causal), seqlens, float(scale), int(deterministic), stream)


NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def attn_check(stream=None) -> int:
    return load().attn_check(stream)


def status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


attn_status_string = status_string


def attn_debug_exp2(x, y, n, mode, stream) -> int:
    return load().attn_debug_exp2(x, y, n, mode, stream)


def attn_debug_inject(fault: int) -> int:
    return load().attn_debug_inject(int(fault))


def attn_debug_rescale_stats(reset=True):
    """The forward's rescale counters (a library built with ATTN_COUNT_RESCALE=1):
    dict(warp_steps, warp_rescales, rows_moved, row_steps), or None when the
    library has no counters."""
    out = (ctypes.c_ulonglong * 4)()
    n = load().attn_debug_rescale_stats(ctypes.cast(out, _P), int(bool(reset)))
    if n < 0:
        raise AttnError(-n, "attn_debug_rescale_stats")
    if n == 0:
        return None
    return dict(warp_steps=out[0], warp_rescales=out[1], rows_moved=out[2], row_steps=out[3])


def attn_debug_stall(stream=None) -> int:
    return load().attn_debug_stall(stream)


FWD_ONE_CTA_PER_TILE = 0
FWD_STRIDING = 1
FWD_BALANCED_LIST = 2
FWD_CLAIMED = 3


def attn_debug_fwd_plan(B, H_q, H_kv, N_q, N_k, d_qk, d_v, causal, varlen, n_sm, want_lists=True):
    """The forward's launch plan for a shape, computed on the host (no GPU):
    dict(mode, grid, tiles, sec_heads, n_mblocks, pair_heads) and, for the balanced-list mode,
    'start' (per-CTA offsets, grid + 1) and 'tiles_of' (the concatenated lists).
    Raises on an argument error."""
    info = (ctypes.c_longlong * 6)()
    lib = load()
    st = lib.attn_debug_fwd_plan(B, H_q, H_kv, N_q, N_k, d_qk, d_v, int(causal), int(varlen),
                                 n_sm, ctypes.cast(info, _P), None, 0)
    if st != 0:
        raise ValueError(ATTN_STATUS.get(st, st))
    out = dict(mode=info[0], grid=info[1], tiles=info[2], sec_heads=info[3], n_mblocks=info[4],
               pair_heads=info[5])
    if want_lists and out["mode"] == FWD_BALANCED_LIST:
        cap = out["grid"] + 1 + out["tiles"]
        buf = (ctypes.c_int * cap)()
        st = lib.attn_debug_fwd_plan(B, H_q, H_kv, N_q, N_k, d_qk, d_v, int(causal), int(varlen),
                                     n_sm, ctypes.cast(info, _P), ctypes.cast(buf, _P), cap)
        if st != 0:
            raise ValueError(ATTN_STATUS.get(st, st))
        g = out["grid"]
        out["start"] = list(buf[:g + 1])
        out["tiles_of"] = list(buf[g + 1:cap])
    return out


def attn_set_wait_limit(cycles: int) -> int:
    return load().attn_set_wait_limit(int(cycles))


def attn_set_bwd_variant(variant: int) -> int:
    """BWD_ONE_CTA (default) or BWD_CTA_PAIR for the d = 128 backward; returns
    the previous selection (-1 for an unknown value)."""
    return load().attn_set_bwd_variant(int(variant))


def attn_set_fwd_variant(variant: int) -> int:
    """FWD_ONE_CTA (default) or FWD_CTA_PAIR for the d_qk = d_v = 128 forward;
    returns the previous selection (-1 for an unknown value)."""
    return load().attn_set_fwd_variant(int(variant))


def attn_profile_enable(enable: bool) -> int:
    return load().attn_profile_enable(int(bool(enable)))


def attn_profile_read(max_records: int = 65536):
    """Returns [(kernel_name, ms), ...] for launches since the last read."""
    buf = (ProfileRecord * max_records)()
    n = load().attn_profile_read(ctypes.cast(buf, ctypes.c_void_p), max_records)
    if n < 0:
        raise AttnError(-n, "attn_profile_read")
    return [(KERNEL_NAMES.get(buf[i].kernel, str(buf[i].kernel)), float(buf[i].ms)) for i in range(n)]


# ------------------------------------------------------------------ torch convenience layer

def _shape(q, k, cu_seqlens):
    if cu_seqlens is not None:
        T, H_q, d = q.shape
        H_kv = k.shape[1]
        return len(cu_seqlens) - 1, H_q, H_kv, T, k.shape[0], d
    B, N_q, H_q, d = q.shape
    return B, H_q, k.shape[2], N_q, k.shape[1], d


def _check_inputs(q, k, v, cu_seqlens):
    """Shapes first (so that a mismatch is reported as such), then dtype, device
    and layout: the C ABI takes sizes from q and k only, so v must match them."""
    import torch
    nd = 3 if cu_seqlens is not None else 4
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dim() != nd:
            raise ValueError(f"{name} must have {nd} dimensions "
                             f"({'[T, H, d] with cu_seqlens' if nd == 3 else '[B, N, H, d]'}), "
                             f"got {tuple(t.shape)}")
    if v.shape[:-1] != k.shape[:-1]:
        raise ValueError(f"v {tuple(v.shape)} and k {tuple(k.shape)} differ outside the head dimension")
    if k.shape[-1] != q.shape[-1]:
        raise ValueError(f"q and k head dimensions differ: {q.shape[-1]} vs {k.shape[-1]}")
    if nd == 4 and k.shape[0] != q.shape[0]:
        raise ValueError(f"q and k batch sizes differ: {q.shape[0]} vs {k.shape[0]}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")
    if cu_seqlens is not None:
        if (cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2
                or not cu_seqlens.is_contiguous() or cu_seqlens.device != q.device):
            raise ValueError("cu_seqlens must be a contiguous 1-D int32 tensor of at least two "
                             "entries on q's device")


def _check_tensor(name, t, shape, dtype, device):
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_contiguous() or t.device != device:
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} on "
                         f"{device}, got {t.dtype} {tuple(t.shape)} on {t.device}")


def _lse_shape(B, H_q, N_q, cu_seqlens):
    return (H_q, N_q) if cu_seqlens is not None else (B, H_q, N_q)


def _stream_ptr():
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(status, what):
    if status != 0:
        raise AttnError(status, what)


def forward(q, k, v, scale=None, causal=False, cu_seqlens=None, out=None, lse=None):
    """q [B, N_q, H_q, d_qk] (or packed [T, H_q, d_qk] with cu_seqlens), k with
    d_qk and v with d_v columns, bf16 CUDA tensors. Returns (o [.., d_v], lse).
    The default scale is 1/sqrt(d_qk)."""
    import torch
    _check_inputs(q, k, v, cu_seqlens)
    B, H_q, H_kv, N_q, N_k, d = _shape(q, k, cu_seqlens)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o_shape = q.shape[:-1] + (v.shape[-1],)
    if out is not None:
        _check_tensor("out", out, o_shape, torch.bfloat16, q.device)
    o = out if out is not None else torch.empty(o_shape, dtype=q.dtype, device=q.device)
    if lse is not None:
        _check_tensor("lse", lse, _lse_shape(B, H_q, N_q, cu_seqlens), torch.float32, q.device)
    else:
        lse = torch.empty(_lse_shape(B, H_q, N_q, cu_seqlens), dtype=torch.float32, device=q.device)
    cu_ptr = cu_seqlens.data_ptr() if cu_seqlens is not None else None
    d_v = v.shape[-1]
    _check(attn_fwd_dims(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                         B, H_q, H_kv, N_q, N_k, d, d_v, causal, cu_ptr, scale, _stream_ptr()),
           "attn_fwd_dims")
    return o, lse


def backward(q, k, v, o, lse, dout, scale=None, causal=False, cu_seqlens=None,
             deterministic=False, workspace=None):
    """Returns (dq, dk, dv): dq like q, dk like k, dv like v (q and k have d_qk
    columns, v, o and dout d_v). The workspace is allocated with torch unless
    given. The default scale is 1/sqrt(d_qk)."""
    import torch
    _check_inputs(q, k, v, cu_seqlens)
    B, H_q, H_kv, N_q, N_k, d = _shape(q, k, cu_seqlens)
    d_v = v.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o_shape = q.shape[:-1] + (d_v,)
    _check_tensor("o", o, o_shape, torch.bfloat16, q.device)
    _check_tensor("dout", dout, o_shape, torch.bfloat16, q.device)
    _check_tensor("lse", lse, _lse_shape(B, H_q, N_q, cu_seqlens), torch.float32, q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    nbytes = attn_bwd_dims_workspace_bytes(B, H_q, H_kv, N_q, N_k, d, d_v, cu_seqlens is not None,
                                           deterministic)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    elif not workspace.is_contiguous() or workspace.device != q.device:
        raise ValueError("workspace must be a contiguous tensor on q's device")
    cu_ptr = cu_seqlens.data_ptr() if cu_seqlens is not None else None
    _check(attn_bwd_dims(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                         dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                         B, H_q, H_kv, N_q, N_k, d, d_v, causal, cu_ptr, scale, deterministic,
                         workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                         _stream_ptr()),
           "attn_bwd_dims")
    return dq, dk, dv
