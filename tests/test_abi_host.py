"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/attn.h declares, and rejects bad arguments with the
documented status codes before anything is launched."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_attention_15_gb300 import build, binding
    build.build()
    return binding.load()


def _declared():
    with open(os.path.join(ROOT, "include", "attn.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "attn_fwd" in names and "attn_bwd" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in attn.h but not exported"


def test_binding_covers_the_header(lib):
    from exact_attention_15_gb300 import binding
    assert set(_declared()) <= set(binding.exported_symbols())


def test_status_strings(lib):
    from exact_attention_15_gb300 import binding
    for code, name in binding.ATTN_STATUS.items():
        s = binding.status_string(code)
        assert s and s != "unknown status", (code, name)
    assert binding.status_string(999) == "unknown status"


# fake, 16-byte aligned addresses: every call below must return before it
# touches memory or a device
A = 0x10000


def _fwd(lib, **kw):
    a = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H_q=2, H_kv=2, N_q=128, N_k=128, d=64, causal=0,
             seqlens=None, scale=0.125)
    a.update(kw)
    return lib.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H_q"], a["H_kv"],
                        a["N_q"], a["N_k"], a["d"], a["causal"], a["seqlens"], a["scale"], None)


def _bwd(lib, **kw):
    a = dict(q=A, k=A, v=A, o=A, lse=A, do=A, dq=A, dk=A, dv=A, B=1, H_q=2, H_kv=2, N_q=128,
             N_k=128, d=64, causal=0, seqlens=None, scale=0.125, det=0, ws=A, wsb=1 << 40)
    a.update(kw)
    return lib.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"],
                        a["dv"], a["B"], a["H_q"], a["H_kv"], a["N_q"], a["N_k"], a["d"],
                        a["causal"], a["seqlens"], a["scale"], a["det"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), 3), (dict(d=256), 3),
    (dict(H_q=3, H_kv=2), 5), (dict(H_kv=0), 4),
    (dict(causal=1, N_k=64), 6),
    (dict(q=None), 1), (dict(lse=None), 1),
    (dict(k=A + 8), 2), (dict(o=A + 2), 2),
    (dict(B=-1), 4), (dict(N_q=-5), 4),
    (dict(scale=float("inf")), 4), (dict(scale=float("nan")), 4),
    (dict(seqlens=A, N_k=100), 6),
])
def test_fwd_argument_errors(lib, kw, code):
    assert _fwd(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(d=32), 3), (dict(H_q=4, H_kv=3), 5), (dict(causal=1, N_q=64), 6),
    (dict(dk=None), 1), (dict(do=None), 1), (dict(dq=A + 4), 2),
    (dict(ws=None), 7), (dict(wsb=16), 7), (dict(ws=A + 16), 2),
])
def test_bwd_argument_errors(lib, kw, code):
    assert _bwd(lib, **kw) == code


def _fwd_dims(lib, d_qk, d_v, **kw):
    a = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H_q=2, H_kv=2, N_q=128, N_k=128, causal=0,
             seqlens=None, scale=0.125)
    a.update(kw)
    return lib.attn_fwd_dims(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H_q"], a["H_kv"],
                             a["N_q"], a["N_k"], d_qk, d_v, a["causal"], a["seqlens"], a["scale"],
                             None)


@pytest.mark.parametrize("d_qk,d_v", [(192, 192), (128, 64), (64, 128), (192, 64), (256, 128),
                                      (128, 192), (96, 96)])
def test_fwd_dims_unsupported_pairs(lib, d_qk, d_v):
    assert _fwd_dims(lib, d_qk, d_v) == 3


@pytest.mark.parametrize("kw,code", [
    (dict(H_q=3, H_kv=2), 5), (dict(causal=1, N_k=64), 6), (dict(v=None), 1), (dict(o=A + 8), 2),
    (dict(scale=float("nan")), 4),
])
def test_fwd_dims_argument_errors(lib, kw, code):
    assert _fwd_dims(lib, 192, 128, **kw) == code


def test_empty_problems_need_no_pointers(lib):
    assert _fwd(lib, B=0, q=None, k=None, v=None, o=None, lse=None) == 0
    assert _bwd(lib, B=0, q=None, k=None, v=None, o=None, lse=None, do=None, dq=None, dk=None,
                dv=None, ws=None) == 0


def test_workspace_size(lib):
    # fixed length: fp32 dQ accumulator + D (+ semaphores and a counter), each 256-byte aligned
    B, H, N, d = 4, 16, 8192, 128
    acc = B * N * H * d * 4
    dvec = B * N * H * 4
    assert lib.attn_bwd_workspace_bytes(B, H, H, N, N, d, 0, 0) == acc + dvec
    sem = B * (N // 128) * H + 1
    assert lib.attn_bwd_workspace_bytes(B, H, H, N, N, d, 0, 1) == acc + dvec + ((sem * 4 + 255) // 256) * 256
    # packed: rows = N_q (the packed total), not B * N_q, and the sequence
    # order (B ints) with each sequence's first work item (B + 1 ints)
    assert lib.attn_bwd_workspace_bytes(16, 32, 8, 1000, 1000, 128, 1, 0) == \
        ((1000 * 32 * 128 * 4 + 255) // 256) * 256 + ((1000 * 32 * 4 + 255) // 256) * 256 + \
        (((2 * 16 + 1) * 4 + 255) // 256) * 256
    assert lib.attn_bwd_workspace_bytes(1, 2, 2, 10, 10, 96, 0, 0) == 0


def test_no_device_is_reported():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this checks the no-device path")
    from exact_attention_15_gb300 import build, binding
    build.build()
    lib = binding.load()
    assert _fwd(lib) == 10
    assert _bwd(lib) == 10
    assert _fwd_dims(lib, 192, 128) == 10


def test_package_exports_resolve(lib):
    import exact_attention_15_gb300 as pkg
    for n in pkg.__all__:
        assert callable(getattr(pkg, n)), n


@pytest.mark.parametrize("which", ["fwd", "bwd"])
def test_variant_setters(lib, which):
    """The kernel-variant hooks are host state only: they return the previous
    selection and reject unknown values without changing it."""
    from exact_attention_15_gb300 import binding
    setter = getattr(binding, f"attn_set_{which}_variant")
    one = getattr(binding, f"{which.upper()}_ONE_CTA")
    pair = getattr(binding, f"{which.upper()}_CTA_PAIR")
    old = setter(pair)
    try:
        assert setter(pair) == pair
        assert setter(-3) == -1
        assert setter(one) == pair
        assert setter(one) == one
    finally:
        setter(old)


def test_pair_forward_checks_arguments_first(lib):
    """With the CTA-pair forward selected, argument errors still come back
    before anything is launched."""
    from exact_attention_15_gb300 import binding
    old = binding.attn_set_fwd_variant(binding.FWD_CTA_PAIR)
    try:
        code = {name: c for c, name in binding.ATTN_STATUS.items()}
        assert _fwd(lib, d=128, H_q=4, H_kv=3) == code["ATTN_ERR_GQA_RATIO"]
        assert _fwd(lib, d=128, q=A + 8) == code["ATTN_ERR_ALIGNMENT"]
        assert _fwd(lib, d=128, causal=1, N_k=64) == code["ATTN_ERR_CAUSAL_SHAPE"]
        assert _fwd(lib, d=96) == code["ATTN_ERR_UNSUPPORTED_HEADDIM"]
        assert _fwd(lib, d=128, B=0, q=None, k=None, v=None, o=None, lse=None) == 0
    finally:
        binding.attn_set_fwd_variant(old)
