"""Host-side argument checks of the Python binding (no GPU): the C ABI takes
its sizes from q and k alone, so the binding rejects tensors whose shapes,
dtypes, devices or layouts disagree with them before anything is launched."""

import pytest

torch = pytest.importorskip("torch")

from exact_attention_15_gb300 import binding  # noqa: E402


def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(*shape, dtype=dtype)


def _raises(match, fn, *a, **kw):
    with pytest.raises(ValueError, match=match):
        fn(*a, **kw)


def test_forward_shape_mismatches():
    q, k = _t(2, 16, 4, 64), _t(2, 16, 2, 64)
    _raises("differ outside the head dimension", binding.forward, q, k, _t(2, 15, 2, 64))
    _raises("differ outside the head dimension", binding.forward, q, k, _t(2, 16, 1, 64))
    _raises("head dimensions differ", binding.forward, q, _t(2, 16, 2, 32), _t(2, 16, 2, 32))
    _raises("batch sizes differ", binding.forward, q, _t(1, 16, 2, 64), _t(1, 16, 2, 64))
    _raises("4 dimensions", binding.forward, _t(16, 4, 64), k, k)
    cu = torch.tensor([0, 16], dtype=torch.int32)
    _raises("3 dimensions", binding.forward, q, k, k, cu_seqlens=cu)


def test_forward_rejects_host_or_wrong_dtype():
    q = _t(1, 8, 2, 64)
    _raises("contiguous bf16 CUDA", binding.forward, q, q, q)
    f = _t(1, 8, 2, 64, dtype=torch.float16)
    _raises("contiguous bf16 CUDA", binding.forward, f, f, f)


def test_backward_checks_head_dims_and_matching_tensors():
    q, k, v = _t(1, 8, 2, 192), _t(1, 8, 2, 128), _t(1, 8, 2, 128)
    _raises("q and k head dimensions differ", binding.backward, q, k, v, None, None, None)
    q = _t(1, 8, 2, 64)
    _raises("contiguous bf16 CUDA", binding.backward, q, q, q, q, _t(1, 2, 8, dtype=torch.float32), q)


def test_forward_checks_out_and_lse_before_launch(monkeypatch):
    """out / lse of the wrong shape are rejected even when q, k, v pass (the
    tensor checks are patched to accept host tensors here)."""
    monkeypatch.setattr(binding, "_check_inputs", lambda *a, **kw: None)
    q = _t(1, 8, 2, 64)
    _raises("out must be", binding.forward, q, q, q, out=_t(1, 8, 2, 32))
    _raises("lse must be", binding.forward, q, q, q, lse=_t(2, 8, dtype=torch.float32))
    _raises("lse must be", binding.forward, q, q, q, lse=_t(1, 2, 8))  # bf16, not fp32
    _raises("o must be", binding.backward, q, q, q, _t(1, 8, 2, 32), _t(1, 2, 8, dtype=torch.float32), q)
    _raises("dout must be", binding.backward, q, q, q, q, _t(1, 2, 8, dtype=torch.float32), _t(1, 8, 1, 64))
    _raises("lse must be", binding.backward, q, q, q, q, _t(1, 2, 9, dtype=torch.float32), q)
    # separate head dimensions: o and dout have v's width
    q1, v1 = _t(1, 8, 2, 192), _t(1, 8, 2, 128)
    _raises("o must be", binding.backward, q1, q1, v1, q1, _t(1, 2, 8, dtype=torch.float32), v1)
    _raises("dout must be", binding.backward, q1, q1, v1, v1, _t(1, 2, 8, dtype=torch.float32), q1)
