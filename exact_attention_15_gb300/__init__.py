"""GB300-native exact softmax attention (forward and backward) for sm_103a.

The compute lives in hand-written CUDA kernels behind a small C ABI
(``include/attn.h``); this package is the thin Python binding over it
(``binding``), the build step (``build``) and the seeded synthetic inputs used
by the tests and the benchmark (``workloads``).

Importing the package does not load the CUDA library; the first call of a
binding function does, and it fails loudly when the library is missing.
"""

__all__ = ["attn_fwd", "attn_fwd_dims", "attn_bwd", "attn_bwd_noalloc", "attn_bwd_workspace_bytes",
           "attn_status_string", "attn_check", "attn_set_wait_limit", "attn_set_fwd_variant",
           "attn_set_bwd_variant", "forward", "backward"]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
