"""CPU oracle for exact softmax attention (forward and backward), in float64.

TEST INFRASTRUCTURE ONLY. Nothing in the product path (the CUDA library and its
Python binding) may import, call or link this package; only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs
of ``bench.py`` use it. It shares no code with the CUDA path: it has its own
masks, its own softmax and its own gradient formulas, written from the
definitions on the source pages, and it never sees a value the GPU produced
except to compare against it.

Modules
-------
``attention``  the plain definitions: materialised S and P, one (batch, head) at
               a time; the backward pass from the chain rule; GQA summation.
``online``     the tile-merge algorithms the fast method is built from: the
               (m, l, u) online merge and its lazily-rescaled variant, written in
               the pages' order, used to pin the algebra the kernels rely on.
``scalar``     a pure-Python scalar restatement for tiny inputs, used to pin the
               numpy version by brute force.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(worked example, closed forms, invariants, finite differences, brute force).
"""

from .attention import (  # noqa: F401
    head_forward,
    head_backward,
    attention_forward,
    attention_backward,
    visible_mask,
)
from .online import online_merge, online_merge_lazy, blockwise_average_merge  # noqa: F401
