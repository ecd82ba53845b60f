"""Exact IO-aware attention for GB300 (sm_103a).

Forward with online softmax and per-row log-sum-exp, recomputing backward, both
in hand-written tcgen05/TMEM/TMA kernels behind the C ABI of ``libfa.so``
(``include/fa.h``).  Python here only marshals arguments.

    from exact_io_aware_flash_gb300 import forward, backward
    o, lse = forward(q, k, v, causal=True)
    dq, dk, dv = backward(q, k, v, o, lse, dO, causal=True)
"""
from ._lib import (FAError, backward, check_errors, forward, forward_fp8, forward_splitkv,  # noqa: F401
                   load, quantize_fp8, selftest_bounded_wait, set_backward_event_hooks, version,
                   workspace_size)
