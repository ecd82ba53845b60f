"""fa_backward_noalloc against fa_backward, through the C ABI.

fa_backward_noalloc serves callers that may not allocate device memory (a
program that reserves all device memory up front, a plugin given no
allocator): it takes its scratch from an array built into the library instead
of a caller-provided workspace.  The backward sums every gradient in a fixed
order, so both entry points must give bitwise identical dq, dk and dv (which
is stricter than the backward parity tolerance, relative Frobenius error
<= 1e-2, that both also meet against the oracle elsewhere).

Two calls in a row, on different inputs and sizes: the second call finds the
array holding what the first call left there, so it shows that a call does
not depend on the array's previous contents.

This file is named so that pytest collects it last.
"""
import ctypes
import math

import pytest
import torch

from exact_io_aware_flash_gb300 import _lib, backward, build, check_errors, forward
from exact_io_aware_flash_gb300.synth import Shape, make_inputs

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, k, v, o, lse, dO, causal, scale):
    B, Hq, N, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rc = lib.fa_backward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), dO.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                 dv.data_ptr(), B, Hq, k.shape[1], N, d, int(causal), scale,
                                 _lib.FA_DTYPE_BF16, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.fa_last_error().decode()
    return dq, dk, dv


def test_noalloc_backward_matches_workspace_backward_twice():
    build.build()
    lib = _lib.load()
    scale = 1.0 / math.sqrt(128)
    # The second call is larger than the first (so it reads array elements the
    # first call never wrote) and runs on other inputs (so stale values the
    # first call left behind would change its result).
    for call, (shape, seed) in enumerate(((Shape(1, 4, 2, 700, 128), 4242),
                                          (Shape(2, 8, 2, 1000, 128), 4343))):
        inp = make_inputs(shape, "bf16", seed=seed)
        q, k, v, dO = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
        o, lse = forward(q, k, v, causal=True, scale=scale)
        ref = backward(q, k, v, o, lse, dO, causal=True, scale=scale)
        check_errors()
        got = _noalloc(lib, q, k, v, o, lse, dO, True, scale)
        torch.cuda.synchronize()
        check_errors()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.isfinite(g.float()).all(), f"call {call}: {name} not finite"
            assert torch.equal(g, r), (
                f"call {call}: {name} differs from fa_backward "
                f"(max abs diff {float((g.float() - r.float()).abs().max()):.3g})")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    build.build()
    lib = _lib.load()
    # 4 bytes of D per query row: 64*64*4096 rows need 64 MiB, more than the 40 MiB array.
    B, Hq, N, d = 64, 64, 4096, 128
    assert lib.fa_backward_workspace_size(B, Hq, N, d) > 40 * 1024 * 1024
    fake = ctypes.c_void_p(4096)  # rejected before any pointer is used
    rc = lib.fa_backward_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                 B, Hq, Hq, N, d, 1, 0.1, _lib.FA_DTYPE_BF16, None)
    assert rc == _lib.FA_ERR_UNSUPPORTED
    assert b"scratch" in lib.fa_last_error()
