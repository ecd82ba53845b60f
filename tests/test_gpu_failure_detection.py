"""Failure detection on the GPU without a fault: a wait that nothing completes
runs out after its limit, the kernel reports it through the device error word,
and the context stays usable for the next call."""
import math

import pytest
import torch

from exact_io_aware_flash_gb300 import FAError, _lib, check_errors, forward, selftest_bounded_wait
from exact_io_aware_flash_gb300.synth import Shape, make_inputs

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_context_survives():
    check_errors()  # start clean
    selftest_bounded_wait(50)
    with pytest.raises(FAError) as e:
        check_errors()
    assert e.value.code == _lib.FA_ERR_TIMEOUT
    check_errors()  # the word was cleared by the report
    # the context still runs work correctly
    inp = make_inputs(Shape(1, 2, 2, 256, 64), "fp16", seed=3, with_dO=False)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = forward(q, k, v, causal=True)
    check_errors()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_selftest_rejects_bad_limits():
    with pytest.raises(FAError):
        selftest_bounded_wait(0)
    with pytest.raises(FAError):
        selftest_bounded_wait(5000)
