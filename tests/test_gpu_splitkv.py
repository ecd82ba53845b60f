"""GPU parity of the split-KV (decoding) forward against the fp64 rectangular oracle.

Tolerances as for the forward: O max-abs <= 2e-3 (fp16) / 1e-2 (bf16), LSE <= 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_flash_gb300 import FAError, check_errors, forward, forward_splitkv
from exact_io_aware_flash_gb300.synth import DTYPES

pytestmark = pytest.mark.gpu

TOL_O = {"fp16": 2e-3, "bf16": 1e-2}


def _inputs(B, Hq, Hkv, Nq, Nk, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, Nq, d, generator=g).to(DTYPES[dtype])
    k = torch.randn(B, Hkv, Nk, d, generator=g).to(DTYPES[dtype])
    v = torch.randn(B, Hkv, Nk, d, generator=g).to(DTYPES[dtype])
    return q, k, v


CASES = [
    # B, Hq, Hkv, Nq, Nk, d, dtype, splits
    (1, 1, 1, 1, 1, 64, "fp16", 0),
    (2, 8, 2, 1, 1000, 128, "bf16", 0),
    (1, 32, 8, 1, 33000, 128, "bf16", 0),
    (2, 4, 4, 7, 513, 64, "fp16", 3),
    (1, 8, 1, 16, 4096, 128, "bf16", 1),
    (1, 2, 1, 200, 300, 128, "bf16", 0),   # 400 stacked rows: several query tiles
    (1, 4, 2, 3, 384, 128, "fp16", 50),    # more splits requested than key tiles
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,dtype,splits", CASES)
def test_splitkv_matches_oracle(B, Hq, Hkv, Nq, Nk, d, dtype, splits):
    q, k, v = _inputs(B, Hq, Hkv, Nq, Nk, d, dtype, seed=Nq * 7 + Nk)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward_splitkv(q.cuda(), k.cuda(), v.cuda(), scale=scale, num_splits=splits)
    check_errors()
    o_ref, lse_ref = oracle.forward_rect(q, k, v, scale)
    err_o = float(np.abs(o.float().cpu().numpy() - o_ref).max())
    err_l = float(np.abs(lse.cpu().numpy() - lse_ref).max())
    assert err_o <= TOL_O[dtype], err_o
    assert err_l <= 1e-3, err_l


def test_splitkv_square_case_agrees_with_forward_and_is_deterministic():
    q, k, v = _inputs(1, 4, 2, 640, 640, 128, "bf16", seed=5)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = forward_splitkv(q, k, v, num_splits=4)
    o2, l2 = forward_splitkv(q, k, v, num_splits=4)
    of, lf = forward(q, k, v, causal=False)
    check_errors()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert float((o1.float() - of.float()).abs().max()) <= 1e-2
    assert float((l1 - lf).abs().max()) <= 1e-3


def test_splitkv_rejects_bad_arguments():
    q = torch.zeros(1, 2, 1, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(FAError):
        forward_splitkv(q, k, k)
