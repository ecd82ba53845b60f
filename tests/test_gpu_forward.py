"""GPU forward parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerances: O max-abs <= 2e-3 (fp16) / 1e-2 (bf16), LSE max-abs <= 1e-3.
Both sides consume the same seeded inputs rounded to the 16-bit dtype.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_flash_gb300 import FAError, check_errors, forward
from exact_io_aware_flash_gb300.synth import WORKLOADS, Shape, make_inputs

pytestmark = pytest.mark.gpu

TOL_O = {"fp16": 2e-3, "bf16": 1e-2}
TOL_LSE = 1e-3


def gpu_forward(inp, causal, scale):
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = forward(q, k, v, causal=causal, scale=scale)
    check_errors()
    return o, lse


def assert_matches(o_gpu, lse_gpu, o_ref, lse_ref, dtype, what=""):
    o_gpu = o_gpu.float().cpu().numpy()
    lse_gpu = lse_gpu.cpu().numpy()
    assert np.isfinite(o_gpu).all() and np.isfinite(lse_gpu).all(), what
    err_o = float(np.abs(o_gpu - o_ref).max())
    err_l = float(np.abs(lse_gpu - lse_ref).max())
    assert err_o <= TOL_O[dtype], f"{what}: O max-abs error {err_o:.3g} > {TOL_O[dtype]}"
    assert err_l <= TOL_LSE, f"{what}: LSE max-abs error {err_l:.3g} > {TOL_LSE}"
    return err_o, err_l


SMALL = [
    # B, Hq, Hkv, N, d
    (1, 1, 1, 1, 64), (1, 1, 1, 7, 128), (1, 2, 2, 64, 64), (2, 1, 1, 127, 128),
    (1, 2, 1, 128, 64), (1, 1, 1, 129, 128), (2, 2, 2, 255, 64), (1, 4, 2, 256, 128),
    (1, 3, 1, 300, 64), (1, 2, 2, 513, 128), (2, 4, 1, 640, 128),
]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,N,d", SMALL)
def test_forward_small_shapes(B, Hq, Hkv, N, d, causal, dtype):
    shape = Shape(B, Hq, Hkv, N, d)
    inp = make_inputs(shape, dtype, seed=7 + N + d, with_dO=False)
    scale = 1.0 / math.sqrt(d)
    o, lse = gpu_forward(inp, causal, scale)
    o_ref, lse_ref = oracle.forward(inp["q"], inp["k"], inp["v"], causal, scale)
    assert_matches(o, lse, o_ref, lse_ref, dtype, f"{shape} causal={causal}")


UNIT_ROUNDOFF = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8}


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("q_scale,scale", [(8.0, None), (1.0, 0.0), (1.0, -0.3), (30.0, None)])
def test_forward_score_ranges(q_scale, scale, dtype):
    """Large scores force the running maximum to move (rescaling path); zero and
    negative scales exercise uniform attention and a reversed score order.

    These inputs lie outside the evaluation workloads: with Q scaled up the
    softmax is nearly one-hot and |O| approaches max|V|, so the flat O tolerance
    no longer applies.  The bound used is the rounding of the arithmetic: P is
    rounded to the 16-bit type before P V (relative error <= u per term, so
    <= u * max|V| on the weighted sum) and O is rounded once on output (<= u|O|),
    u the unit roundoff of the type; fp32 accumulation adds far less.
    """
    shape = Shape(1, 2, 1, 700, 128)
    inp = make_inputs(shape, dtype, seed=99, with_dO=False, q_scale=q_scale)
    s = 1.0 / math.sqrt(128) if scale is None else scale
    u = UNIT_ROUNDOFF[dtype]
    vmax = float(inp["v"].float().abs().max())
    for causal in (False, True):
        o, lse = gpu_forward(inp, causal, s)
        o_ref, lse_ref = oracle.forward(inp["q"], inp["k"], inp["v"], causal, s)
        o_gpu = o.float().cpu().numpy()
        bound = u * (np.abs(o_ref) + vmax) + 1e-4
        worst = float((np.abs(o_gpu - o_ref) / bound).max())
        assert worst <= 1.0, f"q_scale={q_scale} scale={s} causal={causal}: {worst:.3f} x bound"
        assert np.abs(lse.cpu().numpy() - lse_ref).max() <= TOL_LSE


def _run_workload(name, causal, heads=None):
    """Full-size launch; the oracle checks every head (heads=None) or the listed (b, h)."""
    w = WORKLOADS[name]
    shape, dtype = w["shape"], w["dtype"]
    inp = make_inputs(shape, dtype, seed=w["seed"], with_dO=False)
    scale = 1.0 / math.sqrt(shape.d)
    o, lse = gpu_forward(inp, causal, scale)
    if heads is None:
        o_ref, lse_ref = oracle.forward(inp["q"], inp["k"], inp["v"], causal, scale)
        o_gpu, lse_gpu = o.float().cpu().numpy(), lse.cpu().numpy()
        for b in range(shape.B):
            for h in range(shape.Hq):
                assert_matches(torch.from_numpy(o_gpu[b, h]), torch.from_numpy(lse_gpu[b, h]),
                               o_ref[b, h], lse_ref[b, h], dtype, f"{name} head ({b},{h})")
        return
    g = shape.group
    for b, h in heads:
        hk = h // g
        q = inp["q"][b:b + 1, h:h + 1]
        k = inp["k"][b:b + 1, hk:hk + 1]
        v = inp["v"][b:b + 1, hk:hk + 1]
        o_ref, lse_ref = oracle.forward(q, k, v, causal, scale)
        assert_matches(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], o_ref, lse_ref, dtype,
                       f"{name} head ({b},{h})")


def test_workload_single_head_n128_d64_fp16():
    _run_workload("single_head_fwd_n128_d64_fp16", False, [(0, 0)])


@pytest.mark.parametrize("causal", [False, True])
def test_workload_b1_h8_n1024_d64_fp16(causal):
    _run_workload("fwd_b1_h8_n1024_d64_fp16", causal, [(0, h) for h in range(8)])


def test_workload_b4_h16_n4096_d128_bf16_causal():
    # every one of the 64 heads, so each head group of the launch order is covered
    _run_workload("fwd_b4_h16_n4096_d128_bf16_causal", True)


def test_workload_gqa_b2_hq32_hkv8_n8192_d128_bf16_causal():
    # every one of the 64 query heads (16 KV heads, groups of 4)
    _run_workload("gqa_fwd_b2_hq32_hkv8_n8192_d128_bf16_causal", True)


def test_forward_is_deterministic_and_writes_every_output():
    shape = Shape(2, 4, 2, 1000, 128)
    inp = make_inputs(shape, "bf16", seed=5, with_dO=False)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    outs = []
    for fill in (float("nan"), 0.0):
        o = torch.full_like(q, fill)
        lse = torch.full((2, 4, 1000), fill, dtype=torch.float32, device="cuda")
        forward(q, k, v, causal=True, out=o, lse=lse)
        check_errors()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        outs.append((o.clone(), lse.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", [(1, 2, 1, 300, 64, True), (2, 2, 2, 257, 128, False),
                                                  (1, 4, 4, 1000, 128, True)])
def test_forward_output_16_byte_aligned_only(B, Hq, Hkv, N, d, causal):
    """O whose base is 16- but not 32-byte aligned (the ABI's minimum) takes the
    kernel's 16-byte store path: same bits as a 32-byte aligned O, and the oracle."""
    shape = Shape(B, Hq, Hkv, N, d)
    inp = make_inputs(shape, "bf16", seed=11 + N, with_dO=False)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(d)
    o_al, lse_al = forward(q, k, v, causal=causal, scale=scale)
    n = B * Hq * N * d
    base = torch.full((n + 16,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o_16 = base[8:8 + n].view(B, Hq, N, d)  # 16-byte offset from a 256-byte aligned allocation
    assert o_16.data_ptr() % 16 == 0 and o_16.data_ptr() % 32 != 0 and o_al.data_ptr() % 32 == 0
    _, lse_16 = forward(q, k, v, causal=causal, scale=scale, out=o_16)
    check_errors()
    assert torch.equal(o_16, o_al) and torch.equal(lse_16, lse_al)
    assert torch.isnan(base[:8].float()).all() and torch.isnan(base[8 + n:].float()).all()
    o_ref, lse_ref = oracle.forward(inp["q"], inp["k"], inp["v"], causal, scale)
    assert_matches(o_16, lse_16, o_ref, lse_ref, "bf16", f"{shape} causal={causal}, 16-byte aligned O")


def test_forward_rejects_bad_arguments():
    q = torch.zeros(1, 2, 64, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(FAError) as e:
        forward(q, q, q)
    assert e.value.code == 2  # unsupported head dimension
    q = torch.zeros(1, 3, 64, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 2, 64, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(FAError) as e:
        forward(q, k, k)
    assert e.value.code == 1  # Hq % Hkv != 0
    base = torch.zeros(1 * 1 * 64 * 64 + 8, dtype=torch.float16, device="cuda")
    mis = base[1:1 + 64 * 64].view(1, 1, 64, 64)  # 2-byte offset: not 16-byte aligned
    with pytest.raises(FAError) as e:
        forward(mis, mis, mis)
    assert e.value.code == 2
