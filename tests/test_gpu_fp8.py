"""GPU parity of the FP8 (e4m3) forward: fa_quantize_fp8 and fa_forward_fp8
through the C ABI against the oracle's FP8 definitions.

* Codes and scales are integer/byte work decided by exactly rounded fp32
  steps, so they must equal the oracle's bit for bit.
* The attention over the dequantized inputs differs from the oracle's fp64
  definition only by the kernel rounding P to e4m3 for the P V product (plus
  fp32 accumulation and the bf16 output).  Per element that error is at most
      (2^-4 sum_j P_ij |Vh_jc| + 2^-10 sum_{j: P_ij < 2^-6} |Vh_jc|) / l_i
  (round to nearest in e4m3: relative 2^-4 for normal values, absolute 2^-10
  below the smallest normal 2^-6; P taken against the true row maximum, which
  bounds the kernel's P against a running maximum from above), plus 2^-8 |O|
  for the bf16 output and 1e-4 for the fp32 arithmetic.  LSE does not involve
  the rounded P: max-abs 1e-3.
* End to end on inputs with outlier channels, the FP8 path must beat the
  per-tensor FP8 baseline against exact attention (the pages report 2.6x lower
  error; the test asks for 2x).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8_baseline
from exact_io_aware_flash_gb300 import check_errors, forward_fp8, quantize_fp8
from exact_io_aware_flash_gb300.synth import Shape, make_inputs

pytestmark = pytest.mark.gpu

TOL_LSE = 1e-3


def signs_for(seed, d=128):
    return torch.from_numpy(np.random.default_rng(seed).choice([-1, 1], d).astype(np.int8))


def gpu_quantize(inp, signs):
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    out = quantize_fp8(q, k, v, None if signs is None else signs.cuda())
    check_errors()
    return out


def oracle_quantize(inp, signs):
    sg = None if signs is None else signs.numpy()
    qc, qs = oracle.fp8_quantize_qk(inp["q"], sg)
    kc, ks = oracle.fp8_quantize_qk(inp["k"], sg)
    vc, vs = oracle.fp8_quantize_v(inp["v"])
    return qc, qs, kc, ks, vc, vs


SHAPES = [
    # B, Hq, Hkv, N
    (1, 1, 1, 1), (1, 2, 1, 7), (2, 2, 2, 127), (1, 4, 2, 128), (1, 2, 2, 129), (1, 3, 1, 300),
    (2, 4, 2, 640),
]


@pytest.mark.parametrize("rotate", [True, False])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("B,Hq,Hkv,N", SHAPES)
def test_quantize_matches_oracle_bitwise(B, Hq, Hkv, N, dtype, rotate):
    inp = make_inputs(Shape(B, Hq, Hkv, N, 128), dtype, seed=300 + N, with_dO=False, q_scale=3.0)
    signs = signs_for(N) if rotate else None
    g = gpu_quantize(inp, signs)
    qc, qs, kc, ks, vc, vs = oracle_quantize(inp, signs)
    assert np.array_equal(g["q8"].cpu().numpy(), qc)
    assert np.array_equal(g["k8"].cpu().numpy(), kc)
    assert np.array_equal(g["q_scale"].cpu().numpy(), qs)
    assert np.array_equal(g["k_scale"].cpu().numpy(), ks)
    assert np.array_equal(g["v_scale"].cpu().numpy(), vs)
    v8t = g["v8t"].cpu().numpy()
    assert np.array_equal(v8t[..., :N], np.swapaxes(vc, 2, 3))
    assert not v8t[..., N:].any()  # padding keys are zero codes


def p_rounding_bound(qh, kh, vh, causal, scale, o_ref):
    """Per-element bound on the effect of rounding P to e4m3 (see the module docstring)."""
    B, Hq, N, d = qh.shape
    Hkv = kh.shape[1]
    bound = np.empty(qh.shape)
    for b in range(B):
        for h in range(Hq):
            g = h * Hkv // Hq
            s = scale * (qh[b, h] @ kh[b, g].T)
            if causal:
                s = np.where(np.tril(np.ones((N, N), dtype=bool)), s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            l = p.sum(axis=1, keepdims=True)
            av = np.abs(vh[b, g])
            bound[b, h] = (2.0 ** -4 * (p @ av) + 2.0 ** -10 * ((p < 2.0 ** -6) @ av)) / l
    return bound + 2.0 ** -8 * np.abs(o_ref) + 1e-4


def check_attention(o, lse, oq, causal, scale, what, heads=None):
    qc, qs, kc, ks, vc, vs = oq
    qh, kh, vh = oracle.fp8_dequantize(qc, qs, kc, ks, vc, vs)
    o_ref, lse_ref = oracle.forward(qh, kh, vh, causal, scale)
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    err_l = float(np.abs(lse - lse_ref).max())
    assert err_l <= TOL_LSE, f"{what}: LSE max-abs {err_l:.3g}"
    bound = p_rounding_bound(qh, kh, vh, causal, scale, o_ref)
    excess = np.abs(o - o_ref) - bound
    assert (excess <= 0).all(), f"{what}: O exceeds the P-rounding bound by {excess.max():.3g}"
    return float(np.sqrt(np.mean((o - o_ref) ** 2)))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,N", SHAPES)
def test_fp8_forward_small_shapes(B, Hq, Hkv, N, causal):
    inp = make_inputs(Shape(B, Hq, Hkv, N, 128), "bf16", seed=400 + N, with_dO=False)
    signs = signs_for(7)
    g = gpu_quantize(inp, signs)
    scale = 1.0 / math.sqrt(128)
    o, lse = forward_fp8(g, causal=causal, scale=scale)
    check_errors()
    check_attention(o, lse, oracle_quantize(inp, signs), causal, scale, f"N={N} causal={causal}")


@pytest.mark.parametrize("q_scale,scale", [(6.0, None), (1.0, 0.0), (1.0, -0.2)])
def test_fp8_forward_score_ranges(q_scale, scale):
    """Peaked scores (the running maximum moves and P spans its whole range),
    uniform and reversed scores."""
    inp = make_inputs(Shape(1, 2, 1, 700, 128), "bf16", seed=41, with_dO=False, q_scale=q_scale)
    s = 1.0 / math.sqrt(128) if scale is None else scale
    signs = signs_for(41)
    g = gpu_quantize(inp, signs)
    for causal in (False, True):
        o, lse = forward_fp8(g, causal=causal, scale=s)
        check_errors()
        check_attention(o, lse, oracle_quantize(inp, signs), causal, s, f"q x{q_scale} scale={scale}")


def test_fp8_beats_per_tensor_baseline_end_to_end():
    """Inputs with outlier channels in Q and K (x20): against exact attention on
    the 16-bit inputs, the rotated, block-scaled FP8 path has a clearly smaller
    error than per-tensor FP8."""
    g = torch.Generator().manual_seed(11)
    q, k, v = (torch.randn(1, 2, 512, 128, generator=g) for _ in range(3))
    for c in (3, 77):
        q[..., c] *= 20.0
        k[..., c] *= 20.0
    q, k, v = q.bfloat16(), k.bfloat16(), v.bfloat16()
    scale = 1.0 / math.sqrt(128) / 10.0
    signs = signs_for(11)
    fp8 = quantize_fp8(q.cuda(), k.cuda(), v.cuda(), signs.cuda())
    o, _ = forward_fp8(fp8, causal=True, scale=scale)
    check_errors()
    o_exact, _ = oracle.forward(q, k, v, True, scale)
    o_base = fp8_baseline.forward(q, k, v, True, scale)
    rmse = lambda a: float(np.sqrt(np.mean((a - o_exact) ** 2)))
    e_gpu, e_base = rmse(o.float().cpu().numpy()), rmse(o_base)
    assert e_base > 2.0 * e_gpu, (e_base, e_gpu)


def test_fp8_forward_is_deterministic():
    inp = make_inputs(Shape(1, 4, 2, 1500, 128), "bf16", seed=6, with_dO=False)
    g = gpu_quantize(inp, signs_for(6))
    a = forward_fp8(g, causal=True)
    b = forward_fp8(g, causal=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("shape,heads", [
    (Shape(4, 16, 16, 4096, 128), [(0, 0), (1, 7), (2, 12), (3, 15)]),
    (Shape(2, 32, 8, 8192, 128), [(0, 0), (1, 31)]),
])
def test_fp8_forward_at_size(shape, heads):
    """The two large forward workloads' shapes (causal, bf16 inputs): the GPU
    quantizes and attends the whole problem; codes are compared bit for bit on
    every head, attention on sampled heads (for GQA the oracle takes the query
    head's KV head)."""
    inp = make_inputs(shape, "bf16", seed=500 + shape.N, with_dO=False)
    signs = signs_for(500)
    g = gpu_quantize(inp, signs)
    scale = 1.0 / math.sqrt(128)
    o, lse = forward_fp8(g, causal=True, scale=scale)
    check_errors()
    qc, qs, kc, ks, vc, vs = oracle_quantize(inp, signs)
    assert np.array_equal(g["q8"].cpu().numpy(), qc) and np.array_equal(g["k8"].cpu().numpy(), kc)
    assert np.array_equal(g["v8t"].cpu().numpy()[..., :shape.N], np.swapaxes(vc, 2, 3))
    grp = shape.Hq // shape.Hkv
    for b, h in heads:
        hk = h // grp
        oq = (qc[b:b + 1, h:h + 1], qs[b:b + 1, h:h + 1], kc[b:b + 1, hk:hk + 1],
              ks[b:b + 1, hk:hk + 1], vc[b:b + 1, hk:hk + 1], vs[b:b + 1, hk:hk + 1])
        check_attention(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], oq, True, scale, f"head ({b},{h})")
