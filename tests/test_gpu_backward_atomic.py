"""GPU parity of the one-pass backward (fa_backward_atomic, dQ summed across key
tiles with float32 atomic adds) through the C ABI against the fp64 oracle.

Tolerance (per gradient): relative Frobenius error <= 1e-2, as for the
deterministic backward.  dK and dV are summed in a fixed order (bitwise
reproducible); dQ's summation order varies between runs, so two runs of dQ
agree only to float32 rounding of the partial sums.  The cases add to the
deterministic backward's: keys past N without a causal mask (their recomputed
probabilities must not reach dQ), peaked scores on a ragged length, a
workspace and outputs filled with NaN before the call (the accumulator is
zeroed by the call, every output element written), sliding windows, and the
full-size sweep and grouped-query shapes.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_flash_gb300 import backward, check_errors, forward, workspace_size
from exact_io_aware_flash_gb300.synth import (BACKWARD_SWEEP_N, Shape, backward_sweep_shape,
                                              make_inputs)

pytestmark = pytest.mark.gpu

TOL_REL = 1e-2


def rel_fro(g, ref):
    """Relative Frobenius error; against the inputs' unit scale where the exact
    gradient vanishes (one visible key: P = [1], so dS = 0 and dQ = dK = 0)."""
    g = g.float().cpu().numpy() if isinstance(g, torch.Tensor) else g
    ref_norm = float(np.linalg.norm(ref))
    if ref_norm < 1e-9:
        return float(np.abs(g).max()) / 0.1
    return float(np.linalg.norm(g - ref) / ref_norm)


def gpu_fwd_bwd(inp, causal, scale, window=None, workspace=None, grads=None):
    q, k, v, dO = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    o, lse = forward(q, k, v, causal=causal, scale=scale, window=window)
    dq, dk, dv = (None, None, None) if grads is None else grads
    dq, dk, dv = backward(q, k, v, o, lse, dO, causal=causal, scale=scale, window=window,
                          workspace=workspace, dq=dq, dk=dk, dv=dv, deterministic=False)
    check_errors()
    return o, lse, dq, dk, dv


def check(grads, refs, what):
    for name, g, r in zip(("dq", "dk", "dv"), grads, refs):
        assert np.isfinite(g.float().cpu().numpy()).all(), f"{what} {name}: non-finite"
        e = rel_fro(g, r)
        assert e <= TOL_REL, f"{what}: {name} rel err {e:.3g}"


SMALL = [
    # B, Hq, Hkv, N, d
    (1, 1, 1, 1, 64), (1, 1, 1, 7, 128), (1, 2, 2, 64, 64), (2, 1, 1, 127, 128),
    (1, 2, 1, 128, 64), (1, 1, 1, 129, 128), (2, 2, 2, 255, 64), (1, 4, 2, 256, 128),
    (1, 3, 1, 300, 64), (1, 2, 2, 513, 128), (2, 4, 1, 640, 128),
]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,N,d", SMALL)
def test_atomic_backward_small_shapes(B, Hq, Hkv, N, d, causal, dtype):
    shape = Shape(B, Hq, Hkv, N, d)
    inp = make_inputs(shape, dtype, seed=11 + N + d)
    scale = 1.0 / math.sqrt(d)
    ws = torch.empty(workspace_size(B, Hq, N, d, deterministic=False), dtype=torch.uint8,
                     device="cuda")
    _, _, dq, dk, dv = gpu_fwd_bwd(inp, causal, scale, workspace=ws)
    dq_r, dk_r, dv_r, D_r = oracle.backward(inp["q"], inp["k"], inp["v"], inp["dO"], causal, scale)
    check((dq, dk, dv), (dq_r, dk_r, dv_r), f"{shape} causal={causal} {dtype}")
    # D = rowsum(dO o O) at the start of the workspace (layout documented in fa.h)
    D_gpu = ws[: 4 * B * Hq * N].view(torch.float32).view(B, Hq, N).cpu().numpy()
    assert rel_fro(D_gpu, D_r) <= TOL_REL


@pytest.mark.parametrize("q_scale", [4.0, 0.0, 30.0])
def test_atomic_backward_score_ranges(q_scale):
    """Peaked (Q x 4, Q x 30) and uniform (Q = 0) attention on a ragged length:
    without a causal mask the padding keys of the last tile meet every query,
    and with Q x 30 a row's LSE can lie far below 0, so exp(0 - LSE) of a
    padding key would overflow if it were not masked."""
    shape = Shape(1, 2, 1, 300, 64)
    inp = make_inputs(shape, "fp16", seed=21, q_scale=q_scale)
    scale = 1.0 / math.sqrt(64)
    for causal in (False, True):
        _, _, dq, dk, dv = gpu_fwd_bwd(inp, causal, scale)
        refs = oracle.backward(inp["q"], inp["k"], inp["v"], inp["dO"], causal, scale)[:3]
        check((dq, dk, dv), refs, f"q_scale={q_scale} causal={causal}")


@pytest.mark.parametrize("scale", [0.0, -0.3])
def test_atomic_backward_degenerate_scales(scale):
    """scale = 0 (uniform attention: dQ = dK = 0 exactly) and a negative scale."""
    shape = Shape(1, 2, 2, 200, 128)
    inp = make_inputs(shape, "bf16", seed=22)
    for causal in (False, True):
        _, _, dq, dk, dv = gpu_fwd_bwd(inp, causal, scale)
        refs = oracle.backward(inp["q"], inp["k"], inp["v"], inp["dO"], causal, scale)[:3]
        check((dq, dk, dv), refs, f"scale={scale} causal={causal}")


def test_atomic_backward_needs_no_zeroed_memory():
    """Workspace and outputs full of NaN before the call: the call zeroes its own
    accumulator and writes every output element."""
    shape = Shape(2, 4, 2, 333, 128)
    inp = make_inputs(shape, "bf16", seed=23)
    scale = 1.0 / math.sqrt(128)
    ws = torch.full((workspace_size(2, 4, 333, 128, deterministic=False) // 4,), float("nan"),
                    dtype=torch.float32, device="cuda").view(torch.uint8)
    grads = tuple(torch.full_like(inp[n].cuda(), float("nan")) for n in ("q", "k", "k"))
    _, _, dq, dk, dv = gpu_fwd_bwd(inp, True, scale, workspace=ws, grads=grads)
    refs = oracle.backward(inp["q"], inp["k"], inp["v"], inp["dO"], True, scale)[:3]
    check((dq, dk, dv), refs, "NaN-filled workspace and outputs")


def test_atomic_backward_matches_deterministic():
    """Both backward algorithms compute the same gradients: dK and dV within
    float32 rounding of each other, dQ within its accumulation-order rounding;
    dK and dV of two one-pass runs agree bitwise."""
    shape = Shape(1, 4, 1, 1000, 128)
    inp = make_inputs(shape, "bf16", seed=8)
    scale = 1.0 / math.sqrt(128)
    q, k, v, dO = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    o, lse = forward(q, k, v, causal=True, scale=scale)
    det = backward(q, k, v, o, lse, dO, causal=True, scale=scale)
    a1 = backward(q, k, v, o, lse, dO, causal=True, scale=scale, deterministic=False)
    a2 = backward(q, k, v, o, lse, dO, causal=True, scale=scale, deterministic=False)
    check_errors()
    assert torch.equal(a1[1], a2[1]) and torch.equal(a1[2], a2[2])
    for name, x, y in zip(("dq", "dk", "dv"), a1, det):
        ref = y.float().cpu().numpy()
        e = rel_fro(x, ref)
        assert e <= 4e-3, f"{name}: one-pass vs two-pass rel err {e:.3g}"
    e = rel_fro(a1[0], a2[0].float().cpu().numpy())
    assert e <= 1e-3, f"dq run to run: {e:.3g}"


WINDOWS = [
    # B, Hq, Hkv, N, d, window
    (1, 1, 1, 7, 128, 3), (1, 2, 2, 127, 64, 1), (2, 1, 1, 129, 64, 128), (1, 4, 2, 256, 64, 129),
    (1, 3, 1, 300, 128, 100), (2, 4, 1, 640, 128, 257), (1, 1, 1, 300, 128, 1000),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,W", WINDOWS)
def test_atomic_backward_window(B, Hq, Hkv, N, d, W):
    shape = Shape(B, Hq, Hkv, N, d)
    inp = make_inputs(shape, "bf16", seed=31 + N + W)
    scale = 1.0 / math.sqrt(d)
    _, _, dq, dk, dv = gpu_fwd_bwd(inp, True, scale, window=W)
    refs = oracle.backward_window(inp["q"], inp["k"], inp["v"], inp["dO"], W, scale)
    check((dq, dk, dv), refs, f"{shape} W={W}")


def spread_heads(B, H, count=8):
    """`count` (b, h) pairs evenly spaced over the linear head index, first and
    last included, so every part of the launch order is touched."""
    n = B * H
    idx = sorted({round(i * (n - 1) / (count - 1)) for i in range(count)}) if n > 1 else [0]
    return [(x // H, x % H) for x in idx]


@pytest.mark.parametrize("N", BACKWARD_SWEEP_N)
def test_atomic_backward_sweep_workload(N):
    """H=16, d=128, bf16, causal, B*N = 32768 at full size; oracle on 8 heads."""
    shape = backward_sweep_shape(N)
    inp = make_inputs(shape, "bf16", seed=1005 + N)
    scale = 1.0 / math.sqrt(128)
    _, _, dq, dk, dv = gpu_fwd_bwd(inp, True, scale)
    for b, h in spread_heads(shape.B, shape.Hq):
        sl = lambda t: t[b:b + 1, h:h + 1]
        refs = oracle.backward(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["dO"]), True,
                               scale)[:3]
        check((sl(dq), sl(dk), sl(dv)), refs, f"N={N} head ({b},{h})")


@pytest.mark.parametrize("causal", [True, False])
def test_atomic_backward_gqa_at_size(causal):
    """B=1, Hq=32, Hkv=8 (groups of 4), N=4096, d=128, bf16: dK, dV summed over
    each KV head's query group, dQ summed over key tiles by many CTAs."""
    shape = Shape(1, 32, 8, 4096, 128)
    inp = make_inputs(shape, "bf16", seed=2718)
    scale = 1.0 / math.sqrt(128)
    _, _, dq, dk, dv = gpu_fwd_bwd(inp, causal, scale)
    g = shape.group
    for b, hk in ((0, 0), (0, 7)):
        qs = lambda t: t[b:b + 1, hk * g:(hk + 1) * g]
        ks = lambda t: t[b:b + 1, hk:hk + 1]
        refs = oracle.backward(qs(inp["q"]), ks(inp["k"]), ks(inp["v"]), qs(inp["dO"]), causal,
                               scale)[:3]
        check((qs(dq), ks(dk), ks(dv)), refs, f"GQA causal={causal} KV head ({b},{hk})")


def test_atomic_backward_rejects_bad_window():
    shape = Shape(1, 1, 1, 64, 64)
    inp = make_inputs(shape, "bf16", seed=1)
    q, k, v, dO = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    o, lse = forward(q, k, v, causal=True)
    with pytest.raises(ValueError):
        backward(q, k, v, o, lse, dO, causal=False, window=16, deterministic=False)
