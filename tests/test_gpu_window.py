"""GPU parity of the sliding-window (local) causal attention: fa_forward_window
and fa_backward_window through the C ABI against the fp64 oracle's window
functions (key k visible to query i iff i - window < k <= i).

Tolerances as for the causal path: O max-abs <= 2e-3 (fp16) / 1e-2 (bf16),
LSE max-abs <= 1e-3, gradients relative Frobenius <= 1e-2.  Windows cover the
degenerate width 1 (each row sees only itself), widths around the 128-key tile
(127, 128, 129), widths that leave some rows of a tile with no visible key in
the first tile they visit, and widths at and beyond N (equal to causal).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_flash_gb300 import backward, check_errors, forward
from exact_io_aware_flash_gb300.synth import Shape, make_inputs

pytestmark = pytest.mark.gpu

TOL_O = {"fp16": 2e-3, "bf16": 1e-2}
TOL_LSE = 1e-3
TOL_REL = 1e-2


def rel_fro(g, ref):
    g = g.float().cpu().numpy() if isinstance(g, torch.Tensor) else g
    ref_norm = float(np.linalg.norm(ref))
    if ref_norm < 1e-9:  # window 1: P = [1] per row, so dS = 0 and dQ = dK = 0 exactly
        return float(np.abs(g).max()) / 0.1
    return float(np.linalg.norm(g - ref) / ref_norm)


def run_gpu(inp, window, scale, with_backward=True):
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = forward(q, k, v, causal=True, scale=scale, window=window)
    grads = None
    if with_backward:
        grads = backward(q, k, v, o, lse, inp["dO"].cuda(), causal=True, scale=scale, window=window)
    check_errors()
    return o, lse, grads


def check_forward(o, lse, o_ref, lse_ref, dtype, what):
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    err_o = float(np.abs(o - o_ref).max())
    err_l = float(np.abs(lse - lse_ref).max())
    assert err_o <= TOL_O[dtype], f"{what}: O max-abs {err_o:.3g}"
    assert err_l <= TOL_LSE, f"{what}: LSE max-abs {err_l:.3g}"


def check_grads(grads, refs, what):
    for name, g, r in zip(("dq", "dk", "dv"), grads, refs):
        e = rel_fro(g, r)
        assert e <= TOL_REL, f"{what} {name}: {e:.3g}"


CASES = [
    # B, Hq, Hkv, N, d, window
    (1, 1, 1, 1, 64, 1), (1, 1, 1, 7, 128, 3), (1, 2, 2, 127, 64, 1), (1, 2, 1, 128, 128, 64),
    (2, 1, 1, 129, 64, 128), (1, 2, 2, 255, 128, 127), (1, 4, 2, 256, 64, 129),
    (1, 3, 1, 300, 128, 100), (1, 2, 2, 513, 64, 200), (2, 4, 1, 640, 128, 257),
    (1, 2, 1, 640, 128, 639), (1, 2, 2, 300, 64, 300), (1, 1, 1, 300, 128, 1000),
]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("B,Hq,Hkv,N,d,W", CASES)
def test_window_small_shapes(B, Hq, Hkv, N, d, W, dtype):
    shape = Shape(B, Hq, Hkv, N, d)
    inp = make_inputs(shape, dtype, seed=31 + N + W)
    scale = 1.0 / math.sqrt(d)
    o, lse, grads = run_gpu(inp, W, scale)
    o_ref, lse_ref = oracle.forward_window(inp["q"], inp["k"], inp["v"], W, scale)
    check_forward(o, lse, o_ref, lse_ref, dtype, f"{shape} W={W}")
    refs = oracle.backward_window(inp["q"], inp["k"], inp["v"], inp["dO"], W, scale)
    check_grads(grads, refs, f"{shape} W={W}")


@pytest.mark.parametrize("q_scale,scale", [(8.0, None), (1.0, 0.0), (1.0, -0.3)])
def test_window_score_ranges(q_scale, scale):
    """Peaked scores (the running maximum moves, and rows whose first tile is
    fully masked start from an empty maximum), uniform and reversed scores."""
    shape = Shape(1, 2, 1, 700, 128)
    inp = make_inputs(shape, "fp16", seed=41, q_scale=q_scale)
    s = 1.0 / math.sqrt(128) if scale is None else scale
    for W in (90, 200):
        o, lse, grads = run_gpu(inp, W, s)
        o_ref, lse_ref = oracle.forward_window(inp["q"], inp["k"], inp["v"], W, s)
        o_np = o.float().cpu().numpy()
        assert np.isfinite(o_np).all()
        # Q x 8 makes the rows nearly one-hot: bound by the rounding of P and O
        # (see the causal forward's score-range test) instead of the flat tolerance.
        u = 2.0 ** -11
        vmax = float(inp["v"].float().abs().max())
        bound = u * (np.abs(o_ref) + vmax) + 1e-4
        assert (np.abs(o_np - o_ref) <= bound).all(), (q_scale, scale, W)
        assert float(np.abs(lse.cpu().numpy() - lse_ref).max()) <= TOL_LSE
        refs = oracle.backward_window(inp["q"], inp["k"], inp["v"], inp["dO"], W, s)
        check_grads(grads, refs, f"q_scale={q_scale} scale={scale} W={W}")


def test_window_at_least_n_equals_causal():
    """A window of N or more keys hides nothing causal masking does not: bitwise
    the causal outputs."""
    shape = Shape(1, 4, 2, 1000, 128)
    inp = make_inputs(shape, "bf16", seed=5)
    scale = 1.0 / math.sqrt(128)
    q, k, v, dO = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    o_c, lse_c = forward(q, k, v, causal=True, scale=scale)
    g_c = backward(q, k, v, o_c, lse_c, dO, causal=True, scale=scale)
    for W in (1000, 5000):
        o_w, lse_w = forward(q, k, v, causal=True, scale=scale, window=W)
        g_w = backward(q, k, v, o_w, lse_w, dO, causal=True, scale=scale, window=W)
        assert torch.equal(o_c, o_w) and torch.equal(lse_c, lse_w)
        for a, b in zip(g_c, g_w):
            assert torch.equal(a, b)
    check_errors()


def test_window_is_deterministic():
    shape = Shape(1, 4, 1, 1500, 128)
    inp = make_inputs(shape, "bf16", seed=6)
    scale = 1.0 / math.sqrt(128)
    a = run_gpu(inp, 300, scale)
    b = run_gpu(inp, 300, scale)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    for x, y in zip(a[2], b[2]):
        assert torch.equal(x, y)


def test_window_rejects_non_causal():
    shape = Shape(1, 1, 1, 64, 64)
    inp = make_inputs(shape, "bf16", seed=1, with_dO=False)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    with pytest.raises(ValueError):
        forward(q, k, v, causal=False, window=16)


@pytest.mark.parametrize("W", [1024, 4000])
def test_window_at_size(W):
    """Long sequences with a local window: B=2, Hq=16, Hkv=4, N=8192, d=128,
    bf16.  The GPU runs the whole problem; the oracle checks 6 heads spread over
    the launch order, forward and backward (dK, dV summed over each KV head's
    query group, so the oracle takes whole groups)."""
    shape = Shape(2, 16, 4, 8192, 128)
    inp = make_inputs(shape, "bf16", seed=8192 + W)
    scale = 1.0 / math.sqrt(128)
    o, lse, (dq, dk, dv) = run_gpu(inp, W, scale)
    g = shape.Hq // shape.Hkv
    for b, hkv in ((0, 0), (0, 3), (1, 1), (1, 3)):
        hs = slice(hkv * g, (hkv + 1) * g)
        sq = lambda t: t[b:b + 1, hs]
        skv = lambda t: t[b:b + 1, hkv:hkv + 1]
        o_ref, lse_ref = oracle.forward_window(sq(inp["q"]), skv(inp["k"]), skv(inp["v"]), W, scale)
        check_forward(sq(o), sq(lse), o_ref, lse_ref, "bf16", f"W={W} b={b} hkv={hkv}")
        refs = oracle.backward_window(sq(inp["q"]), skv(inp["k"]), skv(inp["v"]), sq(inp["dO"]), W,
                                      scale)
        check_grads((sq(dq), skv(dk), skv(dv)), refs, f"W={W} b={b} hkv={hkv}")
