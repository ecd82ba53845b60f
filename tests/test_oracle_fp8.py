"""Pins of the oracle's FP8 (e4m3) input definitions (CPU).

The e4m3 codec is checked against the format's defining values and against
PyTorch's float8_e4m3fn conversion (a library routine); the rotation and the
block quantization against a brute-force recomputation with the explicit
Sylvester Hadamard matrix; the method's claim (block scaling plus the random
Hadamard rotation beats a per-tensor FP8 baseline on inputs with outlier
channels) against the oracle's own exact attention; and planted mistakes in
copies of oracle.c must each fail one of these checks.
"""
import math
import os
import tempfile

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8_baseline

F8 = torch.float8_e4m3fn


def torch_encode(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(F8).view(torch.uint8).numpy()


def hadamard(d: int) -> np.ndarray:
    h = np.array([[1.0]])
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


# ------------------------------------------------------------------ e4m3 codec
def test_e4m3_decode_defining_values():
    dec = oracle.e4m3_decode(np.array([0x7E, 0x01, 0x07, 0x08, 0x38, 0x3F, 0x40, 0x80, 0xFE]))
    assert list(dec[:7]) == [448.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.875, 2.0]
    assert dec[7] == 0.0 and math.copysign(1.0, dec[7]) < 0
    assert dec[8] == -448.0
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF]))).all()


def test_e4m3_decode_matches_library():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(F8).double().numpy()
    got = oracle.e4m3_decode(codes)
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), ~finite)
    assert np.array_equal(got[finite], ref[finite])
    pos = got[:0x7F]
    assert (np.diff(pos) > 0).all()  # codes 0x00..0x7E increase with the code


def test_e4m3_encode_matches_library():
    rng = np.random.default_rng(0)
    mags = np.exp2(rng.uniform(-13, math.log2(463.9), 200000)).astype(np.float32)
    x = mags * rng.choice([-1.0, 1.0], mags.shape).astype(np.float32)
    # every code, every midpoint between neighbours (ties), and zeros
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, vals.astype(np.float32), mids, -mids, [0.0, -0.0]]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), torch_encode(x))


def test_e4m3_encode_ties_and_saturation():
    x = np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 448.0, 464.0, 1e9, -1e9, -0.0, 0.0],
                 dtype=np.float32)
    # 1 + 1/16 lies halfway between 1 (mantissa 000) and 1.125 (001): even -> 1;
    # 1 + 3/16 halfway between 1.125 (001) and 1.25 (010): even -> 1.25;
    # 2^-10 halfway between 0 and the smallest subnormal 2^-9: even -> 0;
    # 3 * 2^-10 halfway between 2^-9 (001) and 2^-8 (010): even -> 2^-8;
    # beyond 448 the value saturates (there is no larger finite code).
    want = [0x38, 0x3A, 0x00, 0x02, 0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x00]
    assert list(oracle.e4m3_encode(x)) == want


def test_e4m3_round_trip():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes).astype(np.float32)), codes)


# ------------------------------------------------------------------ quantization
def brute_force_qk(x, signs):
    """Per head and 128-row block: y = (x * s) H (fp64, exact for the small
    integer inputs used here), amax, f = fl32(448 / amax), codes = e4m3(fl32(y * f))."""
    B, H, N, d = x.shape
    Hd = hadamard(d)
    T = (N + 127) // 128
    codes = np.empty(x.shape, np.uint8)
    scales = np.empty((B, H, T), np.float32)
    cfac = np.float32(1.0 / (448.0 * math.sqrt(d))) if signs is not None else np.float32(1.0 / 448.0)
    for b in range(B):
        for h in range(H):
            xs = x[b, h].astype(np.float64) * (1.0 if signs is None else signs[None, :])
            y = xs @ Hd if signs is not None else xs
            for t in range(T):
                blk = y[t * 128:(t + 1) * 128].astype(np.float32)
                amax = np.float32(np.abs(blk).max())
                f = np.float32(448.0) / amax if amax > 0 else np.float32(0.0)
                codes[b, h, t * 128:(t + 1) * 128] = torch_encode(blk * f)
                scales[b, h, t] = amax * cfac
    return codes, scales


@pytest.mark.parametrize("rotate", [True, False])
def test_quantize_qk_brute_force(rotate):
    rng = np.random.default_rng(1)
    B, H, N, d = 2, 3, 300, 128  # three blocks per head, the last one ragged
    x = rng.integers(-8, 9, (B, H, N, d)).astype(np.float32)  # rotated sums stay exact in fp32
    x[0, 1, 130:140, 5] = 40.0  # an outlier channel in one block
    signs = rng.choice([-1, 1], d).astype(np.int8) if rotate else None
    codes, scales = oracle.fp8_quantize_qk(x, signs)
    want_c, want_s = brute_force_qk(x, None if signs is None else signs.astype(np.float64))
    assert np.array_equal(codes, want_c)
    assert np.array_equal(scales, want_s)


def test_quantize_qk_zero_block():
    x = np.zeros((1, 1, 200, 64), np.float32)
    x[0, 0, 150] = 1.0
    codes, scales = oracle.fp8_quantize_qk(x, np.ones(64, np.int8))
    assert scales[0, 0, 0] == 0 and (codes[0, 0, :128] == 0).all()
    assert scales[0, 0, 1] > 0


def test_quantize_v_brute_force():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal((2, 2, 257, 64)) * rng.uniform(0.1, 20, 64)).astype(np.float32)
    v = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    codes, scales = oracle.fp8_quantize_v(v)
    amax = np.abs(v).max(axis=2)  # [B, H, d]
    f = np.float32(448.0) / amax.astype(np.float32)
    assert np.array_equal(codes, torch_encode(v * f[:, :, None, :]))
    assert np.array_equal(scales, amax.astype(np.float32) * np.float32(1.0 / 448.0))
    # the largest magnitude of each channel maps to the largest code
    assert ((codes & 0x7F).max(axis=2) == 0x7E).all()


def test_dequantized_rotation_is_orthogonal():
    """The dequantized rotated rows approximate (x * s) H / sqrt(d), an orthogonal
    map: dot products and norms of the original rows are kept to FP8 accuracy."""
    rng = np.random.default_rng(3)
    q = torch.randn(1, 2, 256, 128, generator=torch.Generator().manual_seed(3)).bfloat16()
    k = torch.randn(1, 2, 256, 128, generator=torch.Generator().manual_seed(4)).bfloat16()
    v = torch.randn(1, 2, 256, 128, generator=torch.Generator().manual_seed(5)).bfloat16()
    signs = rng.choice([-1, 1], 128).astype(np.int8)
    qc, qs = oracle.fp8_quantize_qk(q, signs)
    kc, ks = oracle.fp8_quantize_qk(k, signs)
    vc, vs = oracle.fp8_quantize_v(v)
    qh, kh, vh = oracle.fp8_dequantize(qc, qs, kc, ks, vc, vs)
    exact = q.double().numpy() @ np.swapaxes(k.double().numpy(), 2, 3)
    approx = qh @ np.swapaxes(kh, 2, 3)
    assert np.abs(approx - exact).max() / np.abs(exact).max() < 0.05
    rel = np.linalg.norm(qh, axis=3) / np.linalg.norm(q.double().numpy(), axis=3)
    assert np.abs(rel - 1).max() < 0.05


def outlier_inputs(seed, N=512, d=128, heads=2, outliers=(3, 77), factor=20.0):
    """N(0,1) Q, K, V in bf16 with a few channels of Q and K scaled up (the
    outlier features incoherent processing is meant to spread)."""
    g = torch.Generator().manual_seed(seed)
    q, k, v = (torch.randn(1, heads, N, d, generator=g) for _ in range(3))
    for c in outliers:
        q[..., c] *= factor
        k[..., c] *= factor
    return q.bfloat16(), k.bfloat16(), v.bfloat16()


def test_block_scaling_and_rotation_beat_per_tensor_baseline():
    """The method's FP8 error claim on the oracle side: with outlier channels,
    block scaling + random Hadamard rotation gives a clearly smaller O error
    against exact attention than one scale per tensor (the pages report 2.6x)."""
    q, k, v = outlier_inputs(11)
    scale = 1.0 / math.sqrt(128) / 10.0  # keep the outlier-dominated scores in a softmax-friendly range
    signs = np.random.default_rng(11).choice([-1, 1], 128).astype(np.int8)
    o_exact, _ = oracle.forward(q, k, v, True, scale)
    qc, qs = oracle.fp8_quantize_qk(q, signs)
    kc, ks = oracle.fp8_quantize_qk(k, signs)
    vc, vs = oracle.fp8_quantize_v(v)
    o_fp8, _ = oracle.forward_fp8(qc, qs, kc, ks, vc, vs, True, scale)
    o_base = fp8_baseline.forward(q, k, v, True, scale)
    rmse = lambda a: float(np.sqrt(np.mean((a - o_exact) ** 2)))
    assert rmse(o_base) > 2.0 * rmse(o_fp8), (rmse(o_base), rmse(o_fp8))


# ------------------------------------------------------------------ planted mistakes
FP8_MUTATIONS = [
    ("ties_to_odd", "else c = (lo & 1) ? lo + 1 : lo;", "else c = (lo & 1) ? lo : lo + 1;"),
    ("exponent_bias_8", "ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    ("fwht_sign", "x[i + h] = a - b;", "x[i + h] = b - a;"),
    ("signed_amax", "if (fabsf(yr[c]) > amax) amax = fabsf(yr[c]);", "if (yr[c] > amax) amax = yr[c];"),
    ("signs_ignored", "yr[c] = (signs && signs[c] < 0) ? -xr[c] : xr[c];", "yr[c] = xr[c];"),
    ("v_scale_without_fl32_448", "scales[(size_t)h * d + c] = amax * cfac;",
     "scales[(size_t)h * d + c] = amax / 448.5f;"),
    ("block_of_64_rows", "const int r0 = t * 128, r1 = (r0 + 128 < N) ? r0 + 128 : N;",
     "const int r0 = t * 128, r1 = (r0 + 64 < N) ? r0 + 64 : N;"),
]


def _fp8_pins_fail(o) -> bool:
    rng = np.random.default_rng(5)
    x = np.concatenate([np.exp2(rng.uniform(-12, 8.5, 5000)), [1.0625, 1.1875, 3 * 2.0 ** -10]])
    x = (x * rng.choice([-1, 1], x.shape)).astype(np.float32)
    if not np.array_equal(o.e4m3_encode(x), torch_encode(x)):
        return True
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(F8).double().numpy()
    got = o.e4m3_decode(codes)
    if not np.array_equal(got[~np.isnan(ref)], ref[~np.isnan(ref)]):
        return True
    xi = rng.integers(-8, 9, (1, 2, 300, 128)).astype(np.float32)
    signs = rng.choice([-1, 1], 128).astype(np.int8)
    c, s = o.fp8_quantize_qk(xi, signs)
    wc, ws = brute_force_qk(xi, signs.astype(np.float64))
    if not (np.array_equal(c, wc) and np.array_equal(s, ws)):
        return True
    v = (rng.standard_normal((1, 1, 130, 64)) * 3).astype(np.float32)
    vc, vs = o.fp8_quantize_v(v)
    amax = np.abs(v).max(axis=2).astype(np.float32)
    if not (np.array_equal(vc, torch_encode(v * (np.float32(448.0) / amax)[:, :, None, :]))
            and np.array_equal(vs, amax * np.float32(1.0 / 448.0))):
        return True
    return False


def test_unmutated_fp8_oracle_passes():
    assert not _fp8_pins_fail(oracle._default())


@pytest.mark.parametrize("name,old,new", FP8_MUTATIONS, ids=[m[0] for m in FP8_MUTATIONS])
def test_fp8_pins_catch_planted_mistake(name, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(old) == 1, name
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "mut.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.build(force=True, src=path, out=os.path.join(tmp, "libmut.so"))
        assert _fp8_pins_fail(oracle.Oracle(lib)), f"planted mistake {name} not caught"
