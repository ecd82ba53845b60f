"""Plant plausible mistakes in copies of the oracle and check the pins catch each one.

Every mutation is applied to the C source text, compiled into a throw-away
library on the CPU, and run through three independent checks: the materialising
numpy schedule, finite differences of the forward, and the closed form for
identical keys.  A mutation that none of them flags would mean the pins have a
blind spot.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import naive

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, exact text in oracle.c, replacement)
MUTATIONS = [
    ("drop_D_term", "(dot(doi, vh + (size_t)kk * d, d) - Di);", "(dot(doi, vh + (size_t)kk * d, d));"),
    ("drop_dq_scale", "dqi[c] *= scale;\n                /* dK_k", "dqi[c] *= 1.0;\n                /* dK_k"),
    ("window_backward_drops_D", "(dot(doi, vh + (size_t)(k0 + t) * d, d) - Di);",
     "(dot(doi, vh + (size_t)(k0 + t) * d, d));"),
    ("dk_without_scale", "const double a = scale * ds[kk];", "const double a = ds[kk];"),
    ("dv_uses_q", "dvk[c] += w * doi[c];", "dvk[c] += w * qi[c];"),
    ("causal_off_by_one", "const int nk = causal ? i + 1 : N;\n            lse",
     "const int nk = causal ? i : N;\n            lse"),
    ("lse_without_max", "return m + log(l);", "return log(l);"),
    ("no_max_shift", "p[k] = exp(p[k] - m);", "p[k] = exp(p[k]);"),
    ("gqa_modulo_map",
     "const int g = (int)(((int64_t)h * Hkv) / Hq);\n            const double* qi = q + (size_t)r * d;\n"
     "            const double* kh = k + ((size_t)b * Hkv + g) * (size_t)N * d;",
     "const int g = (int)(h % Hkv);\n            const double* qi = q + (size_t)r * d;\n"
     "            const double* kh = k + ((size_t)b * Hkv + g) * (size_t)N * d;"),
    ("window_off_by_one",
     "const int k0 = i - window + 1 > 0 ? i - window + 1 : 0;\n            lse[r]",
     "const int k0 = i - window > 0 ? i - window : 0;\n            lse[r]"),
    ("rect_drops_last_key", "lse[r] = softmax_row(qi, kh, Nk, d, scale, p);",
     "lse[r] = softmax_row(qi, kh, Nk - 1, d, scale, p);"),
    ("unnormalised_p", "for (int k = 0; k < nk; ++k) p[k] /= l;", ""),
    ("transposed_dq_operand", "dqi[c] += ds[kk] * kh[(size_t)kk * d + c];",
     "dqi[c] += ds[kk] * vh[(size_t)kk * d + c];"),
]


def _checks_fail(o: "oracle.Oracle") -> bool:
    rng = np.random.default_rng(99)
    B, Hq, Hkv, N, d, s = 1, 4, 2, 6, 3, 0.8
    q, k, v, dO = (rng.standard_normal(x) for x in
                   ((B, Hq, N, d), (B, Hkv, N, d), (B, Hkv, N, d), (B, Hq, N, d)))
    # Large-magnitude queries make a missing max-shift overflow.
    q_big = 300.0 * q
    for causal in (False, True):
        for qq in (q, q_big):
            try:
                got_o, got_lse = o.forward(qq, k, v, causal, s)
            except ValueError:
                return True
            ref_o, ref_lse, _ = naive.forward(qq, k, v, causal, s)
            if not (np.allclose(got_o, ref_o, atol=1e-9) and np.allclose(got_lse, ref_lse, atol=1e-9)):
                return True
        dq, dk, dv, _ = o.backward(q, k, v, dO, causal, s)
        h = 1e-6
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            idx = tuple(int(rng.integers(0, n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = dict(q=q, k=k, v=v)
            args[name] = xp
            lp = float((oracle.forward(args["q"], args["k"], args["v"], causal, s)[0] * dO).sum())
            args[name] = xm
            lm = float((oracle.forward(args["q"], args["k"], args["v"], causal, s)[0] * dO).sum())
            if abs((lp - lm) / (2 * h) - g[idx]) > 1e-5 * max(1.0, abs(g[idx])):
                return True
        ref = naive.backward(q, k, v, dO, causal, s)
        for a, b in zip((dq, dk, dv), ref[:3]):
            if not np.allclose(a, b, atol=1e-9):
                return True
    # sliding window of 3 over 6 positions
    qw, kw, vw = rng.standard_normal((B, Hq, 6, d)), rng.standard_normal((B, Hkv, 6, d)), \
        rng.standard_normal((B, Hkv, 6, d))
    o_w, l_w = o.forward_window(qw, kw, vw, 3, s)
    o_n, l_n, _ = naive.forward(qw, kw, vw, True, s, window=3)
    if not (np.allclose(o_w, o_n, atol=1e-9) and np.allclose(l_w, l_n, atol=1e-9)):
        return True
    dOw = rng.standard_normal((B, Hq, 6, d))
    gw = o.backward_window(qw, kw, vw, dOw, 3, s)
    gn = naive.backward(qw, kw, vw, dOw, True, s, window=3)
    for a, b in zip(gw, gn[:3]):
        if not np.allclose(a, b, atol=1e-9):
            return True
    # rectangular (decoding) forward: 3 query rows against 9 keys
    qr, kr, vr = rng.standard_normal((B, Hq, 3, d)), rng.standard_normal((B, Hkv, 9, d)), \
        rng.standard_normal((B, Hkv, 9, d))
    o_r, l_r = o.forward_rect(qr, kr, vr, s)
    o_n, l_n, _ = naive.forward(qr, kr, vr, False, s)
    if not (np.allclose(o_r, o_n, atol=1e-9) and np.allclose(l_r, l_n, atol=1e-9)):
        return True
    return False


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not unique in oracle.c"
    src = tmp_path / f"oracle_{name}.c"
    src.write_text(text.replace(old, new))
    lib = oracle.build(force=True, src=str(src), out=str(tmp_path / f"lib_{name}.so"))
    assert _checks_fail(oracle.Oracle(lib)), f"pins did not catch mutation {name}"


def test_unmutated_oracle_passes_the_same_checks(tmp_path):
    lib = oracle.build(force=True, src=SRC, out=str(tmp_path / "lib_clean.so"))
    assert not _checks_fail(oracle.Oracle(lib))


def _key_shift_invariance_fails(o: "oracle.Oracle") -> bool:
    """The key-shift pin alone: shifting every key by one vector must leave dQ
    unchanged (rows of dS sum to zero), for causal, non-causal and windowed
    attention."""
    rng = np.random.default_rng(7)
    B, Hq, Hkv, N, d, s = 1, 2, 1, 7, 4, 0.9
    q, k, v, dO = (rng.standard_normal(x) for x in
                   ((B, Hq, N, d), (B, Hkv, N, d), (B, Hkv, N, d), (B, Hq, N, d)))
    c = rng.standard_normal((B, Hkv, 1, d))
    for causal in (False, True):
        dq, _, _, _ = o.backward(q, k, v, dO, causal, s)
        dq2, _, _, _ = o.backward(q, k + c, v, dO, causal, s)
        if not np.allclose(dq, dq2, atol=1e-10):
            return True
    dq, _, _ = o.backward_window(q, k, v, dO, 3, s)
    dq2, _, _ = o.backward_window(q, k + c, v, dO, 3, s)
    return not np.allclose(dq, dq2, atol=1e-10)


@pytest.mark.parametrize("name", ["drop_D_term", "window_backward_drops_D"])
def test_key_shift_pin_catches_a_dropped_D(tmp_path, name):
    old, new = next((m[1], m[2]) for m in MUTATIONS if m[0] == name)
    text = open(SRC).read()
    src = tmp_path / f"oracle_{name}.c"
    src.write_text(text.replace(old, new))
    lib = oracle.build(force=True, src=str(src), out=str(tmp_path / f"lib_{name}.so"))
    assert _key_shift_invariance_fails(oracle.Oracle(lib))
    clean = oracle.build(force=True, src=SRC, out=str(tmp_path / "lib_clean.so"))
    assert not _key_shift_invariance_fails(oracle.Oracle(clean))
