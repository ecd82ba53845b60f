"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these re-types the oracle's own formula: each compares it with an
independent implementation (the materialising numpy schedule, the pages'
online recurrences), a closed form, an invariant, or finite differences of the
forward map.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import naive, online

RNG = np.random.default_rng(1234)


def rand(*shape, rng=RNG):
    return rng.standard_normal(shape)


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("B,Hq,Hkv,N,d", [(1, 1, 1, 1, 1), (1, 1, 1, 5, 4), (2, 2, 2, 7, 8),
                                          (2, 2, 1, 16, 8), (1, 4, 2, 13, 4), (1, 3, 1, 9, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_bruteforce_forward(B, Hq, Hkv, N, d, causal):
    q, k, v = rand(B, Hq, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.forward(q, k, v, causal, scale)
    o_n, lse_n, _ = naive.forward(q, k, v, causal, scale)
    np.testing.assert_allclose(o, o_n, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_n, rtol=0, atol=1e-12)


@pytest.mark.parametrize("B,Hq,Hkv,N,d", [(1, 1, 1, 1, 1), (2, 2, 2, 7, 8), (2, 2, 1, 16, 8),
                                          (1, 4, 2, 13, 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_bruteforce_backward(B, Hq, Hkv, N, d, causal):
    q, k, v, dO = rand(B, Hq, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, Hq, N, d)
    scale = 0.7
    dq, dk, dv, D = oracle.backward(q, k, v, dO, causal, scale)
    dq_n, dk_n, dv_n, rs = naive.backward(q, k, v, dO, causal, scale)
    for a, b in ((dq, dq_n), (dk, dk_n), (dv, dv_n)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    # D = rowsum(dO o O) equals rowsum(P o dP) in exact arithmetic
    np.testing.assert_allclose(D, rs, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- closed forms
def test_softmax_rows_sum_to_one():
    # With V = I (N <= d) the output row is the probability row itself.
    N, d = 6, 8
    q, k = rand(1, 1, N, d), rand(1, 1, N, d)
    v = np.zeros((1, 1, N, d))
    v[0, 0, :, :N] = np.eye(N)
    for causal in (False, True):
        o, _ = oracle.forward(q, k, v, causal, 0.9)
        p = o[0, 0, :, :N]
        np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
        assert (p >= 0).all()
        if causal:
            assert np.all(np.triu(p, 1) == 0.0)


def test_equal_v_rows_give_that_row():
    N, d = 11, 4
    row = rand(d)
    v = np.broadcast_to(row, (1, 2, N, d)).copy()
    for causal in (False, True):
        o, _ = oracle.forward(rand(1, 2, N, d), rand(1, 2, N, d), v, causal, 1.3)
        np.testing.assert_allclose(o, np.broadcast_to(row, o.shape), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_k_rows_give_mean_of_v(causal):
    N, d, s = 9, 5, 0.45
    q = rand(1, 1, N, d)
    krow = rand(d)
    k = np.broadcast_to(krow, (1, 1, N, d)).copy()
    v = rand(1, 1, N, d)
    o, lse = oracle.forward(q, k, v, causal, s)
    counts = np.arange(1, N + 1) if causal else np.full(N, N)
    if causal:
        expect_o = np.cumsum(v[0, 0], axis=0) / counts[:, None]
    else:
        expect_o = np.broadcast_to(v[0, 0].mean(axis=0), (N, d))
    np.testing.assert_allclose(o[0, 0], expect_o, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], s * (q[0, 0] @ krow) + np.log(counts), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_and_zero_scale(causal):
    N, d = 10, 3
    k, v = rand(1, 1, N, d), rand(1, 1, N, d)
    counts = np.arange(1, N + 1) if causal else np.full(N, N)
    for q, s in ((np.zeros((1, 1, N, d)), 0.8), (rand(1, 1, N, d), 0.0)):
        o, lse = oracle.forward(q, k, v, causal, s)
        np.testing.assert_allclose(lse[0, 0], np.log(counts), atol=1e-12)
        if not causal:
            np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0].mean(0), (N, d)),
                                       atol=1e-12)


def test_causal_first_row_and_single_token():
    N, d, s = 8, 6, 0.3
    q, k, v = rand(1, 1, N, d), rand(1, 1, N, d), rand(1, 1, N, d)
    o, lse = oracle.forward(q, k, v, True, s)
    assert np.array_equal(o[0, 0, 0], v[0, 0, 0])
    assert lse[0, 0, 0] == pytest.approx(s * q[0, 0, 0] @ k[0, 0, 0], abs=1e-14)
    o1, lse1 = oracle.forward(q[:, :, :1], k[:, :, :1], v[:, :, :1], False, s)
    assert np.array_equal(o1, v[:, :, :1])


def test_large_scores_stay_finite():
    # Max-shifted softmax: huge scores must not overflow.
    N, d = 12, 8
    q, k, v = 60 * rand(1, 1, N, d), 60 * rand(1, 1, N, d), rand(1, 1, N, d)
    o, lse = oracle.forward(q, k, v, False, 1.0)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    # The largest score dominates: output row equals the argmax key's value row.
    s = q[0, 0] @ k[0, 0].T
    am = s.argmax(axis=1)
    gap = np.sort(s, axis=1)[:, -1] - np.sort(s, axis=1)[:, -2]
    sel = gap > 50
    np.testing.assert_allclose(o[0, 0][sel], v[0, 0][am[sel]], atol=1e-12)
    np.testing.assert_allclose(lse[0, 0][sel], s.max(axis=1)[sel], atol=1e-12)


# ---------------------------------------------------------------- structure
def test_gqa_equals_repeat_interleaved_mha():
    B, Hq, Hkv, N, d = 2, 6, 2, 7, 4
    q, k, v, dO = rand(B, Hq, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, Hq, N, d)
    kr, vr = np.repeat(k, Hq // Hkv, axis=1), np.repeat(v, Hq // Hkv, axis=1)
    for causal in (False, True):
        o, lse = oracle.forward(q, k, v, causal, 0.5)
        o2, lse2 = oracle.forward(q, kr, vr, causal, 0.5)
        np.testing.assert_array_equal(o, o2)
        np.testing.assert_array_equal(lse, lse2)
        dq, dk, dv, _ = oracle.backward(q, k, v, dO, causal, 0.5)
        dq2, dk2, dv2, _ = oracle.backward(q, kr, vr, dO, causal, 0.5)
        np.testing.assert_allclose(dq, dq2, atol=1e-13)
        np.testing.assert_allclose(dk, dk2.reshape(B, Hkv, Hq // Hkv, N, d).sum(2), atol=1e-12)
        np.testing.assert_allclose(dv, dv2.reshape(B, Hkv, Hq // Hkv, N, d).sum(2), atol=1e-12)


def test_noncausal_key_permutation_invariance():
    N, d = 10, 4
    q, k, v, dO = rand(1, 2, N, d), rand(1, 2, N, d), rand(1, 2, N, d), rand(1, 2, N, d)
    perm = RNG.permutation(N)
    o, lse = oracle.forward(q, k, v, False, 0.6)
    o2, lse2 = oracle.forward(q, k[:, :, perm], v[:, :, perm], False, 0.6)
    np.testing.assert_allclose(o, o2, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, atol=1e-12)
    _, dk, dv, _ = oracle.backward(q, k, v, dO, False, 0.6)
    _, dk2, dv2, _ = oracle.backward(q, k[:, :, perm], v[:, :, perm], dO, False, 0.6)
    np.testing.assert_allclose(dk[:, :, perm], dk2, atol=1e-12)
    np.testing.assert_allclose(dv[:, :, perm], dv2, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(causal):
    """Adding one vector c to every key of a KV head adds scale * q_i . c to all
    of row i's scores: P and O are unchanged and LSE_i moves by scale * q_i . c.
    dS is unchanged, so dK and dV are too, and dQ_i = scale * sum_k dS_ik k_k is
    unchanged only because every row of dS sums to zero (the softmax-Jacobian
    term -D_i makes it so)."""
    B, Hq, Hkv, N, d, s = 2, 4, 2, 11, 6, 0.7
    q, k, v, dO = rand(B, Hq, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, Hq, N, d)
    c = rand(B, Hkv, 1, d)
    o, lse = oracle.forward(q, k, v, causal, s)
    o2, lse2 = oracle.forward(q, k + c, v, causal, s)
    g = Hq // Hkv
    shift = s * np.einsum("bhnd,bhd->bhn", q, np.repeat(c[:, :, 0, :], g, axis=1))
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(lse2, lse + shift, atol=1e-12)
    dq, dk, dv, _ = oracle.backward(q, k, v, dO, causal, s)
    dq2, dk2, dv2, _ = oracle.backward(q, k + c, v, dO, causal, s)
    for a, b in ((dq2, dq), (dk2, dk), (dv2, dv)):
        np.testing.assert_allclose(a, b, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_invariants(causal):
    B, Hq, Hkv, N, d = 1, 4, 2, 9, 5
    q, k, v, dO = rand(B, Hq, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, Hq, N, d)
    dq, dk, dv, D = oracle.backward(q, k, v, dO, causal, 0.8)
    # Shifting every key by the same vector leaves softmax unchanged: sum_k dK_k = 0.
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    # Rows of P sum to 1: sum_k dV_k = sum over the group's heads of sum_i dO_i.
    g = Hq // Hkv
    np.testing.assert_allclose(dv.sum(axis=2), dO.reshape(B, Hkv, g, N, d).sum(axis=(2, 3)),
                               atol=1e-12)
    # D_i = dO_i . O_i with O from the forward
    o, _ = oracle.forward(q, k, v, causal, 0.8)
    np.testing.assert_allclose(D, (dO * o).sum(-1), atol=1e-12)


# ---------------------------------------------------------------- finite differences
def _loss(q, k, v, dO, causal, s):
    o, _ = oracle.forward(q, k, v, causal, s)
    return float((o * dO).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,N,d", [(1, 1, 1, 6, 3), (1, 2, 1, 5, 4)])
def test_backward_matches_finite_differences(causal, B, Hq, Hkv, N, d):
    s = 0.9
    q, k, v, dO = rand(B, Hq, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, Hq, N, d)
    dq, dk, dv, _ = oracle.backward(q, k, v, dO, causal, s)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], dO, causal, s)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], dO, causal, s)
            fd[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g, fd, rtol=1e-6, atol=1e-7, err_msg=f"d{name}")


# ---------------------------------------------------------------- the pages' recurrences
@pytest.mark.parametrize("form", [online.fa1_form, online.fa2_form])
@pytest.mark.parametrize("causal", [False, True])
def test_online_recurrence_reproduces_definition(form, causal):
    rng = np.random.default_rng(7)
    for trial in range(6):
        N = int(rng.integers(1, 70))
        d = int(rng.integers(1, 9))
        q, k, v = 3 * rng.standard_normal((N, d)), rng.standard_normal((N, d)), \
            rng.standard_normal((N, d))
        sizes = tuple(int(x) for x in rng.integers(1, 17, size=5))
        o, lse = form(q, k, v, 0.5, causal, sizes)
        o_ref, lse_ref = oracle.forward(q[None, None], k[None, None], v[None, None], causal, 0.5)
        np.testing.assert_allclose(o, o_ref[0, 0], atol=1e-12)
        np.testing.assert_allclose(lse, lse_ref[0, 0], atol=1e-12)


def test_rejects_bad_head_grouping():
    with pytest.raises(ValueError):
        oracle.forward(rand(1, 3, 4, 2), rand(1, 2, 4, 2), rand(1, 2, 4, 2), False, 1.0)


# ---------------------------------------------------------------- rectangular (decoding) forward
@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d", [(1, 1, 1, 1, 1, 4), (2, 4, 2, 1, 13, 8),
                                              (1, 3, 1, 5, 40, 4), (1, 2, 2, 17, 3, 8)])
def test_rect_forward_bruteforce(B, Hq, Hkv, Nq, Nk, d):
    q, k, v = rand(B, Hq, Nq, d), rand(B, Hkv, Nk, d), rand(B, Hkv, Nk, d)
    o, lse = oracle.forward_rect(q, k, v, 0.7)
    o_n, lse_n, _ = naive.forward(q, k, v, False, 0.7)
    np.testing.assert_allclose(o, o_n, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_n, rtol=0, atol=1e-12)


def test_rect_forward_closed_forms_and_square_case():
    # identical keys: O = mean(V), LSE = s q.k + ln Nk; one key: O = V_0
    Nq, Nk, d, s = 3, 11, 5, 0.4
    q, v = rand(1, 1, Nq, d), rand(1, 1, Nk, d)
    krow = rand(d)
    k = np.broadcast_to(krow, (1, 1, Nk, d)).copy()
    o, lse = oracle.forward_rect(q, k, v, s)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0].mean(0), (Nq, d)), atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], s * (q[0, 0] @ krow) + np.log(Nk), atol=1e-12)
    o1, _ = oracle.forward_rect(q, k[:, :, :1], v[:, :, :1], s)
    np.testing.assert_allclose(o1[0, 0], np.broadcast_to(v[0, 0, 0], (Nq, d)), atol=1e-15)
    # Nq = Nk agrees with the square non-causal forward
    qs, ks, vs = rand(1, 2, 9, 4), rand(1, 2, 9, 4), rand(1, 2, 9, 4)
    a, la = oracle.forward_rect(qs, ks, vs, 0.5)
    b, lb = oracle.forward(qs, ks, vs, False, 0.5)
    np.testing.assert_allclose(a, b, atol=1e-14)
    np.testing.assert_allclose(la, lb, atol=1e-14)


# ---------------------------------------------------------------- sliding window
@pytest.mark.parametrize("W", [1, 2, 5, 16])
@pytest.mark.parametrize("B,Hq,Hkv,N,d", [(1, 1, 1, 9, 4), (2, 4, 2, 13, 8)])
def test_window_bruteforce(W, B, Hq, Hkv, N, d):
    q, k, v, dO = rand(B, Hq, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, Hq, N, d)
    o, lse = oracle.forward_window(q, k, v, W, 0.6)
    o_n, lse_n, _ = naive.forward(q, k, v, True, 0.6, window=W)
    np.testing.assert_allclose(o, o_n, atol=1e-12)
    np.testing.assert_allclose(lse, lse_n, atol=1e-12)
    g = oracle.backward_window(q, k, v, dO, W, 0.6)
    r = naive.backward(q, k, v, dO, True, 0.6, window=W)
    for a, b in zip(g, r[:3]):
        np.testing.assert_allclose(a, b, atol=1e-12)


def test_window_special_cases():
    N, d, s = 10, 4, 0.7
    q, k, v, dO = rand(1, 2, N, d), rand(1, 2, N, d), rand(1, 2, N, d), rand(1, 2, N, d)
    # window >= N is causal attention
    for W in (N, N + 7):
        o, lse = oracle.forward_window(q, k, v, W, s)
        oc, lc = oracle.forward(q, k, v, True, s)
        np.testing.assert_allclose(o, oc, atol=1e-14)
        np.testing.assert_allclose(lse, lc, atol=1e-14)
        g = oracle.backward_window(q, k, v, dO, W, s)
        gc = oracle.backward(q, k, v, dO, True, s)
        for a, b in zip(g, gc[:3]):
            np.testing.assert_allclose(a, b, atol=1e-12)
    # window 1: every query sees only itself
    o, lse = oracle.forward_window(q, k, v, 1, s)
    np.testing.assert_array_equal(o, v)
    np.testing.assert_allclose(lse, s * np.einsum("bhnd,bhnd->bhn", q, k), atol=1e-14)
    dq, dk, dv = oracle.backward_window(q, k, v, dO, 1, s)
    np.testing.assert_allclose(dq, 0.0, atol=1e-14)  # P = 1 exactly: no gradient through S
    np.testing.assert_allclose(dv, dO, atol=1e-14)


@pytest.mark.parametrize("W", [2, 3])
def test_window_backward_finite_differences(W):
    B, Hq, Hkv, N, d, s = 1, 2, 1, 6, 3, 0.9
    q, k, v, dO = rand(B, Hq, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, Hq, N, d)
    dq, dk, dv = oracle.backward_window(q, k, v, dO, W, s)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args = {"q": q, "k": k, "v": v}
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args[name] = xp
            lp = float((oracle.forward_window(args["q"], args["k"], args["v"], W, s)[0] * dO).sum())
            args[name] = xm
            lm = float((oracle.forward_window(args["q"], args["k"], args["v"], W, s)[0] * dO).sum())
            fd[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g, fd, rtol=1e-6, atol=1e-7, err_msg=f"d{name}")
