"""The oracle pinned to what the pages and the mathematics fix (CPU only)."""
import os

import numpy as np
import pytest

import pins
from oracle import gdn_recurrence_f64
from oracle.chunk_reference import (chunk_step, forward_substitution,
                                    gdn_chunk_reference_f64)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def oracle_impl(q, k, v, log_alpha, beta, S0=None, eta=None, cu_seqlens=None):
    return gdn_recurrence_f64(q, k, v, log_alpha, beta, S0=S0, eta=eta,
                              cu_seqlens=cu_seqlens, n_threads=2)


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle_impl)


def _random_strict_lower(rng, n, scale=1.0):
    return np.tril(rng.uniform(-scale, scale, (n, n)), -1)


def test_forward_substitution_worked_example():
    """The 4x4 symbolic T of the page's forward-substitution example."""
    rows = pins.read_golden(os.path.join(GOLDEN, "forward_substitution_4x4.txt"))
    assert len(rows) == 16
    rng = np.random.default_rng(0)
    for _ in range(5):
        A = _random_strict_lower(rng, 4)
        T = forward_substitution(A)
        for (i, j), expr in rows:
            assert abs(T[i - 1, j - 1] - pins.parse_expr(expr, A)) < 1e-14, (i, j, expr)


def test_path_powers_worked_example():
    """A^2, A^3 path sums and A^4 = 0 at t = 4; the Neumann sum is exact."""
    rows = pins.read_golden(os.path.join(GOLDEN, "path_powers_4x4.txt"))
    rng = np.random.default_rng(1)
    A = _random_strict_lower(rng, 4)
    powers = {2: A @ A, 3: A @ A @ A}
    expect = {2: np.zeros((4, 4)), 3: np.zeros((4, 4))}
    for (p, i, j), expr in rows:
        expect[p][i - 1, j - 1] = pins.parse_expr(expr, A)
    for p in (2, 3):
        np.testing.assert_allclose(powers[p], expect[p], atol=1e-14)
    assert np.all(A @ A @ A @ A == 0.0)
    np.testing.assert_allclose(forward_substitution(A),
                               np.eye(4) + A + A @ A + A @ A @ A, atol=1e-14)


def test_w_expansion_worked_example():
    """w_1..w_4 over b_j = beta_j k_j with A_ij = -beta_i k_j.k_i equal the
    page's w_t recursion and T diag(beta) K."""
    rows = pins.read_golden(os.path.join(GOLDEN, "w_expansion_4x4.txt"))
    rng = np.random.default_rng(2)
    d = 5
    K = rng.standard_normal((4, d))
    beta = rng.uniform(0, 1, 4)
    A = np.zeros((4, 4))
    for i in range(4):
        for j in range(i):
            A[i, j] = -beta[i] * np.dot(K[j], K[i])
    b = beta[:, None] * K
    coef = np.zeros((4, 4))
    for (t, j), expr in rows:
        coef[t - 1, j - 1] = pins.parse_expr(expr, A)
    w_fixture = coef @ b
    w_rec = []
    for t in range(4):
        wt = beta[t] * K[t]
        for tau in range(t):
            wt = wt - beta[t] * np.dot(K[tau], K[t]) * w_rec[tau]
        w_rec.append(wt)
    np.testing.assert_allclose(w_fixture, np.array(w_rec), atol=1e-13)
    np.testing.assert_allclose(forward_substitution(A) @ b, np.array(w_rec), atol=1e-13)


def test_forward_substitution_inverts():
    rng = np.random.default_rng(3)
    for n in (1, 2, 16, 64):
        A = _random_strict_lower(rng, n, 0.2)
        T = forward_substitution(A)
        np.testing.assert_allclose((np.eye(n) - A) @ T, np.eye(n), atol=1e-12)
        assert np.all(np.triu(T, 1) == 0) and np.all(np.diag(T) == 1.0)


def _rand_inputs(rng, B, T, H, dk, dv):
    q = rng.standard_normal((B, T, H, dk))
    k = pins._unit(rng.standard_normal((B, T, H, dk)))
    v = rng.standard_normal((B, T, H, dv))
    la = -np.logaddexp(0, rng.standard_normal((B, T, H))) * 0.3
    be = 1 / (1 + np.exp(-rng.standard_normal((B, T, H))))
    return q, k, v, la, be


@pytest.mark.parametrize("T,C", [(64, 16), (50, 16), (5, 16), (130, 32), (1, 8)])
def test_chunk_form_matches_recurrence(T, C):
    """The four-step chunk summary of the GDN derivation page reaches the
    sequential result (full chunks, a ragged tail, T < C, T = 1)."""
    rng = np.random.default_rng(T * 7 + C)
    B, H, dk, dv = 2, 2, 8, 12
    q, k, v, la, be = _rand_inputs(rng, B, T, H, dk, dv)
    S0 = rng.standard_normal((B, H, dv, dk)) * 0.1
    o1, S1 = gdn_recurrence_f64(q, k, v, la, be, S0=S0)
    o2, S2 = gdn_chunk_reference_f64(q, k, v, la, be, S0=S0, C=C)
    np.testing.assert_allclose(o2, o1, atol=1e-11, rtol=0)
    np.testing.assert_allclose(S2, S1, atol=1e-11, rtol=0)


def test_chunk_form_varlen_matches_recurrence():
    rng = np.random.default_rng(11)
    lens = [17, 64, 1, 0, 40]
    Tt = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v, la, be = _rand_inputs(rng, 1, Tt, 3, 8, 8)
    S0 = rng.standard_normal((len(lens), 3, 8, 8)) * 0.1
    o1, S1 = gdn_recurrence_f64(q, k, v, la, be, S0=S0, cu_seqlens=cu)
    o2, S2 = gdn_chunk_reference_f64(q, k, v, la, be, S0=S0, C=16, cu_seqlens=cu)
    np.testing.assert_allclose(o2, o1, atol=1e-11, rtol=0)
    np.testing.assert_allclose(S2, S1, atol=1e-11, rtol=0)


def test_chunk_stage_identities():
    """Stage-level facts of one chunk: L strictly lower, T (I + L) = I, and the
    state update of the WY form equals the dense product form."""
    rng = np.random.default_rng(12)
    n, dk, dv = 16, 8, 6
    q, k, v, la, be = (x[0, :, 0] for x in _rand_inputs(rng, 1, n, 1, dk, dv))
    S = rng.standard_normal((dv, dk))
    r = chunk_step(q, k, v, la, be, S)
    assert np.all(np.triu(r["L"]) == 0)
    np.testing.assert_allclose(r["T"] @ (np.eye(n) + r["L"]), np.eye(n), atol=1e-12)
    a = np.exp(la)
    St = S.copy()
    for t in range(n):
        St = St @ (a[t] * (np.eye(dk) - be[t] * np.outer(k[t], k[t]))) + be[t] * np.outer(v[t], k[t])
    np.testing.assert_allclose(r["S_next"], St, atol=1e-11)


def test_resume_and_thread_invariance():
    """Split-and-resume equals one call; the thread count changes nothing."""
    rng = np.random.default_rng(13)
    q, k, v, la, be = _rand_inputs(rng, 2, 40, 3, 8, 4)
    o, S = gdn_recurrence_f64(q, k, v, la, be, n_threads=1)
    o4, S4 = gdn_recurrence_f64(q, k, v, la, be, n_threads=4)
    assert np.array_equal(o, o4) and np.array_equal(S, S4)
    oa, Sa = gdn_recurrence_f64(q[:, :25], k[:, :25], v[:, :25], la[:, :25], be[:, :25])
    ob, Sb = gdn_recurrence_f64(q[:, 25:], k[:, 25:], v[:, 25:], la[:, 25:], be[:, 25:], S0=Sa)
    np.testing.assert_allclose(np.concatenate([oa, ob], axis=1), o, atol=1e-12)
    np.testing.assert_allclose(Sb, S, atol=1e-12)


def test_oracle_rejects_bad_cu_seqlens():
    rng = np.random.default_rng(14)
    q, k, v, la, be = _rand_inputs(rng, 1, 10, 1, 4, 4)
    with pytest.raises(ValueError):
        gdn_recurrence_f64(q, k, v, la, be, cu_seqlens=np.array([0, 6, 4, 10], np.int32))
    with pytest.raises(ValueError):
        gdn_recurrence_f64(q, k, v, la, be, cu_seqlens=np.array([0, 4, 9], np.int32))
