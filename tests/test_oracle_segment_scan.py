"""Pins of the segment decomposition behind the chunk-level scan (CPU).

The scan rests on one fact of the recurrence: over a run of tokens the state
update is affine, S_end = S_start M + B.  These tests pin the reference
decomposition in ``oracle.segment_scan`` to the plain recurrence and to the
one-token closed form."""
import numpy as np
import pytest

from gated_delta_rule_09_gb300 import inputs as I
from oracle import gdn_recurrence_f64
from oracle.segment_scan import segment_propagator, segment_scan_f64


def test_one_token_propagator_closed_form():
    """One token: M = alpha (I - beta k k^T), B = beta v k^T."""
    rng = np.random.default_rng(3)
    dk, dv, H = 5, 3, 2
    k = rng.standard_normal((1, 1, H, dk))
    v = rng.standard_normal((1, 1, H, dv))
    q = rng.standard_normal((1, 1, H, dk))
    la = np.log(rng.uniform(0.5, 1.0, (1, 1, H)))
    beta = rng.uniform(0.0, 2.0, (1, 1, H))
    M, B = segment_propagator(q, k, v, la, beta)
    for h in range(H):
        kk = k[0, 0, h][:, None]
        a, b = np.exp(la[0, 0, h]), beta[0, 0, h]
        np.testing.assert_allclose(M[h], a * (np.eye(dk) - b * kk @ kk.T), atol=1e-14)
        np.testing.assert_allclose(B[h], b * v[0, 0, h][:, None] @ kk.T, atol=1e-14)


def test_propagator_composes_per_token_maps():
    """The run's (M, B) is the ordered composition of its tokens' maps."""
    x = I.custom(1, 2, 7, 6, 4, 16, dtype="f32", seed=4)
    M, B = segment_propagator(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"])
    Mc = np.broadcast_to(np.eye(6), (2, 6, 6)).copy()
    Bc = np.zeros((2, 4, 6))
    for t in range(7):
        sl = (slice(None), slice(t, t + 1))
        Mt, Bt = segment_propagator(*(x[n][sl] for n in ("q", "k", "v", "log_alpha", "beta")))
        Mc = np.einsum("hij,hjk->hik", Mc, Mt)
        Bc = np.einsum("hvi,hij->hvj", Bc, Mt) + Bt
    np.testing.assert_allclose(M, Mc, atol=1e-12)
    np.testing.assert_allclose(B, Bc, atol=1e-12)


@pytest.mark.parametrize("segments,T", [(1, 200), (2, 200), (3, 200), (4, 130), (13, 800)])
def test_segment_scan_equals_recurrence(segments, T):
    x = I.custom(2, 2, T, 8, 6, 16, dtype="f32", seed=segments + T, s0="normal_0.02",
                 beta="uniform_0_2")
    ro, rS = gdn_recurrence_f64(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S0=x["S0"])
    o, S, _ = segment_scan_f64(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], segments,
                               C=16, S0=x["S0"])
    np.testing.assert_allclose(o, ro, atol=1e-10, rtol=1e-10)
    np.testing.assert_allclose(S, rS, atol=1e-10, rtol=1e-10)


def test_mutant_scan_order_fails():
    """Composing the segment maps in the wrong order is caught."""
    x = I.custom(1, 1, 96, 8, 6, 16, dtype="f32", seed=9, s0="normal_0.02")
    args = [x[n] for n in ("q", "k", "v", "log_alpha", "beta")]
    M1, B1 = segment_propagator(*(a[:, :48] for a in args))
    M2, B2 = segment_propagator(*(a[:, 48:] for a in args))
    S0 = np.asarray(x["S0"], np.float64)[0]
    good = np.einsum("hvi,hij->hvj", np.einsum("hvi,hij->hvj", S0, M1) + B1, M2) + B2
    bad = np.einsum("hvi,hij->hvj", np.einsum("hvi,hij->hvj", S0, M2) + B2, M1) + B1
    _, rS = gdn_recurrence_f64(*args, S0=x["S0"])
    assert np.allclose(good, rS[0], atol=1e-10)
    assert not np.allclose(bad, rS[0], atol=1e-3)
