"""Pins of the two UT-inverse statements in the chunk reference (CPU): the
doubling product (finite Neumann series) against forward substitution, the
nilpotency it rests on, and the factor it cannot drop."""
import numpy as np

from gated_delta_rule_09_gb300 import inputs as I
from oracle.chunk_reference import forward_substitution, ut_inverse_doubling


def test_doubling_equals_forward_substitution():
    for C, scale in ((16, 0.3), (32, 0.1), (64, 0.04), (64, 0.2)):
        A = np.asarray(I.ut_matrices(3, C, scale, seed=C)[0], np.float64)
        Tf = forward_substitution(-A)          # (E - (-A))^{-1} = (I + A)^{-1}
        Td = ut_inverse_doubling(A)
        np.testing.assert_allclose(Td, Tf, atol=1e-12 * max(1.0, np.abs(Tf).max()))
        np.testing.assert_allclose((np.eye(C) + A) @ Td, np.eye(C), atol=1e-11)


def test_strictly_lower_is_nilpotent():
    A = np.asarray(I.ut_matrices(1, 64, 1.0, seed=5)[0], np.float64)
    assert np.abs(np.linalg.matrix_power(A, 63)).max() > 0  # one nonzero path remains
    np.testing.assert_array_equal(np.linalg.matrix_power(A, 64), np.zeros((64, 64)))


def test_dropping_the_last_factor_is_wrong():
    """Without (I + A^32) the powers 32..63 are missing: detectable when they
    are not negligible (entries of order 1)."""
    A = np.asarray(I.ut_matrices(1, 64, 1.0, seed=7)[0], np.float64)
    Tf = forward_substitution(-A)
    X = -A
    T = np.eye(64) + X
    for _ in range(4):  # up to (I + A^16): powers < 32 only
        X = X @ X
        T = T @ (np.eye(64) + X)
    assert not np.allclose(T, Tf, atol=1e-6 * np.abs(Tf).max())
