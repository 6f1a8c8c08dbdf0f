"""Pins for the GEMM oracle (C = A B^T), independent of the oracle's own code."""
import numpy as np
import pytest

from oracle import gemm_nt, gemm_nt_rows


def brute(a, b):
    """Triple loop in pure Python floats: an evaluator that shares nothing with the oracle."""
    M, K = len(a), len(a[0])
    N = len(b)
    return [[sum(float(a[m][k]) * float(b[n][k]) for k in range(K)) for n in range(N)] for m in range(M)]


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (8, 4, 16), (5, 9, 2)])
def test_matches_brute_force(M, N, K):
    r = np.random.default_rng(M * 100 + N * 10 + K)
    a = r.standard_normal((M, K))
    b = r.standard_normal((N, K))
    c = gemm_nt(a, b)
    ref = np.array(brute(a.tolist(), b.tolist()))
    assert c.shape == (M, N)
    assert np.max(np.abs(c - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_transposition_and_identity():
    r = np.random.default_rng(7)
    a = r.standard_normal((6, 4))
    b = r.standard_normal((3, 4))
    # (A B^T)^T = B A^T: catches a transposed operand
    assert np.array_equal(gemm_nt(a, b).T, gemm_nt(b, a))
    # X I^T = X and I W^T = W^T
    assert np.array_equal(gemm_nt(a, np.eye(4)), a)
    assert np.array_equal(gemm_nt(np.eye(4), b), b.T)


def test_small_integers_exact():
    a = np.array([[1, 2, 3], [4, 5, 6]], dtype=np.float64)
    b = np.array([[1, 0, -1], [2, 2, 2], [0, 1, 0], [-3, 1, 4]], dtype=np.float64)
    # by hand: row 0 = (1-3, 2+4+6, 2, -3+2+12), row 1 = (4-6, 8+10+12, 5, -12+5+24)
    expect = np.array([[-2, 12, 2, 11], [-2, 30, 5, 17]], dtype=np.float64)
    assert np.array_equal(gemm_nt(a, b), expect)


def test_linearity_and_rows():
    r = np.random.default_rng(11)
    a1, a2 = r.standard_normal((5, 8)), r.standard_normal((5, 8))
    b = r.standard_normal((7, 8))
    assert np.allclose(gemm_nt(a1 + 2.0 * a2, b), gemm_nt(a1, b) + 2.0 * gemm_nt(a2, b), rtol=0, atol=1e-12)
    assert np.array_equal(gemm_nt_rows(a1, b, [4, 0]), gemm_nt(a1, b)[[4, 0]])


def test_shape_errors():
    with pytest.raises(ValueError):
        gemm_nt(np.zeros((2, 3)), np.zeros((4, 5)))


def test_planted_transpose_mistake_is_caught():
    """A plausible bug (A B instead of A B^T on square shapes) must fail the brute-force pin."""
    r = np.random.default_rng(3)
    a = r.standard_normal((4, 4))
    b = r.standard_normal((4, 4))
    wrong = a @ b
    ref = np.array(brute(a.tolist(), b.tolist()))
    assert np.max(np.abs(wrong - ref)) > 1e-3
