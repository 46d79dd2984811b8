"""Pins of the oracle's general form C = alpha * op(A) * op(B) + beta * C.

The pages define only C = A * B; the general form is the standard BLAS GEMM
(beta = 0 means C is not read). Each check below fails for a plausible slip:
a transposed index (explicit numpy transposes), a lost or misplaced scale
(integer closed forms with alpha, beta != 1), reading C when beta = 0 (NaN C),
a wrong error scale S.
"""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_major_gb300 import workloads as wl


def _ints(shape, seed):
    return np.random.default_rng(seed).integers(-5, 6, size=shape).astype(np.float32)


@pytest.mark.parametrize("transA,transB", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_transposes_match_explicit_transposition(transA, transB):
    rng = np.random.default_rng(transA * 2 + transB)
    M, N, K = 13, 17, 29
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    As = np.ascontiguousarray(A.T) if transA else A  # stored form
    Bs = np.ascontiguousarray(B.T) if transB else B
    C64, S = oracle.gemm_f64(As, Bs, transA=bool(transA), transB=bool(transB))
    R64, RS = oracle.sgemm_f64(A, B)
    # Same products, same k order: bit-identical.
    assert np.array_equal(C64.view(np.uint64), R64.view(np.uint64))
    assert np.array_equal(S.view(np.uint64), RS.view(np.uint64))


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (3.0, -2.0), (-1.0, 1.0), (0.0, 4.0), (2.0, 0.0)])
def test_alpha_beta_integer_closed_form(alpha, beta):
    M, N, K = 9, 11, 21
    A, B, C = _ints((M, K), 1), _ints((K, N), 2), _ints((M, N), 3)
    exact = int(alpha) * (A.astype(np.int64) @ B.astype(np.int64)) + int(beta) * C.astype(np.int64)
    C64, S = oracle.gemm_f64(A, B, alpha=alpha, beta=beta, C_in=C if beta else None)
    assert np.array_equal(C64, exact.astype(np.float64))
    s_exact = abs(int(alpha)) * (np.abs(A).astype(np.int64) @ np.abs(B).astype(np.int64))
    if beta:
        s_exact = s_exact + abs(int(beta)) * np.abs(C).astype(np.int64)
    assert np.array_equal(S, s_exact.astype(np.float64))


def test_beta_zero_does_not_read_c():
    A, B = _ints((4, 6), 4), _ints((6, 5), 5)
    C = np.full((4, 5), np.nan, np.float32)
    C64, _ = oracle.gemm_f64(A, B, alpha=1.0, beta=0.0, C_in=C)
    assert np.all(np.isfinite(C64))
    assert np.array_equal(C64, (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64))


def test_alpha_zero_scales_c_only():
    A = np.full((3, 4), np.float32(1e30))
    B = np.full((4, 2), np.float32(1e30))
    C = _ints((3, 2), 6)
    C64, S = oracle.gemm_f64(A, B, alpha=0.0, beta=-3.0, C_in=C)
    assert np.array_equal(C64, -3.0 * C.astype(np.float64))
    assert np.array_equal(S, 3.0 * np.abs(C).astype(np.float64))


@pytest.mark.parametrize("transA,transB", [(0, 0), (1, 1), (1, 0)])
def test_rational_brute_force_general(transA, transB):
    rng = np.random.default_rng(40 + transA + 2 * transB)
    M, N, K = 3, 4, 7
    A = rng.standard_normal((K, M) if transA else (M, K)).astype(np.float32)
    B = rng.standard_normal((N, K) if transB else (K, N)).astype(np.float32)
    C = rng.standard_normal((M, N)).astype(np.float32)
    alpha, beta = 0.75, -1.25  # exact in binary
    C64, S = oracle.gemm_f64(A, B, transA=bool(transA), transB=bool(transB), alpha=alpha, beta=beta,
                             C_in=C)
    g = (K + 2) * 2.0 ** -53 / (1 - (K + 2) * 2.0 ** -53)
    for i in range(M):
        for j in range(N):
            acc = Fraction(0)
            sc = Fraction(0)
            for k in range(K):
                a = Fraction(float(A[k, i] if transA else A[i, k]))
                b = Fraction(float(B[j, k] if transB else B[k, j]))
                acc += a * b
                sc += abs(a) * abs(b)
            exact = Fraction(alpha) * acc + Fraction(beta) * Fraction(float(C[i, j]))
            scale = abs(Fraction(alpha)) * sc + abs(Fraction(beta)) * abs(Fraction(float(C[i, j])))
            assert abs(Fraction(float(C64[i, j])) - exact) <= Fraction(g) * scale
            assert abs(Fraction(float(S[i, j])) - scale) <= Fraction(g) * scale


def test_sampled_general_matches_full():
    A, B = wl.make_pair(37, 41, 23, "normal", 12)
    At = np.ascontiguousarray(A.T)
    C = np.random.default_rng(3).standard_normal((37, 41)).astype(np.float32)
    C64, S = oracle.gemm_f64(At, B, transA=True, alpha=-0.5, beta=2.0, C_in=C)
    r, c = wl.sample_positions(37, 41, 60, seed=3)
    c64, s = oracle.gemm_f64_at(At, B, r, c, transA=True, alpha=-0.5, beta=2.0, C_in=C)
    assert np.array_equal(c64, C64[r, c]) and np.array_equal(s, S[r, c])


def test_general_form_rejects_bad_strides():
    with pytest.raises(ValueError):
        oracle.gemm_f64(np.zeros((3, 4), np.float32), np.zeros((5, 2), np.float32))
    with pytest.raises(ValueError):  # beta != 0 without C_in
        oracle.gemm_f64(np.zeros((3, 4), np.float32), np.zeros((4, 2), np.float32), beta=1.0)
