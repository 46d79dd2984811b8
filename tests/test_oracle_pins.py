"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each check is chosen so that a plausible mistake in the oracle fails it: a
dropped or extra term (all-ones, closed form, single nonzero), a transposed
operand or swapped index (closed form with asymmetric entries, permutation,
block identity), a wrong accumulation precision or order (float32 brute force
bit for bit, exact rational brute force within the rounding bound), a wrong
stride (padded rows).
"""

import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_major_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            vals[key] = rest
    return vals


# ---------------------------------------------------------------- closed forms

def test_allones_page_value():
    g = _golden("allones_1024.txt")
    M, N, K = int(g["M"]), int(g["N"]), int(g["K"])
    A = np.full((M, K), float(g["value_A"]), dtype=np.float32)
    B = np.full((K, N), float(g["value_B"]), dtype=np.float32)
    expected = float(g["expected_C"])
    C32 = oracle.sgemm_f32(A, B)
    assert np.all(C32 == np.float32(expected))
    # The double twin on a band of rows (the full 1024^3 in double is slow).
    C64, S = oracle.sgemm_f64_rows(A, B, 0, 64)
    assert np.all(C64 == expected) and np.all(S == expected)


@pytest.mark.parametrize("K", [1, 7, 100, 4096])
def test_allones_any_k(K):
    A = np.ones((3, K), dtype=np.float32)
    B = np.ones((K, 5), dtype=np.float32)
    assert np.all(oracle.sgemm_f32(A, B) == K)
    C64, S = oracle.sgemm_f64(A, B)
    assert np.all(C64 == K) and np.all(S == K)


def _closed_form(M, N, K):
    """A[i][k] = i + k + 1, B[k][j] = k - 2j + 3: exact integer C from power sums.

    C[i][j] = sum_k (i + k + 1)(k - 2j + 3)
            = (i + 1)(3 - 2j) K + ((i + 1) + (3 - 2j)) S1 + S2
    with S1 = sum k = K(K-1)/2 and S2 = sum k^2 = (K-1)K(2K-1)/6.
    """
    i = np.arange(M, dtype=np.int64)[:, None]
    j = np.arange(N, dtype=np.int64)[None, :]
    S1 = K * (K - 1) // 2
    S2 = (K - 1) * K * (2 * K - 1) // 6
    a0, b0 = i + 1, 3 - 2 * j
    return a0 * b0 * K + (a0 + b0) * S1 + S2


@pytest.mark.parametrize("M,N,K", [(5, 7, 3), (17, 9, 33), (40, 23, 64)])
def test_polynomial_closed_form(M, N, K):
    i = np.arange(M)[:, None]
    k = np.arange(K)[None, :]
    A = (i + k + 1).astype(np.float32)
    kk = np.arange(K)[:, None]
    j = np.arange(N)[None, :]
    B = (kk - 2 * j + 3).astype(np.float32)
    exact = _closed_form(M, N, K)
    assert np.abs(exact).max() < 2**24  # every partial sum is exact in float32
    assert np.array_equal(oracle.sgemm_f32(A, B).astype(np.int64), exact)
    C64, _ = oracle.sgemm_f64(A, B)
    assert np.array_equal(C64.astype(np.int64), exact)
    # A transposed operand or a swapped output index would not match: the
    # closed form is not symmetric in (i, j) nor in the roles of A and B.
    assert not np.array_equal(exact[: min(M, N), : min(M, N)], exact[: min(M, N), : min(M, N)].T)


def test_identity_and_permutation():
    rng = np.random.default_rng(7)
    B = rng.standard_normal((6, 9)).astype(np.float32)
    A = rng.standard_normal((4, 6)).astype(np.float32)
    I6 = np.eye(6, dtype=np.float32)
    I9 = np.eye(9, dtype=np.float32)
    assert np.array_equal(oracle.sgemm_f32(I6, B), B)
    assert np.array_equal(oracle.sgemm_f32(A, I6), A)
    C64, S = oracle.sgemm_f64(I6, B)
    assert np.array_equal(C64, B.astype(np.float64))
    assert np.array_equal(S, np.abs(B).astype(np.float64))
    C64, _ = oracle.sgemm_f64(B, I9)
    assert np.array_equal(C64, B.astype(np.float64))
    perm = rng.permutation(6)
    P = I6[perm]
    assert np.array_equal(oracle.sgemm_f32(P, B), B[perm])
    # Column permutation via a permutation on the right.
    Q = np.ascontiguousarray(I9[:, rng.permutation(9)])
    assert np.array_equal(oracle.sgemm_f32(B, Q), B @ Q)


def test_single_nonzero_term():
    rng = np.random.default_rng(3)
    B = rng.standard_normal((11, 13)).astype(np.float32)
    A = np.zeros((5, 11), dtype=np.float32)
    A[2, 7] = np.float32(-1.75)
    C = oracle.sgemm_f32(A, B)
    expected = np.zeros((5, 13), dtype=np.float32)
    expected[2] = np.float32(-1.75) * B[7]
    assert np.array_equal(C, expected)
    # In double the single product is exact.
    exact = np.zeros((5, 13), dtype=np.float64)
    exact[2] = -1.75 * B[7].astype(np.float64)
    C64, S = oracle.sgemm_f64(A, B)
    assert np.array_equal(C64, exact)
    assert np.array_equal(S, np.abs(exact))


def test_empty_sum_and_empty_shapes():
    A = np.zeros((3, 0), dtype=np.float32)
    B = np.zeros((0, 4), dtype=np.float32)
    assert np.array_equal(oracle.sgemm_f32(A, B), np.zeros((3, 4), np.float32))
    C64, S = oracle.sgemm_f64(A, B)
    assert np.all(C64 == 0) and np.all(S == 0)
    assert oracle.sgemm_f32(np.zeros((0, 5), np.float32), np.zeros((5, 2), np.float32)).shape == (0, 2)
    assert oracle.sgemm_f32(np.zeros((2, 5), np.float32), np.zeros((5, 0), np.float32)).shape == (2, 0)


# ------------------------------------------------------ block identity (page toy)

def test_block_identity_page_toy():
    g = _golden("tiled_toy_8x8.txt")
    n, t = int(g["N"]), int(g["TILE"])
    rng = np.random.default_rng(11)
    A = rng.integers(-9, 10, size=(n, n)).astype(np.float32)
    B = rng.integers(-9, 10, size=(n, n)).astype(np.float32)
    C = oracle.sgemm_f32(A, B)

    def blk(X, r, c):
        return np.ascontiguousarray(X[r * t:(r + 1) * t, c * t:(c + 1) * t])

    for spec in g["blocks"].split():
        lhs, rhs = spec.split("=")
        r, c = int(lhs[1]), int(lhs[2])
        total = np.zeros((t, t), dtype=np.float32)
        for term in rhs.split("+"):
            a, b = term.split("*")
            total += oracle.sgemm_f32(blk(A, int(a[1]), int(a[2])), blk(B, int(b[1]), int(b[2])))
        assert np.array_equal(blk(C, r, c), total), spec


# ----------------------------------------------------------------- brute force

def _exact(A, B):
    M, K = A.shape
    N = B.shape[1]
    Af = [[Fraction(float(A[i, k])) for k in range(K)] for i in range(M)]
    Bf = [[Fraction(float(B[k, j])) for j in range(N)] for k in range(K)]
    C = [[sum((Af[i][k] * Bf[k][j] for k in range(K)), Fraction(0)) for j in range(N)]
         for i in range(M)]
    S = [[sum((abs(Af[i][k]) * abs(Bf[k][j]) for k in range(K)), Fraction(0)) for j in range(N)]
         for i in range(M)]
    return C, S


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 1, 0), (2, 3, 4, 1), (5, 4, 9, 2), (3, 6, 17, 3)])
def test_rational_brute_force(M, N, K, seed):
    rng = np.random.default_rng(seed)
    A = (rng.standard_normal((M, K)) * 10.0 ** rng.integers(-3, 4, (M, K))).astype(np.float32)
    B = (rng.standard_normal((K, N)) * 10.0 ** rng.integers(-3, 4, (K, N))).astype(np.float32)
    Cx, Sx = _exact(A, B)
    C32 = oracle.sgemm_f32(A, B)
    C64, S = oracle.sgemm_f64(A, B)
    u32, u64 = 2.0 ** -24, 2.0 ** -53
    g32 = K * u32 / (1 - K * u32)
    g64 = K * u64 / (1 - K * u64)
    for i in range(M):
        for j in range(N):
            s = float(Sx[i][j])
            # Recursive summation bound: |computed - exact| <= gamma_K * sum |terms|.
            assert abs(Fraction(float(C64[i, j])) - Cx[i][j]) <= Fraction(g64) * Sx[i][j]
            assert abs(Fraction(float(C32[i, j])) - Cx[i][j]) <= Fraction(g32 * 1.0000001) * Sx[i][j]
            assert abs(float(S[i, j]) - s) <= g64 * s


@pytest.mark.parametrize("M,N,K,seed", [(3, 4, 5, 0), (7, 2, 31, 1), (4, 9, 64, 2)])
def test_float32_brute_force_bit_exact(M, N, K, seed):
    """The pages' CPU loop evaluated with numpy float32 scalars, product then sum."""
    rng = np.random.default_rng(100 + seed)
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    ref = np.zeros((M, N), dtype=np.float32)
    for i in range(M):
        for j in range(N):
            s = np.float32(0.0)
            for k in range(K):
                p = np.float32(A[i, k] * B[k, j])
                s = np.float32(s + p)
            ref[i, j] = s
    got = oracle.sgemm_f32(A, B)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    # A fused multiply-add (one rounding) would differ somewhere on these
    # inputs: check that the fused variant really is distinguishable.
    fused = np.zeros((M, N), dtype=np.float32)
    for i in range(M):
        for j in range(N):
            s = 0.0
            for k in range(K):
                s = float(np.float32(float(A[i, k]) * float(B[k, j]) + s))
            fused[i, j] = s
    assert not np.array_equal(fused, ref)


def test_small_integer_exact():
    rng = np.random.default_rng(5)
    A = rng.integers(-4, 5, (37, 300)).astype(np.float32)
    B = rng.integers(-4, 5, (300, 29)).astype(np.float32)
    exact = A.astype(np.int64) @ B.astype(np.int64)
    assert np.array_equal(oracle.sgemm_f32(A, B).astype(np.int64), exact)
    C64, S = oracle.sgemm_f64(A, B)
    assert np.array_equal(C64.astype(np.int64), exact)
    assert np.array_equal(S.astype(np.int64), np.abs(A).astype(np.int64) @ np.abs(B).astype(np.int64))


# ------------------------------------------------------------ twins and strides

def test_rows_twin_bit_identical():
    A, B = wl.make_pair(37, 53, 71, "normal", 9)
    C64, S = oracle.sgemm_f64(A, B)
    for nthreads in (1, 3, 8):
        R64, RS = oracle.sgemm_f64_rows(A, B, 0, 37, nthreads=nthreads)
        assert np.array_equal(R64.view(np.uint64), C64.view(np.uint64))
        assert np.array_equal(RS.view(np.uint64), S.view(np.uint64))
    R64, RS = oracle.sgemm_f64_rows(A, B, 10, 20, nthreads=4)
    assert np.array_equal(R64, C64[10:20]) and np.array_equal(RS, S[10:20])


@pytest.mark.parametrize("dist", ["normal", "uniform01"])
def test_float_rows_twin_bit_identical(dist):
    """The timed float twin (i-k-j, threaded by rows) adds the same rounded
    products in the same k order as the pages' i-j-k loop: every bit equal,
    for any band of rows, thread count and padded stride."""
    A, B = wl.make_pair(41, 67, 203, dist, 11)
    C = oracle.sgemm_f32(A, B)
    for nthreads in (1, 3, 16):
        R = oracle.sgemm_f32_rows(A, B, nthreads=nthreads)
        assert np.array_equal(R.view(np.uint32), C.view(np.uint32))
    R = oracle.sgemm_f32_rows(A, B, 7, 30, nthreads=4)
    assert np.array_equal(R.view(np.uint32), C[7:30].view(np.uint32))
    Rp = oracle.sgemm_f32_rows(wl.strided(A, 211), wl.strided(B, 70), nthreads=2)
    assert np.array_equal(Rp.view(np.uint32), C.view(np.uint32))
    # And it is the float loop, not a double one: a long same-sign sum
    # differs from the double product rounded once.
    A1, B1 = wl.make_pair(3, 5, 4096, "uniform01", 2)
    C64, _ = oracle.sgemm_f64(A1, B1)
    assert not np.array_equal(oracle.sgemm_f32_rows(A1, B1), C64.astype(np.float32))


def test_sampled_twin_matches():
    A, B = wl.make_pair(29, 31, 47, "uniform", 4)
    C64, S = oracle.sgemm_f64(A, B)
    r, c = wl.sample_positions(29, 31, 50, seed=1)
    c64, s = oracle.sgemm_f64_at(A, B, r, c)
    assert np.array_equal(c64, C64[r, c]) and np.array_equal(s, S[r, c])


def test_padded_rows_change_nothing():
    A, B = wl.make_pair(13, 17, 19, "normal", 8)
    Ap = wl.strided(A, 23)
    Bp = wl.strided(B, 21)
    assert Ap.strides[0] == 23 * 4 and Bp.strides[0] == 21 * 4
    assert np.array_equal(oracle.sgemm_f32(Ap, Bp), oracle.sgemm_f32(A, B))
    assert np.array_equal(oracle.sgemm_f64(Ap, Bp)[0], oracle.sgemm_f64(A, B)[0])


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.sgemm_f32(np.zeros((2, 3), np.float32), np.zeros((4, 2), np.float32))
    with pytest.raises(TypeError):
        oracle.sgemm_f32(np.zeros((2, 3), np.float64), np.zeros((3, 2), np.float32))


# ------------------------------------------------------------ acceptance measure

def test_normalized_error_measure():
    A, B = wl.make_pair(8, 9, 10, "normal", 2)
    C64, S = oracle.sgemm_f64(A, B)
    assert oracle.normalized_error(C64, C64, S) == 0.0
    planted = C64.copy()
    planted[3, 4] += 2.5e-6 * S[3, 4]
    assert oracle.normalized_error(planted, C64, S) == pytest.approx(2.5e-6, rel=1e-9)
    nan = C64.copy()
    nan[0, 0] = np.nan
    assert oracle.normalized_error(nan, C64, S) == float("inf")
    # Where S is zero the output must be exactly zero.
    Z64 = np.zeros((2, 2))
    assert oracle.normalized_error(np.zeros((2, 2)), Z64, Z64) == 0.0
    bad = np.zeros((2, 2))
    bad[1, 1] = 1e-30
    assert oracle.normalized_error(bad, Z64, Z64) == float("inf")


@pytest.mark.parametrize("dist,seed", [("normal", 0), ("uniform", 1)])
def test_float32_loop_within_north_bound(dist, seed):
    """The pages' own float loop meets the 1e-5 acceptance bound against the double twin."""
    A, B = wl.make_pair(64, 48, 1024, dist, seed)
    C32 = oracle.sgemm_f32(A, B)
    C64, S = oracle.sgemm_f64(A, B)
    err = oracle.normalized_error(C32, C64, S)
    assert 0.0 < err <= 1e-5


def test_transposed_operand_is_caught():
    """A planted transposition of B (in a CPU stand-in) fails the acceptance measure."""
    A, B = wl.make_pair(16, 16, 16, "normal", 6)
    C64, S = oracle.sgemm_f64(A, B)
    wrong = oracle.sgemm_f32(A, np.ascontiguousarray(B.T))
    assert oracle.normalized_error(wrong, C64, S) > 1e-2
