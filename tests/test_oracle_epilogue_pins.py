"""Pins of the oracle's fused epilogue act(alpha * op(A) op(B) + beta * C + bias).

The pages stop at the product; the epilogue is a bias vector and one of
three activations, each checked against facts that do not come from the
oracle's own formula: printed values of the standard normal distribution
function, exact values of the logistic function, an odd-part identity that
every correct implementation satisfies, integer closed forms for ReLU and the
bias, and the transposition identity that relates per-row and per-column
bias. A plausible slip -- a sign inside erf or exp, a dropped factor 1/2, a
bias indexed by the wrong coordinate, |bias| missing from the error scale --
fails at least one check.
"""

import math

import numpy as np
import pytest

import oracle


def _ints(shape, seed, lo=-5, hi=6):
    return np.random.default_rng(seed).integers(lo, hi, size=shape).astype(np.float32)


# Standard normal distribution function Phi(x) at a few points, as printed in
# tables of the normal probability integral (e.g. Abramowitz and Stegun,
# Handbook of Mathematical Functions, table 26.1), to 16 significant digits.
PHI_TABLE = {
    0.5: 0.6914624612740131,
    1.0: 0.8413447460685429,
    2.0: 0.9772498680518208,
    3.0: 0.9986501019683699,
}


@pytest.mark.parametrize("x,phi", sorted(PHI_TABLE.items()))
def test_gelu_matches_normal_table(x, phi):
    for sign in (1.0, -1.0):
        xs = sign * x
        expected = xs * (phi if sign > 0 else 1.0 - phi)  # Phi(-x) = 1 - Phi(x)
        c64, s = oracle.epilogue_f64(np.array([[xs]]), np.array([[1.0]]), act="gelu")
        assert abs(c64[0, 0] - expected) <= 4e-16 * max(1.0, abs(expected)), (xs, c64[0, 0], expected)
        assert s[0, 0] == 1.0


def test_silu_exact_points():
    # sigma(ln 3) = 3/4 and sigma(-ln 3) = 1/4, so SiLU(+-ln 3) = +-ln 3 * (3/4, 1/4).
    l3 = math.log(3.0)
    c64, _ = oracle.epilogue_f64(np.array([[l3, -l3, 0.0]]), np.ones((1, 3)), act="silu")
    assert abs(c64[0, 0] - 0.75 * l3) <= 1e-16 * 4
    assert abs(c64[0, 1] + 0.25 * l3) <= 1e-16 * 4
    assert c64[0, 2] == 0.0


@pytest.mark.parametrize("act", ["gelu", "silu"])
def test_odd_part_identity(act):
    # Phi(x) + Phi(-x) = 1 and sigma(x) + sigma(-x) = 1 give f(x) - f(-x) = x.
    x = np.random.default_rng(7).standard_normal(200) * 4
    pos, _ = oracle.epilogue_f64(x.reshape(1, -1), np.ones((1, 200)), act=act)
    neg, _ = oracle.epilogue_f64(-x.reshape(1, -1), np.ones((1, 200)), act=act)
    assert np.max(np.abs(pos - neg - x)) <= 1e-14


@pytest.mark.parametrize("act", ["gelu", "silu"])
def test_large_arguments(act):
    # Both tend to x for large positive x and to 0 for large negative x.
    c64, _ = oracle.epilogue_f64(np.array([[40.0, -40.0]]), np.ones((1, 2)), act=act)
    assert c64[0, 0] == 40.0
    assert abs(c64[0, 1]) < 1e-15


def test_relu_and_nan():
    vals = np.array([[-2.0, -0.0, 0.0, 3.5, np.nan, -np.inf, np.inf]])
    c64, _ = oracle.epilogue_f64(vals, np.ones_like(vals), act="relu")
    assert np.array_equal(c64[0, :4], [0.0, 0.0, 0.0, 3.5])
    assert math.isnan(c64[0, 4]) and c64[0, 5] == 0.0 and c64[0, 6] == math.inf


@pytest.mark.parametrize("bias_kind", ["col", "row"])
def test_bias_relu_integer_closed_form(bias_kind):
    M, N, K = 7, 11, 13  # M != N so a bias indexed by the wrong coordinate fails
    A, B, C = _ints((M, K), 1), _ints((K, N), 2), _ints((M, N), 3)
    bias = _ints((N,) if bias_kind == "col" else (M,), 4, -40, 41)
    C64, S = oracle.gemm_f64(A, B, alpha=2.0, beta=-1.0, C_in=C)
    out, S2 = oracle.epilogue_f64(C64, S, bias=bias, bias_kind=bias_kind, act="relu")
    pre = 2 * (A.astype(np.int64) @ B.astype(np.int64)) - C.astype(np.int64)
    b = bias.astype(np.int64)
    pre = pre + (b[None, :] if bias_kind == "col" else b[:, None])
    assert np.array_equal(out, np.maximum(pre, 0).astype(np.float64))
    s_exact = 2 * (np.abs(A).astype(np.int64) @ np.abs(B).astype(np.int64)) + np.abs(C).astype(np.int64)
    s_exact = s_exact + (np.abs(b)[None, :] if bias_kind == "col" else np.abs(b)[:, None])
    assert np.array_equal(S2, s_exact.astype(np.float64))


def test_row_bias_is_column_bias_of_the_transpose():
    # (A B + b 1^T)^T = B^T A^T + 1 b^T: a per-row bias of C is a per-column
    # bias of C^T, element for element.
    rng = np.random.default_rng(9)
    M, N, K = 6, 10, 9
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    b = rng.standard_normal(M).astype(np.float32)
    C64, S = oracle.gemm_f64(A, B)
    out, s = oracle.epilogue_f64(C64, S, bias=b, bias_kind="row", act="gelu")
    Ct, St = oracle.gemm_f64(B, A, transA=True, transB=True)
    out_t, s_t = oracle.epilogue_f64(Ct, St, bias=b, bias_kind="col", act="gelu")
    assert np.array_equal(out, out_t.T) and np.array_equal(s, s_t.T)


def test_sampled_matches_full():
    rng = np.random.default_rng(11)
    M, N = 9, 14
    c64 = rng.standard_normal((M, N))
    s = np.abs(rng.standard_normal((M, N)))
    bias = rng.standard_normal(N).astype(np.float32)
    full, sfull = oracle.epilogue_f64(c64, s, bias=bias, bias_kind="col", act="silu")
    r = rng.integers(0, M, 40)
    c = rng.integers(0, N, 40)
    part, spart = oracle.epilogue_f64(c64[r, c], s[r, c], bias=bias, bias_kind="col", act="silu",
                                      rows=r, cols=c, shape=(M, N))
    assert np.array_equal(part, full[r, c]) and np.array_equal(spart, sfull[r, c])


def test_no_epilogue_is_identity():
    c64 = np.random.default_rng(2).standard_normal((4, 5))
    s = np.ones((4, 5))
    out, s2 = oracle.epilogue_f64(c64, s)
    assert np.array_equal(out, c64) and np.array_equal(s2, s)


def test_rejects_bad_arguments():
    c64, s = np.zeros((3, 4)), np.zeros((3, 4))
    with pytest.raises(ValueError):
        oracle.epilogue_f64(c64, s, bias=np.zeros(3, np.float32), bias_kind="col")  # needs N = 4
    with pytest.raises(ValueError):
        oracle.epilogue_f64(c64, s, bias=np.zeros(4, np.float32), bias_kind="row")  # needs M = 3
    with pytest.raises(KeyError):
        oracle.epilogue_f64(c64, s, act="tanh")
