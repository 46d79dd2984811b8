"""Non-finite inputs on every kernel: the positions and kinds of +inf, -inf
and NaN in C match the oracle's IEEE product exactly, and every finite
output stays within the parity tolerance.

IEEE rules the planted values exercise (the reading of the operation as a
plain sum of products in fp32): inf * finite = +-inf by sign, inf * 0 = NaN,
inf + (-inf) = NaN, NaN anywhere in a sum gives NaN. The three-term TF32
split would turn an infinity into NaN (its low part is inf - inf); the
kernels recompute such outputs with IEEE arithmetic, so both variants follow
the same rules.
"""

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_major_gb300 import workloads as wl
from tests.gpu_harness import TOL, outside_box_intact, run_fused, run_gemm_ex

FORMS = [(0, 0), (1, 0), (0, 1), (1, 1)]
# (variant, ffma tile, stream-K mode, tensor-core kernel); kernels: 1 = per-thread
# loads, 2 = TMA, 3 = TMA with A in tensor memory, 4 = SM pairs.
SETTINGS = [
    ("auto", 0, 0, 0), ("ffma", 1, 0, 0), ("ffma", 3, 3, 0),
    ("tf32x3", 0, 0, 1), ("tf32x3", 0, 3, 1), ("tf32x3", 0, 0, 2), ("tf32x3", 0, 3, 2),
    ("tf32x3", 0, 0, 3), ("tf32x3", 0, 3, 3), ("tf32x3", 0, 0, 4), ("tf32x3", 0, 1, 4), ("tf32x3", 0, 3, 4),
]
IDS = [f"{s[0]}-t{s[1]}-sk{s[2]}-k{s[3]}" for s in SETTINGS]
# Several tiles and fold intervals; a K that leaves a ragged k-block; an
# aligned shape for the TMA kernels; a deep K split across units.
SHAPES = [(130, 260, 40), (300, 270, 1537), (512, 512, 1024), (256, 384, 4096)]


@pytest.fixture(scope="module")
def lib():
    from dense_fp32_matrix_major_gb300 import sgemm

    yield sgemm
    sgemm.set_variant(0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_FFMA_TILE, 0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_STREAM_K, 0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_TF32X3_KERNEL, 0)


def _apply(lib, setting):
    variant, tile, sk, tc = setting
    lib.set_variant(variant)
    lib.set_tuning(lib.SGEMM_TUNE_FFMA_TILE, tile)
    lib.set_tuning(lib.SGEMM_TUNE_STREAM_K, sk)
    lib.set_tuning(lib.SGEMM_TUNE_TF32X3_KERNEL, tc)


def planted(M, N, K, seed):
    """op(A) (M x K) and op(B) (K x N), N(0,1) with infinities, NaN and zeros
    planted so that every IEEE rule above decides some outputs, in the first,
    a middle and the last k-block."""
    A, B = wl.make_pair(M, N, K, "normal", seed)
    B[0, ::5] = 0.0            # inf * 0 in row 3
    B[1, ::7] = 0.0
    A[::11, K - 2] = 0.0       # 0 * -inf in column N - 1
    A[3, 0] = np.inf           # row 3: +-inf by the sign of B[0, j], NaN where B[0, j] == 0
    A[M - 2, K - 1] = -np.inf  # a row whose infinity sits in the last k-block
    A[M // 2, 1] = np.inf      # two infinities: NaN where B[1, j], B[K // 2, j] differ in sign
    A[M // 2, K // 2] = np.inf
    A[7, K // 3] = np.nan      # row 7 all NaN
    B[K - 2, N - 1] = -np.inf  # column N - 1
    B[0, 5] = np.inf           # column 5, and C[3, 5] = inf * inf
    B[K // 3, 9] = np.nan      # column 9 all NaN
    return A, B


def kinds(C):
    """0 finite, 1 +inf, 2 -inf, 3 NaN."""
    C = np.asarray(C)
    return np.select([np.isnan(C), np.isposinf(C), np.isneginf(C)], [3, 1, 2], 0)


def check_against_oracle(C, C64, S, what):
    got, want = kinds(C), kinds(C64)
    bad = np.argwhere(got != want)
    assert bad.size == 0, (what, bad[:5].tolist(), [(C[i, j], C64[i, j]) for i, j in bad[:5]])
    fin = (want == 0) & np.isfinite(S)
    assert np.count_nonzero(want) > 0 and np.count_nonzero(fin) > 0
    err = np.max(np.abs(C[fin].astype(np.float64) - C64[fin]) / np.maximum(S[fin], 1e-300))
    assert err <= TOL, (what, err)


def test_planted_values_cover_every_rule():
    """The fixture itself: the oracle sees +inf, -inf, NaN from inf * 0, NaN
    from inf - inf and NaN from a NaN input."""
    M, N, K = 130, 260, 40
    A, B = planted(M, N, K, 1)
    C64, _ = oracle.gemm_f64(A, B)
    k = kinds(C64)
    assert np.any(k[3] == 1) and np.any(k[3] == 2) and np.isnan(C64[3, 0])  # B[0, 0] == 0
    assert np.all(np.isnan(C64[7])) and np.all(np.isnan(C64[:, 9]))
    assert C64[3, 5] == np.inf
    opp = (B[1] * B[K // 2] < 0)
    assert np.all(np.isnan(C64[M // 2][opp]))
    assert np.isnan(C64[0, N - 1])  # A[0, K - 2] == 0


@pytest.mark.gpu
@pytest.mark.parametrize("setting", SETTINGS, ids=IDS)
@pytest.mark.parametrize("shape", SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in SHAPES])
def test_nonfinite_match_oracle(lib, setting, shape):
    _apply(lib, setting)
    M, N, K = shape
    A, B = planted(M, N, K, M + N + K)
    C, flat, rc = run_gemm_ex(A, B)
    assert rc == 0
    assert outside_box_intact(flat, M, N, N, 0)
    C64, S = oracle.gemm_f64(A, B)
    check_against_oracle(C, C64, S, (setting, shape))


@pytest.mark.gpu
@pytest.mark.parametrize("setting", [("auto", 0, 0, 0), ("ffma", 2, 0, 0), ("tf32x3", 0, 0, 3),
                                     ("tf32x3", 0, 0, 4), ("tf32x3", 0, 3, 4)],
                         ids=["auto", "ffma", "k3", "k4", "k4-sk3"])
@pytest.mark.parametrize("tA,tB", FORMS)
def test_nonfinite_transposed_forms(lib, setting, tA, tB):
    _apply(lib, setting)
    for (M, N, K) in [(300, 270, 1537), (512, 512, 1024)]:
        A, B = planted(M, N, K, 7 * M + K)
        As = np.ascontiguousarray(A.T) if tA else A
        Bs = np.ascontiguousarray(B.T) if tB else B
        C, flat, rc = run_gemm_ex(As, Bs, transA=tA, transB=tB)
        assert rc == 0
        C64, S = oracle.gemm_f64(As, Bs, transA=bool(tA), transB=bool(tB))
        check_against_oracle(C, C64, S, (setting, tA, tB, M, N, K))


@pytest.mark.gpu
@pytest.mark.parametrize("setting", [("auto", 0, 0, 0), ("tf32x3", 0, 0, 4), ("tf32x3", 0, 3, 4),
                                     ("tf32x3", 0, 0, 1)], ids=["auto", "k4", "k4-sk3", "k1"])
def test_nonfinite_fused_relu_bias(lib, setting):
    """Through the fused epilogue: ReLU keeps +inf and NaN and maps -inf to 0;
    a per-column bias is added before it."""
    _apply(lib, setting)
    M, N, K = 512, 512, 1024
    A, B = planted(M, N, K, 99)
    bias = np.random.default_rng(5).standard_normal(N).astype(np.float32)
    C, flat, rc = run_fused(A, B, bias=bias, bias_kind=1, act=1)
    assert rc == 0
    C64, S = oracle.gemm_f64(A, B)
    E64, ES = oracle.epilogue_f64(C64, S, bias=bias, bias_kind="col", act="relu")
    check_against_oracle(C, E64, ES, setting)
