"""GPU parity of the general form C = alpha * op(A) * op(B) + beta * C
(sgemm_f32_ex) against the oracle's general form."""

import itertools

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_major_gb300 import workloads as wl
from tests.gpu_harness import TOL, outside_box_intact, run_gemm_ex

pytestmark = pytest.mark.gpu

FORMS = [(0, 0), (1, 0), (0, 1), (1, 1)]
SCALES = [(1.0, 0.0), (2.5, -1.5), (-1.0, 1.0), (0.75, 0.0), (1.0, 1.0)]


@pytest.fixture(scope="module")
def lib():
    from dense_fp32_matrix_major_gb300 import sgemm

    yield sgemm
    sgemm.set_variant(0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_FFMA_TILE, 0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_STREAM_K, 0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_TF32X3_KERNEL, 0)


def _stored(M, N, K, transA, transB, dist, seed):
    A, B = wl.make_pair(M, N, K, dist, seed)
    As = np.ascontiguousarray(A.T) if transA else A
    Bs = np.ascontiguousarray(B.T) if transB else B
    return As, Bs


def _check(lib, As, Bs, tA, tB, alpha, beta, C0, **kw):
    C, flat, rc = run_gemm_ex(As, Bs, transA=tA, transB=tB, alpha=alpha, beta=beta,
                              C_init=C0 if beta else None, **kw)
    assert rc == 0  # every form at any alignment, on either variant
    M, N = C.shape
    ldc = kw.get("ldc") or max(N, 1)
    assert outside_box_intact(flat, M, N, ldc, kw.get("offsets", (0, 0, 0))[2])
    C64, S = oracle.gemm_f64(As, Bs, transA=bool(tA), transB=bool(tB), alpha=alpha, beta=beta,
                             C_in=C0 if beta else None)
    err = oracle.normalized_error(C, C64, S)
    assert err <= TOL, (tA, tB, alpha, beta, err)


@pytest.mark.parametrize("variant,tile,sk", [("auto", 0, 0), ("ffma", 1, 3), ("ffma", 3, 0), ("ffma", 2, 1),
                                             ("tf32x3", 0, 0), ("tf32x3", 0, 3)])
@pytest.mark.parametrize("tA,tB", FORMS)
def test_forms_and_scales(lib, variant, tile, sk, tA, tB):
    lib.set_variant(variant)
    lib.set_tuning(lib.SGEMM_TUNE_FFMA_TILE, tile)
    lib.set_tuning(lib.SGEMM_TUNE_STREAM_K, sk)
    for (M, N, K) in [(1, 1, 1), (5, 3, 7), (129, 257, 47), (300, 200, 513), (64, 300, 1000),
                      (128, 256, 64), (260, 516, 300)]:
        As, Bs = _stored(M, N, K, tA, tB, "normal", M + N + K)
        C0 = np.random.default_rng(K).standard_normal((M, N)).astype(np.float32)
        for alpha, beta in SCALES:
            _check(lib, As, Bs, tA, tB, alpha, beta, C0)


@pytest.mark.parametrize("tc,sk", [(4, 0), (4, 1), (4, 3), (3, 0)])
@pytest.mark.parametrize("tA,tB", FORMS)
def test_forms_on_each_tensor_core_kernel(lib, tc, sk, tA, tB):
    """Every operand form on the SM-pair kernel (4) and the single-SM
    tensor-memory kernel (3), under each schedule; 16-byte aligned rows."""
    lib.set_variant("tf32x3")
    lib.set_tuning(lib.SGEMM_TUNE_TF32X3_KERNEL, tc)
    lib.set_tuning(lib.SGEMM_TUNE_STREAM_K, sk)
    for (M, N, K) in [(129, 257, 48), (300, 200, 516), (64, 300, 1000), (260, 516, 300), (512, 768, 2048)]:
        As, Bs = _stored(M, N, K, tA, tB, "normal", M + 2 * N + K)
        C0 = np.random.default_rng(K).standard_normal((M, N)).astype(np.float32)
        for alpha, beta in [(1.0, 0.0), (-0.5, 2.0)]:
            _check(lib, As, Bs, tA, tB, alpha, beta, C0)
    assert lib.get_tuning(lib.SGEMM_TUNE_LAST_TC_KERNEL) == tc
    lib.set_tuning(lib.SGEMM_TUNE_TF32X3_KERNEL, 0)
    lib.set_tuning(lib.SGEMM_TUNE_STREAM_K, 0)


@pytest.mark.parametrize("variant", ["ffma", "tf32x3"])
@pytest.mark.parametrize("tA,tB", FORMS)
def test_integer_forms_bit_exact(lib, variant, tA, tB):
    lib.set_variant(variant)
    for (M, N, K) in [(256, 132, 1000), (64, 300, 4096)]:
        As, Bs = _stored(M, N, K, tA, tB, "int4", K)
        C0 = np.random.default_rng(1).integers(-9, 10, (M, N)).astype(np.float32)
        C, flat, rc = run_gemm_ex(As, Bs, transA=tA, transB=tB, alpha=3.0, beta=-2.0, C_init=C0)
        assert rc == 0
        A = As.T if tA else As
        B = Bs.T if tB else Bs
        exact = 3 * (A.astype(np.int64) @ B.astype(np.int64)) - 2 * C0.astype(np.int64)
        assert np.array_equal(C, exact.astype(np.float32))


@pytest.mark.parametrize("tA,tB", FORMS)
def test_strided_unaligned_forms(lib, tA, tB):
    lib.set_variant("auto")
    M, N, K = 150, 270, 90
    As, Bs = _stored(M, N, K, tA, tB, "uniform", 8)
    C0 = np.random.default_rng(2).standard_normal((M, N)).astype(np.float32)
    for kw in [dict(lda=As.shape[1] + 3, ldb=Bs.shape[1] + 5, ldc=N + 7, offsets=(1, 3, 2)),
               dict(lda=As.shape[1] + 4, ldb=Bs.shape[1] + 4, ldc=N + 4, offsets=(0, 0, 0))]:
        _check(lib, As, Bs, tA, tB, 1.5, -0.5, C0, **kw)


def test_beta_zero_ignores_nan_c_and_alpha_zero(lib):
    for variant in ("ffma", "tf32x3"):
        lib.set_variant(variant)
        As, Bs = _stored(200, 300, 64, 0, 0, "normal", 3)
        C, flat, rc = run_gemm_ex(As, Bs, alpha=1.0, beta=0.0)  # C starts as NaN
        assert rc == 0 and np.all(np.isfinite(C))
        C0 = np.random.default_rng(4).standard_normal((200, 300)).astype(np.float32)
        C, flat, rc = run_gemm_ex(As, Bs, alpha=0.0, beta=-1.25, C_init=C0)
        assert rc == 0 and np.array_equal(C, np.float32(-1.25) * C0)
        C, flat, rc = run_gemm_ex(As, Bs, alpha=0.0, beta=0.0)
        assert rc == 0 and np.all(C == 0)


@pytest.mark.parametrize("tA,tB", FORMS)
def test_forced_tensor_cores_on_unaligned_transposes(lib, tA, tB):
    """Forced tensor cores serve every form with rows that are not 16-byte
    aligned (the transposed forms on the SM-pair kernel's cp.async loaders),
    at a size that spans several pair tiles and a ragged edge, with alpha and
    beta."""
    lib.set_variant("tf32x3")
    M, N, K = 300, 270, 301
    As, Bs = _stored(M, N, K, tA, tB, "uniform", 5)
    C0 = np.random.default_rng(6).standard_normal((M, N)).astype(np.float32)
    _check(lib, As, Bs, tA, tB, 0.75, -1.5, C0, lda=As.shape[1] + 1, ldb=Bs.shape[1] + 3, ldc=N + 1,
           offsets=(1, 2, 3))
    if tA or tB:  # the per-thread-load kernel serves op(A) = A, op(B) = B only
        assert lib.get_tuning(lib.SGEMM_TUNE_LAST_TC_KERNEL) == 4


@pytest.mark.parametrize("sk", [0, 3])
@pytest.mark.parametrize("tA,tB", FORMS)
def test_forced_pair_kernel_on_tiny_and_ragged_shapes(lib, sk, tA, tB):
    """The SM-pair kernel forced on products far smaller than its 256 x 128
    tile (a single row or column of C, M or N below one tile) with K long
    enough for several fold intervals and, under stream-K, several units per
    tile: results match the oracle and nothing outside C's box is written, on
    aligned and unaligned rows."""
    lib.set_variant("tf32x3")
    lib.set_tuning(lib.SGEMM_TUNE_TF32X3_KERNEL, 4)
    lib.set_tuning(lib.SGEMM_TUNE_STREAM_K, sk)
    try:
        for i, (M, N, K) in enumerate([(1, 7, 1100), (129, 3, 1100), (3, 129, 700), (1, 1, 2049),
                                       (17, 300, 2049), (257, 129, 600), (8, 8, 1024)]):
            As, Bs = _stored(M, N, K, tA, tB, "normal", 40 + i)
            C0 = np.random.default_rng(i).standard_normal((M, N)).astype(np.float32)
            _check(lib, As, Bs, tA, tB, 1.25, -0.5, C0)
            assert lib.get_tuning(lib.SGEMM_TUNE_LAST_TC_KERNEL) == 4, (M, N, K)
            _check(lib, As, Bs, tA, tB, 1.0, 0.0, C0, lda=As.shape[1] + 1, ldb=Bs.shape[1] + 1, ldc=N + 2,
                   offsets=(1, 1, 1))
            assert lib.get_tuning(lib.SGEMM_TUNE_LAST_TC_KERNEL) == 4, (M, N, K)
    finally:
        lib.set_tuning(lib.SGEMM_TUNE_TF32X3_KERNEL, 0)
        lib.set_tuning(lib.SGEMM_TUNE_STREAM_K, 0)


@pytest.mark.parametrize("tA,tB", FORMS)
def test_headline_shape_forms(lib, tA, tB):
    lib.set_variant("auto")
    w = wl.C5_HEAD
    As, Bs = _stored(w.M, w.N, w.K, tA, tB, "normal", 4)
    C0 = np.random.default_rng(5).standard_normal((w.M, w.N)).astype(np.float32)
    C, flat, rc = run_gemm_ex(As, Bs, transA=tA, transB=tB, alpha=0.5, beta=2.0, C_init=C0)
    assert rc == 0
    r, c = wl.sample_positions(w.M, w.N, 3000, seed=tA * 2 + tB)
    c64, s = oracle.gemm_f64_at(As, Bs, r, c, transA=bool(tA), transB=bool(tB), alpha=0.5, beta=2.0,
                                C_in=C0)
    assert oracle.normalized_error(C[r, c], c64, s) <= TOL
