"""Operands whose rows TMA cannot address (row strides or base addresses not
16-byte aligned, "CUDA内存优化入门：从Naive到Tiled矩阵乘法" section 六's
sizes that are not multiples of the tile): the tensor-core path copies them
into aligned scratch rows and runs the TMA kernels (automatically from 1.25 * 2^30
multiply-adds on; here forced at small sizes with tensor-core kernel mode 5,
and automatically at one large size). Every output is compared with the
oracle, the inputs are left untouched and nothing outside C's box is
written."""

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_major_gb300 import workloads as wl
from tests.gpu_harness import (TOL, batched_outside_intact, device_matrix, outside_box_intact, run_batched,
                               run_gemm_ex)

pytestmark = pytest.mark.gpu

FORMS = [(0, 0), (1, 0), (0, 1), (1, 1)]


@pytest.fixture(scope="module")
def lib():
    from dense_fp32_matrix_major_gb300 import sgemm

    sgemm.set_variant("tf32x3")
    sgemm.set_tuning(sgemm.SGEMM_TUNE_TF32X3_KERNEL, 5)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_STREAM_K, 0)
    yield sgemm
    sgemm.set_variant(0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_TF32X3_KERNEL, 0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_STREAM_K, 0)


def _stored(M, N, K, tA, tB, seed, dist="normal"):
    A, B = wl.make_pair(M, N, K, dist, seed)
    return (np.ascontiguousarray(A.T) if tA else A), (np.ascontiguousarray(B.T) if tB else B)


@pytest.mark.parametrize("sk", [0, 3])
@pytest.mark.parametrize("tA,tB", FORMS)
def test_unaligned_rows_every_form(lib, sk, tA, tB):
    lib.set_tuning(lib.SGEMM_TUNE_STREAM_K, sk)
    for (M, N, K), kw in [((300, 270, 301), dict(lda=None, ldb=None, ldc=None, offsets=(1, 2, 3))),
                          ((257, 513, 515), dict(lda=None, ldb=None, ldc=None, offsets=(0, 0, 0))),
                          ((512, 512, 512), dict(pad=1, offsets=(0, 0, 1)))]:
        As, Bs = _stored(M, N, K, tA, tB, M + K)
        pad = kw.pop("pad", 0)
        if pad:
            kw.update(lda=As.shape[1] + pad, ldb=Bs.shape[1] + pad, ldc=N + 2)
        C0 = np.random.default_rng(K).standard_normal((M, N)).astype(np.float32)
        C, flat, rc = run_gemm_ex(As, Bs, transA=tA, transB=tB, alpha=1.5, beta=-0.5, C_init=C0, **kw)
        assert rc == 0
        assert lib.get_tuning(lib.SGEMM_TUNE_LAST_TC_KERNEL) == 4, (M, N, K)
        ldc = kw.get("ldc") or N
        assert outside_box_intact(flat, M, N, ldc, kw["offsets"][2])
        C64, S = oracle.gemm_f64(As, Bs, transA=bool(tA), transB=bool(tB), alpha=1.5, beta=-0.5, C_in=C0)
        assert oracle.normalized_error(C, C64, S) <= TOL, (M, N, K)


def test_only_one_operand_copied_and_inputs_untouched(lib):
    """A unaligned, B aligned (and the reverse): the result is right and the
    caller's A and B buffers (with their padding) are bit-for-bit unchanged."""
    import torch
    from dense_fp32_matrix_major_gb300 import sgemm

    M, N, K = 384, 640, 333
    A, B = wl.make_pair(M, N, K, "uniform01", 9)
    for lda, ldb in [(K + 1, N), (K + 3, N + 1), (336, N + 2)]:
        fa, vA = device_matrix(A, lda, 0)
        fb, vB = device_matrix(B, ldb, 0)
        before_a, before_b = fa.cpu().numpy().copy(), fb.cpu().numpy().copy()
        C = torch.full((M, N), float("nan"), device="cuda")
        rc = sgemm.sgemm_f32_raw(M, N, K, vA.data_ptr(), lda, vB.data_ptr(), ldb, C.data_ptr(), N,
                                 torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert rc == 0
        assert sgemm.get_tuning(sgemm.SGEMM_TUNE_LAST_TC_KERNEL) == 4
        assert np.array_equal(fa.cpu().numpy().view(np.uint32), before_a.view(np.uint32))
        assert np.array_equal(fb.cpu().numpy().view(np.uint32), before_b.view(np.uint32))
        C64, S = oracle.sgemm_f64(A, B)
        assert oracle.normalized_error(C.cpu().numpy(), C64, S) <= TOL, (lda, ldb)


@pytest.mark.parametrize("share", ["none", "a", "b"])
def test_unaligned_batch(lib, share):
    """A strided batch whose rows (K = 101 floats) and item strides are not
    16-byte aligned; stride 0 shares an operand."""
    batch, M, N, K = 9, 96, 200, 101
    rng = np.random.default_rng(3)
    As = [rng.standard_normal((M, K)).astype(np.float32) for _ in range(1 if share == "a" else batch)]
    Bs = [rng.standard_normal((K, N)).astype(np.float32) for _ in range(1 if share == "b" else batch)]
    Af = As * batch if share == "a" else As
    Bf = Bs * batch if share == "b" else Bs
    out, flat, rc, sC = run_batched(Af, Bf, strideA=None if share == "a" else M * K + 1,
                                    strideB=None if share == "b" else K * N + 3, share_a=share == "a",
                                    share_b=share == "b")
    assert rc == 0
    assert lib.get_tuning(lib.SGEMM_TUNE_LAST_TC_KERNEL) in (3, 4)  # a TMA kernel on the copies
    assert batched_outside_intact(flat, batch, M, N, sC)
    for b in range(batch):
        C64, S = oracle.sgemm_f64(Af[b], Bf[b])
        assert oracle.normalized_error(out[b], C64, S) <= TOL, b


def test_repeated_calls_reuse_pool(lib):
    """Many calls of different sizes in a row (scratch freed behind each on
    the stream and taken again from the pool) stay correct."""
    import torch
    from dense_fp32_matrix_major_gb300 import sgemm

    cases = [(300, 270, 301), (1023, 2049, 1537), (129, 700, 999), (300, 270, 301)]
    inputs = []
    for i, (M, N, K) in enumerate(cases):
        A, B = wl.make_pair(M, N, K, "normal", 70 + i)
        fa, vA = device_matrix(A, K + 1, 0)
        fb, vB = device_matrix(B, N + 1, 0)
        C = torch.full((M, N), float("nan"), device="cuda")
        inputs.append((A, B, fa, vA, fb, vB, C))
    stream = torch.cuda.current_stream().cuda_stream
    for rep in range(3):
        for (M, N, K), (A, B, fa, vA, fb, vB, C) in zip(cases, inputs):
            assert sgemm.sgemm_f32_raw(M, N, K, vA.data_ptr(), K + 1, vB.data_ptr(), N + 1, C.data_ptr(), N,
                                       stream) == 0
    torch.cuda.synchronize()
    for (M, N, K), (A, B, fa, vA, fb, vB, C) in zip(cases, inputs):
        C64, S = oracle.sgemm_f64_rows(A, B)
        assert oracle.normalized_error(C.cpu().numpy(), C64, S) <= TOL, (M, N, K)


def test_automatic_copy_at_large_size(lib):
    """AUTO takes the copies by itself at the ragged benchmark shape (rows of
    1537 and 2049 floats), every output compared."""
    import torch
    from dense_fp32_matrix_major_gb300 import sgemm

    sgemm.set_variant("auto")
    sgemm.set_tuning(sgemm.SGEMM_TUNE_TF32X3_KERNEL, 0)
    try:
        w = wl.C3_RAGGED
        A, B = wl.make_inputs(w)
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        C = torch.full((w.M, w.N), float("nan"), device="cuda")
        rc = sgemm.sgemm_f32_raw(w.M, w.N, w.K, dA.data_ptr(), w.K, dB.data_ptr(), w.N, C.data_ptr(), w.N,
                                 torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert rc == 0
        assert sgemm.get_tuning(sgemm.SGEMM_TUNE_LAST_TC_KERNEL) == 4
        assert sgemm.last_launch_count() >= 2  # the copies, then the product
        C64, S = oracle.sgemm_f64_rows(A, B)
        assert oracle.normalized_error(C.cpu().numpy(), C64, S) <= TOL
    finally:
        sgemm.set_variant("tf32x3")
        sgemm.set_tuning(sgemm.SGEMM_TUNE_TF32X3_KERNEL, 5)


@pytest.mark.parametrize("tA,tB", FORMS)
def test_unaligned_rows_fused_epilogue(lib, tA, tB):
    """The fused epilogue (per-column bias + ReLU, and per-row bias + GELU with
    beta) on the aligned copies, every form."""
    from tests.gpu_harness import run_fused

    M, N, K = 300, 270, 301
    As, Bs = _stored(M, N, K, tA, tB, 17)
    rng = np.random.default_rng(11)
    C0 = rng.standard_normal((M, N)).astype(np.float32)
    for bias_kind, act, kind_name, act_name, beta in [(1, 1, "col", "relu", 0.0), (2, 2, "row", "gelu", 0.5)]:
        bias = rng.standard_normal(N if bias_kind == 1 else M).astype(np.float32)
        C, flat, rc = run_fused(As, Bs, bias=bias, bias_kind=bias_kind, act=act, transA=tA, transB=tB, alpha=1.25,
                                beta=beta, C_init=C0 if beta else None, lda=As.shape[1] + 1, ldb=Bs.shape[1] + 3,
                                ldc=N + 1)
        assert rc == 0
        assert lib.get_tuning(lib.SGEMM_TUNE_LAST_TC_KERNEL) == 4
        assert outside_box_intact(flat, M, N, N + 1, 0)
        C64, S = oracle.gemm_f64(As, Bs, transA=bool(tA), transB=bool(tB), alpha=1.25, beta=beta,
                                 C_in=C0 if beta else None)
        E64, ES = oracle.epilogue_f64(C64, S, bias=bias, bias_kind=kind_name, act=act_name)
        assert oracle.normalized_error(C, E64, ES) <= TOL, (bias_kind, act)


@pytest.mark.parametrize("K", [1537, 4097])
def test_unaligned_rows_same_sign_accuracy(lib, K):
    """U[0,1] inputs (the pages' rand() / RAND_MAX) through the copies: the
    copy is exact, so the bounded accumulation chains keep the bound."""
    import torch
    from dense_fp32_matrix_major_gb300 import sgemm

    M, N = 300, 517
    A, B = wl.make_mixed(M, N, K, "uniform01", "uniform01", K)
    fa, vA = device_matrix(A, K + 1, 0)
    fb, vB = device_matrix(B, N + 3, 0)
    C = torch.full((M, N), float("nan"), device="cuda")
    rc = sgemm.sgemm_f32_raw(M, N, K, vA.data_ptr(), K + 1, vB.data_ptr(), N + 3, C.data_ptr(), N,
                             torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    assert sgemm.get_tuning(sgemm.SGEMM_TUNE_LAST_TC_KERNEL) == 4
    C64, S = oracle.sgemm_f64_rows(A, B)
    assert oracle.normalized_error(C.cpu().numpy(), C64, S) <= TOL
