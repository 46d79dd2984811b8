"""sgemm_f32_noalloc: sgemm_f32 with the aligned copies of unaligned operands
in one fixed per-device buffer instead of pool memory. Compared with
sgemm_f32 (and the oracle) on two calls in a row; oversize products are
rejected before anything runs. This file is collected last and sets every
setting it relies on, so it passes alone and after the other tests."""

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_major_gb300 import workloads as wl
from tests.gpu_harness import TOL, device_matrix, outside_box_intact

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from dense_fp32_matrix_major_gb300 import sgemm

    sgemm.set_variant("auto")
    sgemm.set_tuning(sgemm.SGEMM_TUNE_TF32X3_KERNEL, 0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_STREAM_K, 0)
    yield sgemm
    sgemm.set_variant("auto")
    sgemm.set_tuning(sgemm.SGEMM_TUNE_TF32X3_KERNEL, 0)


def _run(fn, A, B, lda, ldb, ldc):
    """One call of `fn` (a raw C-ABI wrapper) on padded device copies; returns
    (status, C box, flat C buffer)."""
    import torch

    M, K = A.shape
    N = B.shape[1]
    fa, vA = device_matrix(A, lda)
    fb, vB = device_matrix(B, ldb)
    fc, vC = device_matrix(np.full((M, N), np.nan, np.float32), ldc)
    rc = fn(M, N, K, vA.data_ptr(), lda, vB.data_ptr(), ldb, vC.data_ptr(), ldc,
            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return rc, vC.cpu().numpy(), fc.cpu().numpy()


CASES = [
    # (M, N, K, lda, ldb, ldc, tensor-core kernel mode): rows of 1537 and 2049
    # floats, large enough for the copies; a small unaligned product with the
    # copies forced (mode 5); aligned rows (no copies); a small product below
    # the copy threshold (per-thread loads).
    (1023, 2049, 1537, 1537, 2049, 2049, 0),
    (300, 270, 301, 302, 271, 271, 5),
    (512, 768, 1024, 1024, 768, 768, 0),
    (200, 130, 257, 258, 131, 133, 0),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}-m{c[6]}" for c in CASES])
def test_matches_sgemm_f32_on_two_calls_in_a_row(lib, case):
    M, N, K, lda, ldb, ldc, mode = case
    lib.set_tuning(lib.SGEMM_TUNE_TF32X3_KERNEL, mode)
    try:
        A, B = wl.make_pair(M, N, K, "normal", M + N)
        rc, C_ref, _ = _run(lib.sgemm_f32_raw, A, B, lda, ldb, ldc)
        assert rc == 0
        C64, S = oracle.sgemm_f64(A, B) if M * N * K <= 2_000_000 else oracle.sgemm_f64_rows(A, B)
        assert oracle.normalized_error(C_ref, C64, S) <= TOL
        for call in range(2):
            rc, C, flat = _run(lib.sgemm_f32_noalloc_raw, A, B, lda, ldb, ldc)
            assert rc == 0, call
            assert outside_box_intact(flat, M, N, ldc, 0)
            # Within the tolerance of sgemm_f32's result and of the oracle.
            assert np.max(np.abs(C.astype(np.float64) - C_ref) / np.maximum(S, 1e-30)) <= TOL, call
            assert oracle.normalized_error(C, C64, S) <= TOL, call
    finally:
        lib.set_tuning(lib.SGEMM_TUNE_TF32X3_KERNEL, 0)


def test_rejects_products_whose_copies_do_not_fit(lib):
    """Rows of 4095 and 521 floats: the copies (4095 x 4096 and 4095 x 524
    floats, 72 MiB) exceed the fixed buffer, so the call fails with
    SGEMM_ERR_SCRATCH and C is not touched; sgemm_f32 runs the same product."""
    import torch

    M, N, K = 4095, 521, 4095
    assert 4 * (M * ((K + 3) // 4 * 4) + K * ((N + 3) // 4 * 4)) > lib.SGEMM_NOALLOC_SCRATCH_BYTES
    A = torch.randn(M, K, device="cuda")
    B = torch.randn(K, N, device="cuda")
    C = torch.full((M, N), float("nan"), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.sgemm_f32_noalloc_raw(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N, stream)
    torch.cuda.synchronize()
    assert rc == lib.SGEMM_ERR_SCRATCH
    assert "scratch" in lib.strerror(rc)
    assert torch.isnan(C).all()
    assert lib.sgemm_f32_raw(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N, stream) == 0
    torch.cuda.synchronize()
    assert not torch.isnan(C).any()
