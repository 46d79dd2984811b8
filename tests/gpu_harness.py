"""Helpers for the GPU parity tests: place matrices in device memory with
chosen row strides and pointer offsets, guard bands around C, and compare
with the CPU oracle."""

from __future__ import annotations

import numpy as np

import oracle

CANARY = np.float32(7777.25)  # every float of C's buffer outside the M x N box
GUARD = 67                    # floats of guard band after each buffer
TOL = 1e-5                    # max |C - C64| / sum_k |A||B|


def device_matrix(values: np.ndarray, ld: int | None = None, offset: int = 0, fill=CANARY):
    """(flat, view): a flat CUDA buffer and a rows x cols strided view into it.

    The view starts ``offset`` floats into the buffer, rows sit ``ld`` floats
    apart; everything else in the buffer holds ``fill``.
    """
    import torch

    rows, cols = values.shape
    ld = cols if ld is None else ld
    assert ld >= cols
    size = offset + max(rows, 1) * ld + GUARD
    flat = torch.full((size,), float(fill), dtype=torch.float32)
    if rows and cols:
        box = flat[offset:offset + rows * ld].view(rows, ld)[:, :cols]
        box.copy_(torch.from_numpy(np.ascontiguousarray(values)))
    flat = flat.cuda()
    view = flat.as_strided((rows, cols), (ld, 1), offset)
    return flat, view


def run_sgemm(A: np.ndarray, B: np.ndarray, *, lda=None, ldb=None, ldc=None, offsets=(0, 0, 0),
              prefill=np.nan):
    """Run the library on numpy inputs; return (C as numpy, C's flat buffer on host, status)."""
    import torch
    from dense_fp32_matrix_major_gb300 import sgemm

    M, K = A.shape
    N = B.shape[1]
    lda = max(K, 1) if lda is None else lda
    ldb = max(N, 1) if ldb is None else ldb
    ldc = max(N, 1) if ldc is None else ldc
    fa, vA = device_matrix(A, lda, offsets[0])
    fb, vB = device_matrix(B, ldb, offsets[1])
    cvals = np.full((M, N), prefill, dtype=np.float32)
    fc, vC = device_matrix(cvals, ldc, offsets[2])
    stream = torch.cuda.current_stream()
    rc = sgemm.sgemm_f32_raw(M, N, K, vA.data_ptr(), lda, vB.data_ptr(), ldb, vC.data_ptr(), ldc,
                             stream.cuda_stream)
    torch.cuda.synchronize()
    flat = fc.cpu().numpy()
    box = vC.cpu().numpy() if M and N else np.zeros((M, N), np.float32)
    return box, flat, rc


def outside_box_intact(flat: np.ndarray, M: int, N: int, ldc: int, offset: int) -> bool:
    """True if every float of C's buffer outside the M x N box still holds CANARY."""
    mask = np.ones(flat.shape[0], dtype=bool)
    for i in range(M):
        mask[offset + i * ldc: offset + i * ldc + N] = False
    return bool(np.all(flat[mask].view(np.uint32) == np.float32(CANARY).view(np.uint32)))


def oracle_error(C: np.ndarray, A: np.ndarray, B: np.ndarray, nthreads=None) -> float:
    """Normalised error of C against the double-accumulating oracle (full product)."""
    if A.shape[0] * A.shape[1] * B.shape[1] <= 2_000_000:
        C64, S = oracle.sgemm_f64(A, B)
    else:
        C64, S = oracle.sgemm_f64_rows(A, B, nthreads=nthreads)
    return oracle.normalized_error(C, C64, S)


def sampled_error(C: np.ndarray, A: np.ndarray, B: np.ndarray, rows, cols) -> float:
    c64, s = oracle.sgemm_f64_at(A, B, rows, cols)
    return oracle.normalized_error(C[rows, cols], c64, s)


def run_gemm_ex(A: np.ndarray, B: np.ndarray, *, transA=False, transB=False, alpha=1.0, beta=0.0,
                C_init=None, lda=None, ldb=None, ldc=None, offsets=(0, 0, 0)):
    """sgemm_f32_ex on numpy inputs given in STORED form (A is K x M when
    transA, B is N x K when transB); returns (C, flat C buffer, status)."""
    import torch
    from dense_fp32_matrix_major_gb300 import sgemm

    M = A.shape[1] if transA else A.shape[0]
    K = A.shape[0] if transA else A.shape[1]
    N = B.shape[0] if transB else B.shape[1]
    lda = max(A.shape[1], 1) if lda is None else lda
    ldb = max(B.shape[1], 1) if ldb is None else ldb
    ldc = max(N, 1) if ldc is None else ldc
    fa, vA = device_matrix(A, lda, offsets[0])
    fb, vB = device_matrix(B, ldb, offsets[1])
    cvals = np.full((M, N), np.nan, dtype=np.float32) if C_init is None else C_init
    fc, vC = device_matrix(cvals, ldc, offsets[2])
    stream = torch.cuda.current_stream()
    rc = sgemm.lib.sgemm_f32_ex(int(transA), int(transB), M, N, K, float(alpha), vA.data_ptr(), lda,
                                vB.data_ptr(), ldb, float(beta), vC.data_ptr(), ldc, stream.cuda_stream)
    torch.cuda.synchronize()
    flat = fc.cpu().numpy()
    box = vC.cpu().numpy() if M and N else np.zeros((M, N), np.float32)
    return box, flat, rc


def run_fused(A: np.ndarray, B: np.ndarray, *, bias=None, bias_kind=0, act=0, transA=False, transB=False,
              alpha=1.0, beta=0.0, C_init=None, lda=None, ldb=None, ldc=None, offsets=(0, 0, 0),
              bias_offset=0):
    """sgemm_f32_fused on numpy inputs in STORED form; the bias vector sits
    ``bias_offset`` floats into its own guarded buffer. Returns (C, flat C
    buffer, status)."""
    import torch
    from dense_fp32_matrix_major_gb300 import sgemm

    M = A.shape[1] if transA else A.shape[0]
    K = A.shape[0] if transA else A.shape[1]
    N = B.shape[0] if transB else B.shape[1]
    lda = max(A.shape[1], 1) if lda is None else lda
    ldb = max(B.shape[1], 1) if ldb is None else ldb
    ldc = max(N, 1) if ldc is None else ldc
    fa, vA = device_matrix(A, lda, offsets[0])
    fb, vB = device_matrix(B, ldb, offsets[1])
    cvals = np.full((M, N), np.nan, dtype=np.float32) if C_init is None else C_init
    fc, vC = device_matrix(cvals, ldc, offsets[2])
    bias_ptr = 0
    if bias is not None:
        fbias, vbias = device_matrix(np.asarray(bias, np.float32).reshape(1, -1), None, bias_offset, fill=np.nan)
        bias_ptr = vbias.data_ptr()
    stream = torch.cuda.current_stream()
    rc = sgemm.lib.sgemm_f32_fused(int(transA), int(transB), M, N, K, float(alpha), vA.data_ptr(), lda,
                                   vB.data_ptr(), ldb, float(beta), vC.data_ptr(), ldc, bias_ptr, int(bias_kind),
                                   int(act), stream.cuda_stream)
    torch.cuda.synchronize()
    flat = fc.cpu().numpy()
    box = vC.cpu().numpy() if M and N else np.zeros((M, N), np.float32)
    return box, flat, rc


def run_batched(As, Bs, *, transA=False, transB=False, alpha=1.0, beta=0.0, C0=None,
                strideA=None, strideB=None, strideC=None, share_a=False, share_b=False):
    """sgemm_f32_batched on lists of stored-form items (dense rows). Items sit
    stride elements apart in one buffer (default: packed); share_a / share_b
    pass stride 0 with a single matrix. Returns (list of C items, flat C
    buffer, status, strideC)."""
    import torch
    from dense_fp32_matrix_major_gb300 import sgemm

    batch = len(As)
    A0, B0 = As[0], Bs[0]
    M = A0.shape[1] if transA else A0.shape[0]
    K = A0.shape[0] if transA else A0.shape[1]
    N = B0.shape[0] if transB else B0.shape[1]
    lda, ldb, ldc = max(A0.shape[1], 1), max(B0.shape[1], 1), max(N, 1)

    def pack(items, stride, share, fill):
        rows, cols = items[0].shape
        stride = 0 if share else (rows * cols if stride is None else stride)
        n = 1 if share else len(items)
        size = (n - 1) * stride + rows * cols + GUARD
        flat = np.full(size, fill, dtype=np.float32)
        for b in range(n):
            flat[b * stride: b * stride + rows * cols] = np.ascontiguousarray(items[b]).ravel()
        return torch.from_numpy(flat).cuda(), stride

    dA, sA = pack(As, strideA, share_a, 0.0)
    dB, sB = pack(Bs, strideB, share_b, 0.0)
    Cs = C0 if C0 is not None else [np.full((M, N), np.nan, np.float32) for _ in range(batch)]
    dC, sC = pack(Cs, strideC, False, CANARY)
    stream = torch.cuda.current_stream()
    rc = sgemm.lib.sgemm_f32_batched(int(transA), int(transB), M, N, K, float(alpha), dA.data_ptr(), lda,
                                     sA, dB.data_ptr(), ldb, sB, float(beta), dC.data_ptr(), ldc, sC,
                                     batch, stream.cuda_stream)
    torch.cuda.synchronize()
    flat = dC.cpu().numpy()
    out = [flat[b * sC: b * sC + M * N].reshape(M, N).copy() for b in range(batch)]
    return out, flat, rc, sC


def batched_outside_intact(flat, batch, M, N, strideC):
    mask = np.ones(flat.shape[0], dtype=bool)
    for b in range(batch):
        mask[b * strideC: b * strideC + M * N] = False
    return bool(np.all(flat[mask].view(np.uint32) == np.float32(CANARY).view(np.uint32)))
