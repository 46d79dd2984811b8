"""ctypes binding of libsgemm_gb300.so (the C ABI declared in include/sgemm.h).

Argument marshalling only: every step of the product runs in the library's
CUDA kernels. PyTorch supplies device memory and streams. Importing this
module loads the library and raises ImportError when it has not been built;
there is no CPU fallback.
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libsgemm_gb300.so")

SGEMM_OK = 0
SGEMM_ERR_INVALID_ARG = 1
SGEMM_ERR_UNSUPPORTED = 2
SGEMM_ERR_LAUNCH = 3
SGEMM_ERR_DEVICE = 4
SGEMM_ERR_TIMEOUT = 5
SGEMM_ERR_SCRATCH = 6
SGEMM_NOALLOC_SCRATCH_BYTES = 64 << 20

SGEMM_OP_N = 0
SGEMM_OP_T = 1

SGEMM_AUTO = 0
SGEMM_FFMA = 1
SGEMM_TF32X3 = 2

SGEMM_BIAS_NONE = 0
SGEMM_BIAS_PER_COL = 1
SGEMM_BIAS_PER_ROW = 2

SGEMM_ACT_NONE = 0
SGEMM_ACT_RELU = 1
SGEMM_ACT_GELU = 2
SGEMM_ACT_SILU = 3

BIAS_KINDS = {None: SGEMM_BIAS_NONE, "none": SGEMM_BIAS_NONE, "col": SGEMM_BIAS_PER_COL,
              "row": SGEMM_BIAS_PER_ROW}
ACTIVATIONS = {None: SGEMM_ACT_NONE, "none": SGEMM_ACT_NONE, "relu": SGEMM_ACT_RELU, "gelu": SGEMM_ACT_GELU,
               "silu": SGEMM_ACT_SILU}

SGEMM_TUNE_FFMA_TILE = 1
SGEMM_TUNE_STREAM_K = 2
SGEMM_TUNE_WATCHDOG_MS = 3
SGEMM_TUNE_TF32X3_KERNEL = 4
SGEMM_TUNE_LAST_TC_KERNEL = 5

# Every symbol that include/sgemm.h declares, with its ctypes signature.
_i64, _int, _vp, _cp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_char_p
SIGNATURES = {
    "sgemm_f32": (_int, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]),
    "sgemm_f32_noalloc": (_int, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]),
    "sgemm_f32_ex": (_int, [_int, _int, _i64, _i64, _i64, ctypes.c_float, _vp, _i64, _vp, _i64,
                            ctypes.c_float, _vp, _i64, _vp]),
    "sgemm_f32_batched": (_int, [_int, _int, _i64, _i64, _i64, ctypes.c_float, _vp, _i64, _i64, _vp, _i64,
                                 _i64, ctypes.c_float, _vp, _i64, _i64, _i64, _vp]),
    "sgemm_f32_fused": (_int, [_int, _int, _i64, _i64, _i64, ctypes.c_float, _vp, _i64, _vp, _i64,
                               ctypes.c_float, _vp, _i64, _vp, _int, _int, _vp]),
    "sgemm_f32_from_host": (_int, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _vp]),
    "sgemm_set_variant": (_int, [_int]),
    "sgemm_get_variant": (_int, []),
    "sgemm_variant_name": (_cp, [_int]),
    "sgemm_last_variant_used": (_int, []),
    "sgemm_last_launch_count": (_int, []),
    "sgemm_strerror": (_cp, [_int]),
    "sgemm_device_status": (_int, []),
    "sgemm_watchdog_selftest": (_int, [_i64, _vp]),
    "sgemm_set_tuning": (_int, [_int, _i64]),
    "sgemm_get_tuning": (_i64, [_int]),
    "sgemm_version": (_cp, []),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with dense_fp32_matrix_major_gb300._build.build() "
            "(nvcc, sm_103a). There is no CPU fallback.")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class SgemmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} (status {status})")


def strerror(status: int) -> str:
    return lib.sgemm_strerror(status).decode()


def variant_name(v: int) -> str:
    return lib.sgemm_variant_name(v).decode()


def set_variant(v) -> None:
    if isinstance(v, str):
        v = {"auto": SGEMM_AUTO, "ffma": SGEMM_FFMA, "tf32x3": SGEMM_TF32X3}[v]
    rc = lib.sgemm_set_variant(int(v))
    if rc:
        raise SgemmError(rc, "sgemm_set_variant")


def get_variant() -> int:
    return lib.sgemm_get_variant()


def last_variant_used() -> int:
    return lib.sgemm_last_variant_used()


def last_launch_count() -> int:
    return lib.sgemm_last_launch_count()


def set_tuning(key: int, value: int) -> None:
    rc = lib.sgemm_set_tuning(int(key), int(value))
    if rc:
        raise SgemmError(rc, "sgemm_set_tuning")


def get_tuning(key: int) -> int:
    return lib.sgemm_get_tuning(int(key))


def device_status() -> int:
    return lib.sgemm_device_status()


def watchdog_selftest(wait_ms: int, stream=None) -> None:
    """Enqueue a kernel whose one bounded wait must time out (see sgemm.h)."""
    rc = lib.sgemm_watchdog_selftest(int(wait_ms), _stream_handle(stream))
    if rc:
        raise SgemmError(rc, "sgemm_watchdog_selftest")


def version() -> str:
    return lib.sgemm_version().decode()


def sgemm_f32_raw(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, stream_handle=0) -> int:
    """Direct C-ABI call with integer device pointers; returns the status code."""
    return lib.sgemm_f32(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, stream_handle)


def sgemm_f32_noalloc_raw(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, stream_handle=0) -> int:
    """sgemm_f32_noalloc through the C ABI (integer device pointers); returns the status code."""
    return lib.sgemm_f32_noalloc(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, stream_handle)


def _rowmajor_2d(t, name):
    import torch

    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.dim() != 2:
        raise TypeError(f"{name} must be a 2-D torch.float32 tensor")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    rows, cols = t.shape
    if cols > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must have unit column stride (row-major)")
    ld = t.stride(0) if rows > 1 else max(cols, 1)
    return ld


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def sgemm_f32(A, B, C=None, stream=None):
    """C = A @ B for row-major float32 CUDA tensors, enqueued on ``stream``.

    A is M x K, B is K x N (row strides allowed, unit column stride). C, if
    given, is an M x N float32 CUDA tensor with unit column stride; otherwise
    a new one is allocated by PyTorch. Returns C.
    """
    import torch

    lda = _rowmajor_2d(A, "A")
    ldb = _rowmajor_2d(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    ldc = _rowmajor_2d(C, "C")
    if tuple(C.shape) != (M, N):
        raise ValueError("C has the wrong shape")
    rc = lib.sgemm_f32(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, C.data_ptr(), ldc,
                       _stream_handle(stream))
    if rc:
        raise SgemmError(rc, "sgemm_f32")
    return C


def gemm(A, B, C=None, *, transA=False, transB=False, alpha=1.0, beta=0.0, stream=None):
    """C = alpha * op(A) @ op(B) + beta * C for row-major float32 CUDA tensors.

    A is given as stored: M x K, or K x M when transA (op(A) = A^T); B is
    K x N, or N x K when transB. C (M x N) is read only when beta != 0; if
    C is None a new tensor is allocated by PyTorch (then beta must be 0).
    """
    import torch

    lda = _rowmajor_2d(A, "A")
    ldb = _rowmajor_2d(B, "B")
    M, K = (A.shape[1], A.shape[0]) if transA else tuple(A.shape)
    K2, N = (B.shape[1], B.shape[0]) if transB else tuple(B.shape)
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    ldc = _rowmajor_2d(C, "C")
    if tuple(C.shape) != (M, N):
        raise ValueError("C has the wrong shape")
    rc = lib.sgemm_f32_ex(int(transA), int(transB), M, N, K, float(alpha), A.data_ptr(), lda,
                          B.data_ptr(), ldb, float(beta), C.data_ptr(), ldc, _stream_handle(stream))
    if rc:
        raise SgemmError(rc, "sgemm_f32_ex")
    return C


def gemm_fused(A, B, C=None, *, bias=None, bias_kind=None, act=None, transA=False, transB=False, alpha=1.0,
               beta=0.0, stream=None):
    """C = act(alpha * op(A) @ op(B) + beta * C + bias) for row-major float32 CUDA tensors.

    Operands as in :func:`gemm`. ``bias`` is a contiguous float32 CUDA
    vector: N values for ``bias_kind="col"`` (one per column of C) or M
    values for ``bias_kind="row"``. ``act`` is None, "relu", "gelu" or
    "silu". Integer codes from sgemm.h are accepted for both.
    """
    import torch

    kind = bias_kind if isinstance(bias_kind, int) else BIAS_KINDS[bias_kind]
    code = act if isinstance(act, int) else ACTIVATIONS[act]
    lda = _rowmajor_2d(A, "A")
    ldb = _rowmajor_2d(B, "B")
    M, K = (A.shape[1], A.shape[0]) if transA else tuple(A.shape)
    K2, N = (B.shape[1], B.shape[0]) if transB else tuple(B.shape)
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    ldc = _rowmajor_2d(C, "C")
    if tuple(C.shape) != (M, N):
        raise ValueError("C has the wrong shape")
    bias_ptr = 0
    if kind != SGEMM_BIAS_NONE:
        if bias is None or bias.dtype != torch.float32 or not bias.is_cuda or not bias.is_contiguous():
            raise TypeError("bias must be a contiguous float32 CUDA tensor")
        if bias.numel() != (N if kind == SGEMM_BIAS_PER_COL else M):
            raise ValueError("bias length must be N (per column) or M (per row)")
        bias_ptr = bias.data_ptr()
    rc = lib.sgemm_f32_fused(int(transA), int(transB), M, N, K, float(alpha), A.data_ptr(), lda,
                             B.data_ptr(), ldb, float(beta), C.data_ptr(), ldc, bias_ptr, kind, code,
                             _stream_handle(stream))
    if rc:
        raise SgemmError(rc, "sgemm_f32_fused")
    return C


def gemm_batched(A, B, C=None, *, transA=False, transB=False, alpha=1.0, beta=0.0, stream=None):
    """C[b] = alpha * op(A[b]) @ op(B[b]) + beta * C[b] for 3-D float32 CUDA tensors.

    A is batch x M x K (batch x K x M when transA), B batch x K x N (batch x N
    x K when transB), C batch x M x N; each item row-major with unit column
    stride; a batch dimension of size 1 with stride 0 (expand) shares one
    matrix across the batch.
    """
    import torch

    def dims(t, name):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.dim() != 3 or not t.is_cuda:
            raise TypeError(f"{name} must be a 3-D float32 CUDA tensor")
        if t.shape[2] > 1 and t.stride(2) != 1:
            raise ValueError(f"{name} must have unit column stride")
        ld = t.stride(1) if t.shape[1] > 1 else max(t.shape[2], 1)
        return ld, t.stride(0)

    batch = A.shape[0]
    lda, sa = dims(A, "A")
    ldb, sb = dims(B, "B")
    M, K = (A.shape[2], A.shape[1]) if transA else (A.shape[1], A.shape[2])
    K2, N = (B.shape[2], B.shape[1]) if transB else (B.shape[1], B.shape[2])
    if K != K2 or B.shape[0] != batch:
        raise ValueError("shape mismatch")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((batch, M, N), dtype=torch.float32, device=A.device)
    ldc, sc = dims(C, "C")
    rc = lib.sgemm_f32_batched(int(transA), int(transB), M, N, K, float(alpha), A.data_ptr(), lda, sa,
                               B.data_ptr(), ldb, sb, float(beta), C.data_ptr(), ldc, sc, batch,
                               _stream_handle(stream))
    if rc:
        raise SgemmError(rc, "sgemm_f32_batched")
    return C


def sgemm_f32_from_host(A_host, B_host, C_host, dA, dB, dC, stream=None):
    """C_host = A_host @ B_host through caller-owned device buffers (see sgemm.h).

    A_host, B_host, C_host: 2-D float32 CPU tensors (pinned for asynchronous
    copies); dA, dB, dC: CUDA tensors with the same shapes and row strides.
    Enqueues copy-in, product and copy-out on ``stream`` and returns.
    """
    M, K = A_host.shape
    K2, N = B_host.shape
    if K != K2 or tuple(C_host.shape) != (M, N):
        raise ValueError("shape mismatch")
    for h, d, name in ((A_host, dA, "A"), (B_host, dB, "B"), (C_host, dC, "C")):
        if h.is_cuda or not d.is_cuda or h.shape != d.shape or h.stride() != d.stride():
            raise ValueError(f"{name}: host and device tensors must match in shape and strides")
    lda, ldb, ldc = (_rowmajor_2d(dA, "dA"), _rowmajor_2d(dB, "dB"), _rowmajor_2d(dC, "dC"))
    rc = lib.sgemm_f32_from_host(M, N, K, A_host.data_ptr(), lda, B_host.data_ptr(), ldb,
                                 C_host.data_ptr(), ldc, dA.data_ptr(), dB.data_ptr(),
                                 dC.data_ptr(), _stream_handle(stream))
    if rc:
        raise SgemmError(rc, "sgemm_f32_from_host")
    return C_host
