"""CPU oracle for dense fp32 row-major matrix multiplication.

TEST INFRASTRUCTURE ONLY. The product path (the CUDA library and its Python
binding) never imports this package. Only the tests, the smoke check and the
bench's cpu-baseline leg use it.

The arithmetic lives in ``sgemm_oracle.c`` (plain C, compiled here for the
host with ``-ffp-contract=off``). This module builds that file with gcc, loads
it with ctypes, and adds one numpy routine, :func:`normalized_error`, which is
the acceptance measure used by every parity test:

    err = max over (i, j) of |C_test[i][j] - C64[i][j]| / S[i][j]

with ``S[i][j] = sum_k |A[i][k]| * |B[k][j]|``. Where ``S`` is zero every term
of the sum is zero, so ``C_test`` must be exactly zero there. The measure is
the componentwise relative error of a dot product, the quantity that the
standard error bound for recursive summation limits (Higham, "Accuracy and
Stability of Numerical Algorithms", section 3.1).

The definition that the C routines follow is the plain sum of products stated
on every source page: "CUDA算子优化(4)：矩阵乘法", section "矩阵乘法的数学定义",
and "CUDA内存优化入门：从Naive到Tiled矩阵乘法", section 三 (formula block).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgemm_oracle.c")
_HDR = os.path.join(_HERE, "sgemm_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libsgemm_oracle.so")

_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle into a host shared library; return its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and all(
        os.path.getmtime(_LIB_PATH) >= os.path.getmtime(p) for p in (_SRC, _HDR)
    )
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = [
        "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
        "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra",
        "-o", tmp, _SRC, "-lm",
    ]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_sgemm_f32.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64]
            lib.oracle_sgemm_f64.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _i64]
            lib.oracle_sgemm_f64_rows.argtypes = [
                _i64, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _i64, ctypes.c_int]
            lib.oracle_sgemm_f32_rows.argtypes = [
                _i64, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, ctypes.c_int]
            lib.oracle_sgemm_f64_at.argtypes = [
                _i64, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _vp, _vp, _vp, _vp]
            _d = ctypes.c_double
            lib.oracle_gemm_f64.argtypes = [ctypes.c_int, ctypes.c_int, _i64, _i64, _i64, _d, _vp, _i64,
                                            _vp, _i64, _d, _vp, _i64, _vp, _vp, _i64]
            lib.oracle_gemm_f64_at.argtypes = [ctypes.c_int, ctypes.c_int, _i64, _i64, _i64, _d, _vp,
                                               _i64, _vp, _i64, _d, _vp, _i64, _i64, _vp, _vp, _vp, _vp]
            lib.oracle_epilogue_f64.argtypes = [_i64, _vp, _vp, _i64, _i64, _vp, ctypes.c_int, ctypes.c_int,
                                                _vp, _vp]
            for fn in (lib.oracle_sgemm_f32, lib.oracle_sgemm_f32_rows, lib.oracle_sgemm_f64, lib.oracle_sgemm_f64_rows,
                       lib.oracle_sgemm_f64_at, lib.oracle_gemm_f64, lib.oracle_gemm_f64_at,
                       lib.oracle_epilogue_f64):
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _rowmajor(x: np.ndarray, name: str):
    """(pointer, row stride in elements) of a 2-D float32 array with unit column stride."""
    if x.dtype != np.float32 or x.ndim != 2:
        raise TypeError(f"{name} must be a 2-D float32 array")
    if x.size == 0:
        return x.ctypes.data, max(x.shape[1], 1)
    if x.shape[1] > 1 and x.strides[1] != 4:
        raise ValueError(f"{name} must have contiguous rows")
    ld = x.strides[0] // 4 if x.shape[0] > 1 else max(x.shape[1], 1)
    if x.shape[0] > 1 and x.strides[0] % 4:
        raise ValueError(f"{name} row stride must be whole elements")
    return x.ctypes.data, ld


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"{what}: oracle rejected the arguments (code {rc})")


def sgemm_f32(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """The pages' CPU loop: float accumulator, k ascending, no fused multiply-add."""
    (M, K), (K2, N) = A.shape, B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    pa, lda = _rowmajor(A, "A")
    pb, ldb = _rowmajor(B, "B")
    C = np.empty((M, N), dtype=np.float32)
    _check(_load().oracle_sgemm_f32(M, N, K, pa, lda, pb, ldb, C.ctypes.data, max(N, 1)),
           "oracle_sgemm_f32")
    return C


def sgemm_f32_rows(A: np.ndarray, B: np.ndarray, row_begin: int = 0, row_end=None,
                   nthreads: int | None = None) -> np.ndarray:
    """Rows [row_begin, row_end) of the pages' float product, i-k-j order,
    threaded by rows; bit-identical to :func:`sgemm_f32` on those rows."""
    (M, K), (K2, N) = A.shape, B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    row_end = M if row_end is None else row_end
    if not 0 <= row_begin <= row_end <= M:
        raise ValueError("row band out of range")
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    pa, lda = _rowmajor(A, "A")
    pb, ldb = _rowmajor(B, "B")
    C = np.empty((row_end - row_begin, N), dtype=np.float32)
    _check(_load().oracle_sgemm_f32_rows(row_begin, row_end, N, K, pa, lda, pb, ldb, C.ctypes.data,
                                         max(N, 1), int(nthreads)), "oracle_sgemm_f32_rows")
    return C


def sgemm_f64(A: np.ndarray, B: np.ndarray):
    """(C64, S): the product accumulated in double, and sum_k |A||B| in double."""
    (M, K), (K2, N) = A.shape, B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    pa, lda = _rowmajor(A, "A")
    pb, ldb = _rowmajor(B, "B")
    C64 = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    _check(_load().oracle_sgemm_f64(M, N, K, pa, lda, pb, ldb, C64.ctypes.data,
                                    S.ctypes.data, max(N, 1)), "oracle_sgemm_f64")
    return C64, S


def sgemm_f64_rows(A: np.ndarray, B: np.ndarray, row_begin: int = 0, row_end=None,
                   nthreads: int | None = None):
    """(C64, S) for rows [row_begin, row_end), i-k-j order, threaded by rows."""
    (M, K), (K2, N) = A.shape, B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    row_end = M if row_end is None else row_end
    if not 0 <= row_begin <= row_end <= M:
        raise ValueError("row band out of range")
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    pa, lda = _rowmajor(A, "A")
    pb, ldb = _rowmajor(B, "B")
    rows = row_end - row_begin
    C64 = np.empty((rows, N), dtype=np.float64)
    S = np.empty((rows, N), dtype=np.float64)
    _check(_load().oracle_sgemm_f64_rows(row_begin, row_end, N, K, pa, lda, pb, ldb,
                                         C64.ctypes.data, S.ctypes.data, max(N, 1),
                                         int(nthreads)), "oracle_sgemm_f64_rows")
    return C64, S


def sgemm_f64_at(A: np.ndarray, B: np.ndarray, rows, cols):
    """(c64, s) at the positions (rows[t], cols[t])."""
    (M, K), (K2, N) = A.shape, B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape or r.ndim != 1:
        raise ValueError("rows and cols must be 1-D and of equal length")
    pa, lda = _rowmajor(A, "A")
    pb, ldb = _rowmajor(B, "B")
    c64 = np.empty(r.shape[0], dtype=np.float64)
    s = np.empty(r.shape[0], dtype=np.float64)
    _check(_load().oracle_sgemm_f64_at(M, N, K, pa, lda, pb, ldb, r.shape[0], r.ctypes.data,
                                       c.ctypes.data, c64.ctypes.data, s.ctypes.data),
           "oracle_sgemm_f64_at")
    return c64, s


def _gemm_shapes(A, B, transA, transB):
    M, K = (A.shape[1], A.shape[0]) if transA else A.shape
    K2, N = (B.shape[1], B.shape[0]) if transB else B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    return M, N, K


def _c_in(C_in, beta, M, N):
    if beta == 0.0:
        return None, max(N, 1)
    if C_in is None or C_in.shape != (M, N):
        raise ValueError("beta != 0 needs C_in of shape (M, N)")
    return _rowmajor(C_in, "C_in")


def gemm_f64(A, B, *, transA=False, transB=False, alpha=1.0, beta=0.0, C_in=None):
    """(C64, S) of alpha * op(A) @ op(B) + beta * C_in (the BLAS GEMM form).

    S = |alpha| sum_k |op(A)||op(B)| + |beta| |C_in|, the scale of the
    acceptance measure. With beta == 0, C_in is not read.
    """
    M, N, K = _gemm_shapes(A, B, transA, transB)
    pa, lda = _rowmajor(A, "A")
    pb, ldb = _rowmajor(B, "B")
    pc, ldc_in = _c_in(C_in, beta, M, N)
    C64 = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    _check(_load().oracle_gemm_f64(int(transA), int(transB), M, N, K, float(alpha), pa, lda, pb,
                                   ldb, float(beta), pc, ldc_in, C64.ctypes.data, S.ctypes.data,
                                   max(N, 1)), "oracle_gemm_f64")
    return C64, S


def gemm_f64_at(A, B, rows, cols, *, transA=False, transB=False, alpha=1.0, beta=0.0, C_in=None):
    """(c64, s) of the GEMM form at (rows[t], cols[t])."""
    M, N, K = _gemm_shapes(A, B, transA, transB)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    pa, lda = _rowmajor(A, "A")
    pb, ldb = _rowmajor(B, "B")
    pc, ldc_in = _c_in(C_in, beta, M, N)
    c64 = np.empty(r.shape[0], dtype=np.float64)
    s = np.empty(r.shape[0], dtype=np.float64)
    _check(_load().oracle_gemm_f64_at(int(transA), int(transB), M, N, K, float(alpha), pa, lda,
                                      pb, ldb, float(beta), pc, ldc_in, r.shape[0], r.ctypes.data,
                                      c.ctypes.data, c64.ctypes.data, s.ctypes.data),
           "oracle_gemm_f64_at")
    return c64, s


_BIAS_KINDS = {None: 0, "none": 0, "col": 1, "row": 2}
_ACTS = {None: 0, "none": 0, "relu": 1, "gelu": 2, "silu": 3}


def epilogue_f64(c64, s, *, bias=None, bias_kind=None, act=None, rows=None, cols=None, shape=None):
    """(act(c64 + bias), s + |bias|) for values of a double product, as new arrays.

    ``c64`` and ``s`` are the full M x N result, or 1-D samples at
    ``(rows[t], cols[t])`` of a result of the given ``shape`` (M, N).
    ``bias_kind`` is None / "col" (bias[j], N values) / "row" (bias[i], M
    values); ``act`` is None / "relu" / "gelu" / "silu".
    """
    kind = _BIAS_KINDS[bias_kind]
    code = _ACTS[act]
    flat = np.array(c64, dtype=np.float64).reshape(-1)
    sflat = np.array(s, dtype=np.float64).reshape(-1)
    if rows is None:
        M, N = np.shape(c64)
        rr, cc = np.indices((M, N))
        r, c = rr.reshape(-1), cc.reshape(-1)
    else:
        if shape is None:
            raise ValueError("samples need the shape (M, N) of the result")
        M, N = shape
        r, c = rows, cols
    r = np.ascontiguousarray(r, dtype=np.int64)
    c = np.ascontiguousarray(c, dtype=np.int64)
    if r.shape != flat.shape or c.shape != flat.shape or sflat.shape != flat.shape:
        raise ValueError("samples, values and scales must have the same length")
    pb = None
    if kind:
        b = np.ascontiguousarray(bias, dtype=np.float32).reshape(-1)
        if b.shape[0] != (N if kind == 1 else M):
            raise ValueError("bias length must be N (per column) or M (per row)")
        pb = b.ctypes.data
    _check(_load().oracle_epilogue_f64(flat.shape[0], r.ctypes.data, c.ctypes.data, M, N, pb, kind, code,
                                       flat.ctypes.data, sflat.ctypes.data), "oracle_epilogue_f64")
    return flat.reshape(np.shape(c64)), sflat.reshape(np.shape(s))


def normalized_error(C_test, C64, S) -> float:
    """max |C_test - C64| / S; inf if C_test is nonzero (or not finite) where S is zero.

    Any NaN or infinity in C_test gives inf, so an output element that was
    never written (tests prefill outputs with NaN) fails the measure.
    """
    C_test = np.asarray(C_test, dtype=np.float64)
    C64 = np.asarray(C64, dtype=np.float64)
    S = np.asarray(S, dtype=np.float64)
    if C_test.shape != C64.shape or C64.shape != S.shape:
        raise ValueError("shape mismatch")
    if C_test.size == 0:
        return 0.0
    if not np.all(np.isfinite(C_test)):
        return float("inf")
    zero = S == 0.0
    if np.any(C_test[zero] != 0.0):
        return float("inf")
    diff = np.abs(C_test - C64)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(zero, 0.0, diff / np.where(zero, 1.0, S))
    return float(ratio.max())
