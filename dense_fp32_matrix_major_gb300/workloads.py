"""Seeded synthetic inputs for the SGEMM workloads.

This module holds the input recipes only: shapes, strides, distributions and
seeds. It does no part of the product's arithmetic, so the tests can feed the
same bytes to the CUDA library and to the CPU oracle.

The shapes follow the workloads that the source pages time:

* square 512 / 1024 / 2048 products, as in "CUDA内存优化入门：从Naive到Tiled
  矩阵乘法" section 七 (performance table, uniform inputs);
* all-ones 1024 x 1024 inputs, as in "CUDA 性能优化实战笔记 + C++示例代码
  （第七章重点）" section 二 (every output must equal 1024);
* M = 2048, K = 4096, N = 3072 with N(0, 1) entries, the benchmark shape of
  "CUDA算子优化(4)：矩阵乘法" (host driver of the V1 and V2 kernels);
* a ragged 1023 x 1537 x 2049 case whose row lengths are not multiples of
  four floats, so no 16-byte vector path applies;
* non-negative entries, U[0, 1) as the complete program of "CUDA内存优化入门：
  从Naive到Tiled矩阵乘法" section 八 initialises its matrices (rand() /
  RAND_MAX), and |N(0, 1)|: every product then has the same sign, so
  rounding errors that lean one way add up instead of cancelling.

Random entries come from numpy's PCG64 generator (``np.random.default_rng``),
which gives the same stream on every platform, drawn in float64 and rounded
once to float32.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dist: str  # "normal", "uniform", "uniform01", "absnormal", "ones", "int4" (integers in [-4, 4])
    seed: int = 0
    lda: int | None = None  # row strides in elements; None = dense rows
    ldb: int | None = None
    ldc: int | None = None

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes that must cross HBM at least once: read A and B, write C."""
        return 4 * (self.M * self.K + self.K * self.N + self.M * self.N)


# The five configurations of the benchmark plan (the 1024 case runs twice).
C1_512 = Workload("sq512_normal_s0", 512, 512, 512, "normal", 0)
C2_ONES = Workload("sq1024_ones", 1024, 1024, 1024, "ones", 0)
C2_UNIF = Workload("sq1024_uniform_s1", 1024, 1024, 1024, "uniform", 1)
C3_RAGGED = Workload("ragged_1023x2049x1537_normal_s2", 1023, 2049, 1537, "normal", 2)
C4_2048 = Workload("sq2048_normal_s3", 2048, 2048, 2048, "normal", 3)
C5_HEAD = Workload("m2048_n3072_k4096_normal_s4", 2048, 3072, 4096, "normal", 4)

ALL = (C1_512, C2_ONES, C2_UNIF, C3_RAGGED, C4_2048, C5_HEAD)
BY_NAME = {w.name: w for w in ALL}


def _draw(rng: np.random.Generator, shape, dist: str) -> np.ndarray:
    if dist == "normal":
        return rng.standard_normal(shape).astype(np.float32)
    if dist == "uniform":
        return (rng.random(shape) * 2.0 - 1.0).astype(np.float32)
    if dist == "uniform01":
        # U[0, 1): the pages' rand() / RAND_MAX initialisation, non-negative
        return rng.random(shape).astype(np.float32)
    if dist == "absnormal":
        return np.abs(rng.standard_normal(shape)).astype(np.float32)
    if dist == "ones":
        return np.ones(shape, dtype=np.float32)
    if dist == "int4":
        return rng.integers(-4, 5, size=shape).astype(np.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def strided(values: np.ndarray, ld: int | None, fill: float = np.nan) -> np.ndarray:
    """A view of ``values`` whose rows sit ``ld`` elements apart (padding = ``fill``)."""
    rows, cols = values.shape
    if ld is None or ld == cols:
        return np.ascontiguousarray(values)
    if ld < cols:
        raise ValueError("row stride shorter than the row")
    buf = np.full((rows, ld), fill, dtype=np.float32)
    buf[:, :cols] = values
    return buf[:, :cols]


def make_inputs(w: Workload):
    """(A, B) float32 arrays for a workload: A is M x K, B is K x N, row-major."""
    rng = np.random.default_rng(w.seed)
    A = _draw(rng, (w.M, w.K), w.dist)
    B = _draw(rng, (w.K, w.N), w.dist)
    return strided(A, w.lda), strided(B, w.ldb)


def make_pair(M: int, N: int, K: int, dist: str = "normal", seed: int = 0):
    """(A, B) for an ad-hoc shape with dense rows."""
    return make_inputs(Workload(f"adhoc_{M}x{N}x{K}", M, N, K, dist, seed))


def make_mixed(M: int, N: int, K: int, dist_a: str, dist_b: str, seed: int = 0):
    """(A, B) with A drawn from ``dist_a`` and B from ``dist_b`` (dense rows)."""
    rng = np.random.default_rng(seed)
    return _draw(rng, (M, K), dist_a), _draw(rng, (K, N), dist_b)


def sample_positions(M: int, N: int, count: int, seed: int = 0):
    """Rows and columns to spot-check: the four corners, the last row and column,
    and ``count`` seeded uniform positions."""
    rng = np.random.default_rng(10_000 + seed)
    fixed_r = [0, 0, M - 1, M - 1, M // 2, M - 1]
    fixed_c = [0, N - 1, 0, N - 1, N // 2, N // 2]
    r = np.concatenate([np.array(fixed_r), rng.integers(0, M, count)])
    c = np.concatenate([np.array(fixed_c), rng.integers(0, N, count)])
    return r.astype(np.int64), c.astype(np.int64)


@dataclass(frozen=True)
class BatchedWorkload:
    """A strided batch of independent products of one shape (items packed)."""
    name: str
    batch: int
    M: int
    N: int
    K: int
    dist: str
    seed: int = 0

    @property
    def flops(self) -> int:
        return 2 * self.batch * self.M * self.N * self.K


# Many small products: the tiled-decomposition workload of "【infra之路】Tiled
# Matrix Multiplication详解" taken per item (each item tiled independently).
B512_128 = BatchedWorkload("batch512_m128_n128_k128_normal_s5", 512, 128, 128, 128, "normal", 5)
B32_512 = BatchedWorkload("batch32_m512_n512_k512_normal_s6", 32, 512, 512, 512, "normal", 6)
BATCHED = (B512_128, B32_512)


def make_batched(w: BatchedWorkload):
    """(A, B) float32 arrays of shape (batch, M, K) and (batch, K, N)."""
    rng = np.random.default_rng(w.seed)
    A = _draw(rng, (w.batch, w.M, w.K), w.dist)
    B = _draw(rng, (w.batch, w.K, w.N), w.dist)
    return A, B
