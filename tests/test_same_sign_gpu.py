"""GPU parity on inputs whose products all share a sign.

The complete program of "CUDA内存优化入门：从Naive到Tiled矩阵乘法" (section
八) fills A and B with rand() / RAND_MAX, i.e. U[0, 1). On such inputs every
partial sum grows in one direction, so a rounding that always leans the same
way (the tensor core's accumulation truncates) adds up along the whole
accumulation chain instead of cancelling as it does on zero-mean data. These
tests hold every kernel and schedule to the acceptance bound
max |C - C64| / sum_k |A||B| <= 1e-5 on U[0,1], |N(0,1)| and U[0,1] x N(0,1)
inputs for K from 512 to 16384, comparing every output with the oracle.
"""

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_major_gb300 import workloads as wl
from tests.gpu_harness import TOL, outside_box_intact, run_sgemm

pytestmark = pytest.mark.gpu

KS = [512, 1024, 1537, 4096, 8192, 8193, 16384]
DISTS = [("uniform01", "uniform01"), ("absnormal", "absnormal"), ("uniform01", "normal")]
# (variant, stream-K mode, tensor-core kernel): AUTO, and every tensor-core
# kernel (1 per-thread loads, 2 TMA, 3 A in tensor memory, 4 SM pairs)
# under the automatic, data-parallel, hybrid and all-stream-K schedules.
SETTINGS = [("auto", 0, 0)] + [("tf32x3", sk, k) for k in (1, 2, 3, 4) for sk in (0, 1, 2, 3)]
IDS = [f"{v}-sk{sk}-k{k}" for v, sk, k in SETTINGS]

_cache = {}


def _case(M, N, K, da, db, seed):
    key = (M, N, K, da, db, seed)
    if key not in _cache:
        A, B = wl.make_mixed(M, N, K, da, db, seed)
        C64, S = oracle.sgemm_f64_rows(A, B)
        _cache[key] = (A, B, C64, S)
    return _cache[key]


@pytest.fixture(scope="module")
def lib():
    import torch

    assert torch.cuda.is_available()
    from dense_fp32_matrix_major_gb300 import sgemm

    yield sgemm
    sgemm.set_variant(0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_STREAM_K, 0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_TF32X3_KERNEL, 0)


@pytest.mark.parametrize("setting", SETTINGS, ids=IDS)
@pytest.mark.parametrize("dists", DISTS, ids=["u01", "absn", "u01xn"])
def test_same_sign_every_k(lib, setting, dists):
    variant, sk, kern = setting
    lib.set_variant(variant)
    lib.set_tuning(lib.SGEMM_TUNE_STREAM_K, sk)
    lib.set_tuning(lib.SGEMM_TUNE_TF32X3_KERNEL, kern)
    M, N = 300, 520  # several tiles of every kernel, ragged in both directions
    for K in KS:
        A, B, C64, S = _case(M, N, K, dists[0], dists[1], K)
        C, flat, rc = run_sgemm(A, B)
        assert rc == 0, K
        assert outside_box_intact(flat, M, N, N, 0)
        err = oracle.normalized_error(C, C64, S)
        assert err <= TOL, (K, err)


@pytest.mark.parametrize("kern", [0, 4])
def test_same_sign_headline_shape(lib, kern):
    """P2's benchmark shape (2048 x 4096 x 3072) with the pages' U[0,1]
    inputs, every output compared."""
    lib.set_variant("auto" if kern == 0 else "tf32x3")
    lib.set_tuning(lib.SGEMM_TUNE_STREAM_K, 0)
    lib.set_tuning(lib.SGEMM_TUNE_TF32X3_KERNEL, kern)
    A, B, C64, S = _case(2048, 3072, 4096, "uniform01", "uniform01", 4)
    C, flat, rc = run_sgemm(A, B)
    assert rc == 0
    assert lib.variant_name(lib.last_variant_used()) == "tf32x3"
    assert oracle.normalized_error(C, C64, S) <= TOL


def test_same_sign_ffma_reference_level(lib):
    """The CUDA-core variant rounds every fused multiply-add to nearest, so
    its error on non-negative inputs stays near the float loop's."""
    lib.set_variant("ffma")
    A, B, C64, S = _case(300, 520, 16384, "uniform01", "uniform01", 16384)
    C, flat, rc = run_sgemm(A, B)
    assert rc == 0
    assert oracle.normalized_error(C, C64, S) <= 2e-6
