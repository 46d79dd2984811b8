"""GPU parity of strided-batched products (sgemm_f32_batched): every item
against the oracle's general form, C gaps between items untouched."""

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_major_gb300 import workloads as wl
from tests.gpu_harness import TOL, batched_outside_intact, run_batched

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from dense_fp32_matrix_major_gb300 import sgemm

    yield sgemm
    sgemm.set_variant(0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_STREAM_K, 0)


def _items(batch, M, N, K, tA, tB, seed, dist="normal"):
    As, Bs = [], []
    for b in range(batch):
        A, B = wl.make_pair(M, N, K, dist, seed * 1000 + b)
        As.append(np.ascontiguousarray(A.T) if tA else A)
        Bs.append(np.ascontiguousarray(B.T) if tB else B)
    return As, Bs


def _verify(As, Bs, out, tA, tB, alpha, beta, C0, share_a=False, share_b=False):
    for b, C in enumerate(out):
        A = As[0] if share_a else As[b]
        B = Bs[0] if share_b else Bs[b]
        C64, S = oracle.gemm_f64(A, B, transA=bool(tA), transB=bool(tB), alpha=alpha, beta=beta,
                                 C_in=C0[b] if beta else None)
        err = oracle.normalized_error(C, C64, S)
        assert err <= TOL, (b, err)


@pytest.mark.parametrize("variant", ["auto", "ffma", "tf32x3"])
@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_batched_forms(lib, variant, tA, tB):
    lib.set_variant(variant)
    for (batch, M, N, K) in [(1, 64, 64, 64), (3, 128, 256, 96), (17, 36, 20, 52), (5, 260, 132, 300)]:
        As, Bs = _items(batch, M, N, K, tA, tB, batch + M)
        C0 = [np.random.default_rng(b).standard_normal((M, N)).astype(np.float32) for b in range(batch)]
        for alpha, beta in [(1.0, 0.0), (-0.5, 2.0)]:
            out, flat, rc, sC = run_batched(As, Bs, transA=tA, transB=tB, alpha=alpha, beta=beta,
                                            C0=C0 if beta else None, strideC=M * N + 13)
            assert rc == 0
            assert batched_outside_intact(flat, batch, M, N, sC)
            _verify(As, Bs, out, tA, tB, alpha, beta, C0)


@pytest.mark.parametrize("variant", ["ffma", "tf32x3"])
def test_shared_operands(lib, variant):
    lib.set_variant(variant)
    batch, M, N, K = 6, 200, 264, 128
    As, Bs = _items(batch, M, N, K, 0, 0, 7)
    for share_a, share_b in [(True, False), (False, True), (True, True)]:
        out, flat, rc, sC = run_batched(As, Bs, share_a=share_a, share_b=share_b)
        assert rc == 0
        _verify(As, Bs, out, 0, 0, 1.0, 0.0, None, share_a, share_b)


def test_many_small_items_integer_exact(lib):
    lib.set_variant("auto")
    batch, M, N, K = 300, 24, 40, 56
    As, Bs = _items(batch, M, N, K, 0, 0, 3, dist="int4")
    out, flat, rc, sC = run_batched(As, Bs)
    assert rc == 0
    for b in range(batch):
        assert np.array_equal(out[b], (As[b].astype(np.int64) @ Bs[b].astype(np.int64)).astype(np.float32))


def test_large_batched_stream_k(lib):
    lib.set_variant("tf32x3")
    lib.set_tuning(lib.SGEMM_TUNE_STREAM_K, 3)  # every tile split along K
    batch, M, N, K = 4, 384, 512, 2048
    As, Bs = _items(batch, M, N, K, 0, 0, 9)
    C0 = [np.random.default_rng(b).standard_normal((M, N)).astype(np.float32) for b in range(batch)]
    out, flat, rc, sC = run_batched(As, Bs, alpha=1.5, beta=-1.0, C0=C0)
    lib.set_tuning(lib.SGEMM_TUNE_STREAM_K, 0)
    assert rc == 0
    for b in range(batch):
        r, c = wl.sample_positions(M, N, 500, seed=b)
        c64, s = oracle.gemm_f64_at(As[b], Bs[b], r, c, alpha=1.5, beta=-1.0, C_in=C0[b])
        assert oracle.normalized_error(out[b][r, c], c64, s) <= TOL


def test_batched_argument_checks(lib):
    import torch

    buf = torch.zeros(4096, device="cuda")
    p = buf.data_ptr()
    # C items overlapping one another (strideC < (M-1)*ldc + N).
    assert lib.lib.sgemm_f32_batched(0, 0, 8, 8, 8, 1.0, p, 8, 64, p + 4 * 1024, 8, 64, 0.0,
                                     p + 4 * 2048, 8, 10, 3, 0) == lib.SGEMM_ERR_INVALID_ARG
    # Negative stride.
    assert lib.lib.sgemm_f32_batched(0, 0, 8, 8, 8, 1.0, p, 8, -64, p + 4 * 1024, 8, 64, 0.0,
                                     p + 4 * 2048, 8, 64, 3, 0) == lib.SGEMM_ERR_INVALID_ARG
    # The last C item running into B.
    assert lib.lib.sgemm_f32_batched(0, 0, 8, 8, 8, 1.0, p, 8, 64, p + 4 * 1024, 8, 64, 0.0,
                                     p + 4 * 900, 8, 64, 3, 0) == lib.SGEMM_ERR_INVALID_ARG
    # batch 0: nothing to do.
    assert lib.lib.sgemm_f32_batched(0, 0, 8, 8, 8, 1.0, p, 8, 64, p + 4 * 1024, 8, 64, 0.0,
                                     p + 4 * 2048, 8, 64, 0, 0) == 0
