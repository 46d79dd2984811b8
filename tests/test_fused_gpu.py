"""GPU parity of the fused epilogue C = act(alpha * op(A) op(B) + beta * C + bias)
(sgemm_f32_fused) against the oracle's product followed by its epilogue.

Acceptance: the normalised error with the scale |alpha| sum |op(A)||op(B)| +
|beta| |C| + |bias| stays within the product's 1e-5 bound (the activations
are at most 1.13-Lipschitz, and the kernels' errors sit far below the
bound). Every schedule is covered: whole tiles (bias and activation in the
kernel's store) and tiles split along K (bias in the pre-pass, activation in
the post-pass).
"""

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_major_gb300 import workloads as wl
from tests.gpu_harness import TOL, outside_box_intact, run_fused

pytestmark = pytest.mark.gpu

KINDS = {None: 0, "col": 1, "row": 2}
ACTS = {None: 0, "relu": 1, "gelu": 2, "silu": 3}
# (variant, FFMA tile, stream-K mode, tensor-core kernel)
SETTINGS = [("ffma", 1, 1, 0), ("ffma", 2, 3, 0), ("ffma", 3, 2, 0), ("tf32x3", 0, 1, 3),
            ("tf32x3", 0, 3, 3), ("tf32x3", 0, 3, 2), ("tf32x3", 0, 3, 1), ("tf32x3", 0, 1, 4),
            ("tf32x3", 0, 3, 4), ("auto", 0, 0, 0)]


@pytest.fixture(scope="module")
def lib():
    from dense_fp32_matrix_major_gb300 import sgemm

    yield sgemm
    sgemm.set_variant(0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_FFMA_TILE, 0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_STREAM_K, 0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_TF32X3_KERNEL, 0)


def _configure(lib, variant, tile, sk, tc):
    lib.set_variant(variant)
    lib.set_tuning(lib.SGEMM_TUNE_FFMA_TILE, tile)
    lib.set_tuning(lib.SGEMM_TUNE_STREAM_K, sk)
    lib.set_tuning(lib.SGEMM_TUNE_TF32X3_KERNEL, tc)


def _stored(M, N, K, tA, tB, dist, seed):
    A, B = wl.make_pair(M, N, K, dist, seed)
    return (np.ascontiguousarray(A.T) if tA else A), (np.ascontiguousarray(B.T) if tB else B)


def _bias(kind, M, N, seed):
    if kind is None:
        return None
    return (np.random.default_rng(seed).standard_normal(N if kind == "col" else M) * 3).astype(np.float32)


def _expected(As, Bs, tA, tB, alpha, beta, C0, bias, kind, act):
    C64, S = oracle.gemm_f64(As, Bs, transA=bool(tA), transB=bool(tB), alpha=alpha, beta=beta,
                             C_in=C0 if beta else None)
    return oracle.epilogue_f64(C64, S, bias=bias, bias_kind=kind, act=act)


def _check(lib, M, N, K, tA, tB, alpha, beta, kind, act, seed, **kw):
    As, Bs = _stored(M, N, K, tA, tB, "normal", seed)
    C0 = np.random.default_rng(seed + 1).standard_normal((M, N)).astype(np.float32)
    bias = _bias(kind, M, N, seed + 2)
    C, flat, rc = run_fused(As, Bs, bias=bias, bias_kind=KINDS[kind], act=ACTS[act], transA=tA, transB=tB,
                            alpha=alpha, beta=beta, C_init=C0 if beta else None, **kw)
    assert rc == 0, lib.strerror(rc)  # every form at any alignment
    ldc = kw.get("ldc") or max(N, 1)
    assert outside_box_intact(flat, M, N, ldc, kw.get("offsets", (0, 0, 0))[2])
    C64, S = _expected(As, Bs, tA, tB, alpha, beta, C0, bias, kind, act)
    err = oracle.normalized_error(C, C64, S)
    assert err <= TOL, (M, N, K, tA, tB, kind, act, err)


@pytest.mark.parametrize("setting", SETTINGS, ids=lambda s: "-".join(map(str, s)))
@pytest.mark.parametrize("kind", [None, "col", "row"])
@pytest.mark.parametrize("act", [None, "relu", "gelu", "silu"])
def test_bias_and_activation(lib, setting, kind, act):
    _configure(lib, *setting)
    for (M, N, K) in [(1, 1, 1), (129, 257, 47), (300, 200, 513), (260, 516, 300)]:
        _check(lib, M, N, K, 0, 0, 1.0, 0.0, kind, act, M + N + K)


@pytest.mark.parametrize("setting", SETTINGS, ids=lambda s: "-".join(map(str, s)))
@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_forms_scales_and_epilogue(lib, setting, tA, tB):
    _configure(lib, *setting)
    for (M, N, K), (alpha, beta), kind, act in [((64, 300, 1000), (2.5, -1.5), "col", "gelu"),
                                               ((300, 200, 513), (-1.0, 1.0), "row", "silu"),
                                               ((128, 256, 64), (0.75, 0.0), "col", "relu"),
                                               ((5, 3, 7), (1.0, 1.0), "row", "gelu")]:
        _check(lib, M, N, K, tA, tB, alpha, beta, kind, act, 3 * M + K)


@pytest.mark.parametrize("setting", SETTINGS, ids=lambda s: "-".join(map(str, s)))
def test_unaligned_rows_and_bias(lib, setting):
    """Row strides and offsets that rule out 16-byte vectors; a bias vector at
    an odd float offset."""
    _configure(lib, *setting)
    M, N, K = 150, 270, 90
    kw = dict(lda=K + 3, ldb=N + 5, ldc=N + 7, offsets=(1, 3, 2), bias_offset=1)
    _check(lib, M, N, K, 0, 0, 1.5, -0.5, "col", "gelu", 8, **kw)
    _check(lib, M, N, K, 0, 0, 1.5, -0.5, "row", "relu", 9, **kw)


@pytest.mark.parametrize("variant", ["ffma", "tf32x3"])
@pytest.mark.parametrize("sk", [1, 3])
def test_integer_relu_bit_exact(lib, variant, sk):
    """Integer inputs: every partial sum is exact, so ReLU(3 A B - 2 C + bias)
    must match the integer closed form bit for bit, split tiles included."""
    _configure(lib, variant, 0, sk, 0)
    M, N, K = 256, 300, 1000
    As, Bs = _stored(M, N, K, 0, 0, "int4", 5)
    C0 = np.random.default_rng(1).integers(-9, 10, (M, N)).astype(np.float32)
    for kind in ("col", "row"):
        bias = np.random.default_rng(2).integers(-300, 301, N if kind == "col" else M).astype(np.float32)
        C, flat, rc = run_fused(As, Bs, bias=bias, bias_kind=KINDS[kind], act=ACTS["relu"], alpha=3.0,
                                beta=-2.0, C_init=C0)
        assert rc == 0
        b = bias.astype(np.int64)
        pre = 3 * (As.astype(np.int64) @ Bs.astype(np.int64)) - 2 * C0.astype(np.int64)
        pre = pre + (b[None, :] if kind == "col" else b[:, None])
        assert np.array_equal(C, np.maximum(pre, 0).astype(np.float32))


@pytest.mark.parametrize("alpha,K", [(0.0, 64), (1.0, 0)])
def test_scale_only_paths_apply_epilogue(lib, alpha, K):
    """alpha = 0 or K = 0: C = act(beta * C + bias) without touching A, B."""
    _configure(lib, "auto", 0, 0, 0)
    M, N = 70, 90
    As = np.random.default_rng(0).standard_normal((M, K)).astype(np.float32)
    Bs = np.random.default_rng(1).standard_normal((K, N)).astype(np.float32)
    C0 = np.random.default_rng(2).standard_normal((M, N)).astype(np.float32)
    for kind, act in [("col", "gelu"), ("row", "relu"), (None, "silu")]:
        bias = _bias(kind, M, N, 3)
        C, flat, rc = run_fused(As, Bs, bias=bias, bias_kind=KINDS[kind], act=ACTS[act], alpha=alpha,
                                beta=-1.5, C_init=C0)
        assert rc == 0
        assert outside_box_intact(flat, M, N, N, 0)
        C64 = -1.5 * C0.astype(np.float64)
        S = 1.5 * np.abs(C0).astype(np.float64)
        e64, eS = oracle.epilogue_f64(C64, S, bias=bias, bias_kind=kind, act=act)
        assert oracle.normalized_error(C, e64, eS) <= TOL


def test_invalid_epilogue_arguments(lib):
    import torch

    _configure(lib, "auto", 0, 0, 0)
    A = torch.zeros((8, 8), device="cuda")
    B = torch.zeros((8, 8), device="cuda")
    C = torch.zeros((8, 8), device="cuda")
    bias = torch.zeros(8, device="cuda")
    call = lib.lib.sgemm_f32_fused
    args = (0, 0, 8, 8, 8, 1.0, A.data_ptr(), 8, B.data_ptr(), 8, 0.0, C.data_ptr(), 8)
    assert call(*args, bias.data_ptr(), 3, 0, None) == lib.SGEMM_ERR_INVALID_ARG   # unknown bias kind
    assert call(*args, bias.data_ptr(), 1, 4, None) == lib.SGEMM_ERR_INVALID_ARG   # unknown activation
    assert call(*args, bias.data_ptr(), -1, 0, None) == lib.SGEMM_ERR_INVALID_ARG
    assert call(*args, 0, 1, 2, None) == lib.SGEMM_ERR_INVALID_ARG                 # null bias
    assert call(*args, C.data_ptr() + 4 * 20, 2, 0, None) == lib.SGEMM_ERR_INVALID_ARG  # bias inside C
    assert call(*args, 0, 0, 2, None) == lib.SGEMM_OK                              # no bias: pointer unused
    torch.cuda.synchronize()


def test_torch_binding(lib):
    import torch

    _configure(lib, "auto", 0, 0, 0)
    A, B = wl.make_pair(200, 300, 128, "normal", 21)
    bias = np.random.default_rng(3).standard_normal(300).astype(np.float32)
    C = lib.gemm_fused(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(),
                       bias=torch.from_numpy(bias).cuda(), bias_kind="col", act="gelu")
    torch.cuda.synchronize()
    C64, S = oracle.gemm_f64(A, B)
    e64, eS = oracle.epilogue_f64(C64, S, bias=bias, bias_kind="col", act="gelu")
    assert oracle.normalized_error(C.cpu().numpy(), e64, eS) <= TOL


@pytest.mark.parametrize("kind,act", [("col", "gelu"), ("row", "silu"), ("col", "relu")])
def test_headline_shape_fused(lib, kind, act):
    """2048 x 3072 x 4096 (whole tiles and split tiles both occur under AUTO),
    checked at sampled outputs."""
    _configure(lib, "auto", 0, 0, 0)
    w = wl.C5_HEAD
    A, B = wl.make_inputs(w)
    bias = _bias(kind, w.M, w.N, 17)
    C, flat, rc = run_fused(A, B, bias=bias, bias_kind=KINDS[kind], act=ACTS[act])
    assert rc == 0
    r, c = wl.sample_positions(w.M, w.N, 3000, seed=5)
    c64, s = oracle.gemm_f64_at(A, B, r, c)
    e64, eS = oracle.epilogue_f64(c64, s, bias=bias, bias_kind=kind, act=act, rows=r, cols=c,
                                  shape=(w.M, w.N))
    assert oracle.normalized_error(C[r, c], e64, eS) <= TOL
    assert np.all(np.isfinite(C))


@pytest.mark.parametrize("setting", [("ffma", 1, 1, 0), ("tf32x3", 0, 1, 3), ("tf32x3", 0, 1, 4),
                                     ("tf32x3", 0, 3, 4)], ids=lambda s: "-".join(map(str, s)))
def test_gelu_pointwise(lib, setting):
    """GELU of chosen values against x * Phi(x) in double: a K = 4 product
    whose row i reproduces x_i (A row (x_i, 0, 0, 0), B all ones) feeds the
    epilogue, in the store of whole tiles and in the pass after split ones.
    The device evaluates Phi by a rational approximation with error below
    7.5e-8; the bound allows for it, the fp32 rounding of the evaluation and
    the 2^-22 relative error with which the three-term product reproduces x."""
    import math

    import torch

    _configure(lib, *setting)
    x = np.concatenate([np.linspace(-14.0, 14.0, 2801), [0.0, -0.0, 1e-30, -1e-30, 1e-7, -1e-7, 0.5, -0.5],
                        [40.0, -40.0, 1e4, -1e4, 1e30, -1e30]]).astype(np.float32)
    M, N, K = 3072, 256, 4
    xs = np.resize(x, M)
    A = np.zeros((M, K), np.float32)
    A[:, 0] = xs
    B = np.ones((K, N), np.float32)
    C = lib.gemm_fused(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), act="gelu")
    torch.cuda.synchronize()
    C = C.cpu().numpy()
    xd = xs.astype(np.float64)
    exact = np.array([v * 0.5 * (1.0 + math.erf(v / math.sqrt(2.0))) for v in xd])
    err = np.abs(C - exact[:, None])
    bound = 1e-6 * np.maximum(1.0, np.abs(xd))[:, None]
    assert np.all(err <= bound), (setting, float((err / bound).max()), xs[np.argmax((err / bound).max(axis=1))])
    # Below about -13 the product x * Phi(x) underflows to (minus) zero.
    assert np.all(C[xs < -14.5] == 0.0)
