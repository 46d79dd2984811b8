"""GPU parity: the CUDA library against the CPU oracle, element by element.

Acceptance: max |C_gpu - C64| / sum_k |A||B| <= 1e-5 (C64 = the oracle's
double-accumulating product), bit-exact where every product and partial sum
is an integer below 2^24, and no write outside the M x N box of C.
"""

import itertools

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_major_gb300 import workloads as wl
from tests.gpu_harness import TOL, outside_box_intact, oracle_error, run_sgemm, sampled_error

pytestmark = pytest.mark.gpu

# (variant, ffma tile, stream-K mode, tensor-core kernel) settings every
# small-shape test runs under. Tensor-core kernels: 0 = automatic,
# 1 = per-thread loads, 2 = TMA, 3 = TMA with A in tensor memory, 4 = SM pairs.
SETTINGS = [
    ("auto", 0, 0, 0),
    ("ffma", 1, 1, 0), ("ffma", 1, 3, 0), ("ffma", 2, 2, 0), ("ffma", 3, 0, 0), ("ffma", 2, 3, 0),
    ("tf32x3", 0, 0, 0), ("tf32x3", 0, 0, 3), ("tf32x3", 0, 1, 3), ("tf32x3", 0, 3, 3),
    ("tf32x3", 0, 0, 2), ("tf32x3", 0, 3, 2), ("tf32x3", 0, 0, 1), ("tf32x3", 0, 3, 1),
    ("tf32x3", 0, 0, 4), ("tf32x3", 0, 1, 4), ("tf32x3", 0, 3, 4),
]
SETTING_IDS = [f"{s[0]}-t{s[1]}-sk{s[2]}-k{s[3]}" for s in SETTINGS]


@pytest.fixture(scope="module")
def lib():
    import torch

    assert torch.cuda.is_available()
    from dense_fp32_matrix_major_gb300 import sgemm

    yield sgemm
    sgemm.set_variant(0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_FFMA_TILE, 0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_STREAM_K, 0)
    sgemm.set_tuning(sgemm.SGEMM_TUNE_TF32X3_KERNEL, 0)


def _apply(lib, setting):
    variant, tile, sk = setting[:3]
    tc = setting[3] if len(setting) > 3 else 0
    lib.set_variant(variant)
    lib.set_tuning(lib.SGEMM_TUNE_FFMA_TILE, tile)
    lib.set_tuning(lib.SGEMM_TUNE_STREAM_K, sk)
    lib.set_tuning(lib.SGEMM_TUNE_TF32X3_KERNEL, tc)


def _check(A, B, C, flat, ldc, offset=0, exact=False):
    M, N = C.shape
    assert outside_box_intact(flat, M, N, ldc, offset), "write outside the M x N box"
    if exact:
        ref = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float32)
        assert np.array_equal(C, ref)
    else:
        err = oracle_error(C, A, B)
        assert err <= TOL, err


TINY = [1, 2, 3, 5, 8, 13, 16, 17]


@pytest.mark.parametrize("setting", SETTINGS, ids=SETTING_IDS)
def test_tiny_shape_sweep(lib, setting):
    _apply(lib, setting)
    for M, N, K in itertools.product(TINY, TINY, TINY):
        A, B = wl.make_pair(M, N, K, "normal", M * 1000 + N * 10 + K)
        C, flat, rc = run_sgemm(A, B)
        assert rc == 0, (M, N, K)
        _check(A, B, C, flat, max(N, 1))


TILE_EDGES = [(63, 65, 15), (64, 64, 16), (65, 63, 17), (127, 255, 31), (128, 256, 33),
              (129, 257, 47), (1, 300, 100), (300, 1, 100), (200, 3, 1), (33, 257, 513)]


@pytest.mark.parametrize("setting", SETTINGS, ids=SETTING_IDS)
@pytest.mark.parametrize("M,N,K", TILE_EDGES)
def test_tile_boundary_crossings(lib, setting, M, N, K):
    _apply(lib, setting)
    A, B = wl.make_pair(M, N, K, "uniform", M + N + K)
    C, flat, rc = run_sgemm(A, B)
    assert rc == 0
    _check(A, B, C, flat, N)


@pytest.mark.parametrize("setting", SETTINGS, ids=SETTING_IDS)
def test_integer_inputs_bit_exact(lib, setting):
    _apply(lib, setting)
    for (M, N, K) in [(257, 129, 1000), (64, 300, 4096), (1000, 40, 77)]:
        A, B = wl.make_pair(M, N, K, "int4", K)
        C, flat, rc = run_sgemm(A, B)
        assert rc == 0
        _check(A, B, C, flat, N, exact=True)


@pytest.mark.parametrize("setting", SETTINGS, ids=SETTING_IDS)
def test_padded_strides_and_unaligned_pointers(lib, setting):
    _apply(lib, setting)
    M, N, K = 150, 270, 90
    A, B = wl.make_pair(M, N, K, "normal", 21)
    cases = [
        dict(lda=K + 6, ldb=N + 2, ldc=N + 10, offsets=(0, 0, 0)),   # padded rows
        dict(lda=K + 1, ldb=N + 1, ldc=N + 3, offsets=(1, 3, 1)),   # no 16-byte alignment anywhere
        dict(lda=K, ldb=N + 4, ldc=N + 4, offsets=(2, 4, 8)),        # aligned B and C, odd A
    ]
    for case in cases:
        C, flat, rc = run_sgemm(A, B, **case)
        assert rc == 0, case
        _check(A, B, C, flat, case["ldc"], case["offsets"][2])


def test_special_cases(lib):
    _apply(lib, ("auto", 0, 0))
    # K = 0: the empty sum, C becomes zero.
    A = np.zeros((5, 0), np.float32)
    B = np.zeros((0, 7), np.float32)
    C, flat, rc = run_sgemm(A, B)
    assert rc == 0 and np.all(C == 0) and outside_box_intact(flat, 5, 7, 7, 0)
    # M = 0 and N = 0: nothing is written.
    for (M, N, K) in [(0, 7, 3), (4, 0, 3), (0, 0, 0)]:
        A = np.ones((M, K), np.float32)
        B = np.ones((K, N), np.float32)
        C, flat, rc = run_sgemm(A, B, prefill=np.float32(7777.25))
        assert rc == 0
        assert np.all(flat == np.float32(7777.25))
    # Single nonzero term and identity: every output is one product plus
    # exact zeros, so FFMA reproduces B bit for bit. The three-term TF32 split
    # carries B's bits to 2^-22 of each value (hi + rounded lo), within the bound.
    A1 = np.zeros((70, 40), np.float32)
    A1[33, 17] = -0.5
    B1 = np.random.default_rng(5).standard_normal((40, 90)).astype(np.float32)
    exp = np.zeros((70, 90), np.float32)
    exp[33] = -0.5 * B1[17]
    I = np.eye(300, dtype=np.float32)
    B2 = np.random.default_rng(6).standard_normal((300, 200)).astype(np.float32)
    for variant in ("ffma", "tf32x3", "auto"):
        _apply(lib, (variant, 0, 0))
        C1, flat, rc1 = run_sgemm(A1, B1)
        C2, flat, rc2 = run_sgemm(I, B2)
        assert rc1 == 0 and rc2 == 0
        if lib.variant_name(lib.last_variant_used()) == "ffma":
            assert np.array_equal(C1, exp) and np.array_equal(C2, B2)
        else:
            assert oracle_error(C1, A1, B1) <= TOL and oracle_error(C2, I, B2) <= TOL
            assert np.max(np.abs(C2 - B2) / np.maximum(np.abs(B2), 1e-30)) <= 2.0**-21


def test_status_codes_on_device(lib):
    import torch

    a = torch.zeros(16, device="cuda")
    # C overlapping A is rejected.
    assert lib.sgemm_f32_raw(2, 2, 2, a.data_ptr(), 2, a.data_ptr() + 64, 2, a.data_ptr() + 4, 2, 0) == 1
    assert lib.device_status() == 0


# ------------------------------------------------------------- benchmark configs


_config_oracle = {}


def _config_reference(w):
    """(A, B, C64, S) of a benchmark workload: the full double product from the
    threaded oracle, computed once per workload and shared by every variant."""
    if w.name not in _config_oracle:
        A, B = wl.make_inputs(w)
        C64, S = oracle.sgemm_f64_rows(A, B)
        _config_oracle[w.name] = (A, B, C64, S)
    return _config_oracle[w.name]


@pytest.mark.parametrize("w", wl.ALL, ids=lambda w: w.name)
@pytest.mark.parametrize("variant,tc", [("auto", 0), ("ffma", 0), ("tf32x3", 3), ("tf32x3", 2), ("tf32x3", 1),
                                        ("tf32x3", 4)])
def test_benchmark_configs(lib, w, variant, tc):
    """Every output of every benchmark configuration against the oracle (the
    headline is the shape of "CUDA算子优化(4)：矩阵乘法", host code of the V1
    kernel: M = 2048, K = 4096, N = 3072)."""
    _apply(lib, (variant, 0, 0, tc))
    A, B, C64, S = _config_reference(w)
    C, flat, rc = run_sgemm(A, B, lda=w.lda, ldb=w.ldb, ldc=w.ldc)
    assert rc == 0
    assert outside_box_intact(flat, w.M, w.N, w.ldc or w.N, 0)
    if w.dist == "ones":
        assert np.all(C == np.float32(w.K))  # the page's closed form: every output is K
    err = oracle.normalized_error(C, C64, S)
    assert err <= TOL, err


def test_from_host_entry_point(lib):
    import torch

    w = wl.C3_RAGGED
    A, B, _, _ = _config_reference(w)
    Ah = torch.from_numpy(A).pin_memory()
    Bh = torch.from_numpy(B).pin_memory()
    Ch = torch.full((w.M, w.N), float("nan")).pin_memory()
    dA, dB, dC = (torch.empty_like(t, device="cuda") for t in (Ah, Bh, Ch))
    lib.set_variant(0)
    lib.sgemm_f32_from_host(Ah, Bh, Ch, dA, dB, dC)
    torch.cuda.synchronize()
    _, _, C64, S = _config_reference(w)
    assert oracle.normalized_error(Ch.numpy(), C64, S) <= TOL


@pytest.mark.parametrize("w", [wl.C5_HEAD, wl.C4_2048], ids=lambda w: w.name)
def test_from_host_pipelined_on_side_stream(lib, w):
    """Large products go through the column-panel pipeline (library streams);
    the call on a side stream must still order everything before that
    stream's later work, and every panel, the last one included, is right."""
    import torch

    A, B, _, _ = _config_reference(w)
    Ah = torch.from_numpy(A).pin_memory()
    Bh = torch.from_numpy(B).pin_memory()
    Ch = torch.full((w.M, w.N), float("nan")).pin_memory()
    dA, dB, dC = (torch.empty_like(t, device="cuda") for t in (Ah, Bh, Ch))
    lib.set_variant(0)
    side = torch.cuda.Stream()
    for _ in range(2):  # a second call reuses the library's streams and events
        Ch.fill_(float("nan"))
        lib.sgemm_f32_from_host(Ah, Bh, Ch, dA, dB, dC, stream=side)
        side.synchronize()
        C = Ch.numpy()
        _, _, C64, S = _config_reference(w)
        assert oracle.normalized_error(C, C64, S) <= TOL  # every panel, every output


def test_repeat_calls_are_stable(lib):
    """Stream-K adds partial sums with atomics: repeated runs stay within the bound."""
    _apply(lib, ("ffma", 1, 3))
    A, B = wl.make_pair(256, 512, 2048, "normal", 77)
    C64, S = oracle.sgemm_f64_rows(A, B)
    for _ in range(3):
        C, flat, rc = run_sgemm(A, B)
        assert rc == 0
        assert oracle.normalized_error(C, C64, S) <= TOL


def test_tf32x3_long_k_margin(lib):
    """The tensor core truncates each accumulation, so a long chain of MMAs
    into one accumulator would drift; at K = 8192 the result must still meet
    the bound."""
    _apply(lib, ("tf32x3", 0, 0))
    A, B = wl.make_pair(256, 512, 8192, "normal", 88)
    C, flat, rc = run_sgemm(A, B)
    assert rc == 0
    r, c = wl.sample_positions(256, 512, 3000, seed=2)
    assert sampled_error(C, A, B, r, c) <= TOL


@pytest.mark.parametrize("variant,tc", [("auto", 0), ("tf32x3", 1), ("tf32x3", 3), ("tf32x3", 4)])
@pytest.mark.parametrize("K", [8193, 20000, 40000])
def test_tf32x3_beyond_k_8192(lib, variant, tc, K):
    """However long K gets, no tensor-core accumulator chains more than a
    few k-blocks of MMAs before its value is added, rounded to nearest, into
    an fp32 sum, so the error stays at the short-K level (one accumulator
    over all of K would drift about linearly with K)."""
    _apply(lib, (variant, 0, 0, tc))
    M, N = 256, 512
    A, B = wl.make_pair(M, N, K, "normal", K)
    C, flat, rc = run_sgemm(A, B)
    assert rc == 0
    assert lib.variant_name(lib.last_variant_used()) == "tf32x3"
    assert outside_box_intact(flat, M, N, N, 0)
    r, c = wl.sample_positions(M, N, 1500, seed=K)
    err = sampled_error(C, A, B, r, c)
    assert err <= 5e-6, err  # half the bound: the split keeps the K = 4096 error
    # Integer inputs stay exact through the split and the atomic adds.
    Ai, Bi = wl.make_pair(M, N, K, "int4", K + 1)
    Ci, _, rc = run_sgemm(Ai, Bi)
    assert rc == 0
    exact = (Ai.astype(np.int64)[:8] @ Bi.astype(np.int64)).astype(np.float32)
    assert np.array_equal(Ci[:8], exact)


def test_nonfinite_inputs_propagate(lib):
    """Non-finite inputs reach exactly the outputs that use them, with IEEE
    results on both variants: an infinity times positive values gives +inf
    (the TF32 split's NaN is recomputed; the planted cases of every rule are
    in test_nonfinite_gpu.py)."""
    for variant in ("ffma", "tf32x3"):
        _apply(lib, (variant, 0, 0))
        A = np.ones((130, 40), np.float32)
        B = np.ones((40, 260), np.float32)
        A[5, 3] = np.inf
        A[77, 0] = np.nan
        C, flat, rc = run_sgemm(A, B)
        assert rc == 0
        assert np.all(np.isposinf(C[5]))
        assert np.all(np.isnan(C[77]))
        rest = np.delete(C, [5, 77], axis=0)
        assert np.all(rest == 40.0)


def test_bounded_wait_reports_timeout(lib):
    """A wait that can never complete gives up, reports SGEMM_ERR_TIMEOUT once,
    and leaves the context usable."""
    import time

    assert lib.device_status() == 0
    t0 = time.perf_counter()
    lib.watchdog_selftest(200)
    assert lib.device_status() == lib.SGEMM_ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 0.15
    assert lib.device_status() == 0  # read-and-clear
    _apply(lib, ("auto", 0, 0))
    A, B = wl.make_pair(300, 500, 700, "normal", 4)
    C, flat, rc = run_sgemm(A, B)
    assert rc == 0 and oracle_error(C, A, B) <= TOL
    assert lib.sgemm_f32_raw(1, 1, 1, 0, 1, 0, 1, 0, 1, 0) == lib.SGEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("setting", [("auto", 0, 0, 0), ("tf32x3", 0, 3, 3), ("ffma", 1, 0, 0)],
                         ids=["auto-pair", "tmem-sk3", "ffma"])
def test_output_beyond_2_31_elements(lib, setting):
    """C with more than 2^31 elements (66000 x 32772, 8.7 GB): element offsets
    past 32 bits in every index path of the kernels and passes. Checked at
    sampled outputs (random, the rows around offset 2^31, the last rows and
    columns) and on a guard row after C that must stay untouched."""
    import torch

    _apply(lib, setting)
    M, N, K = 66000, 32772, 68
    assert M * N > 2**31
    A, B = wl.make_pair(M, N, K, "normal", 31)
    flat = torch.full(((M + 1) * N,), float("nan"), dtype=torch.float32, device="cuda")
    C = flat[: M * N].view(M, N)
    lib.gemm(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), C)
    torch.cuda.synchronize()
    assert bool(torch.isnan(flat[M * N:]).all()), "write past the last row"
    r0 = 2**31 // N
    rows = [np.repeat(np.arange(r0 - 2, r0 + 3), 64), np.repeat(np.arange(M - 3, M), 64)]
    cols = [np.tile(np.linspace(0, N - 1, 64).astype(np.int64), 5), np.tile(np.linspace(0, N - 1, 64).astype(np.int64), 3)]
    rr, cc = wl.sample_positions(M, N, 4000, seed=13)
    r = np.concatenate([rr] + rows)
    c = np.concatenate([cc] + cols)
    vals = C[torch.from_numpy(r).cuda(), torch.from_numpy(c).cuda()].cpu().numpy()
    c64, s = oracle.sgemm_f64_at(A, B, r, c)
    assert oracle.normalized_error(vals, c64, s) <= TOL
    del flat, C
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M,N,K,lda_pad,variant,tc", [
    (16, 16, 16, 0, "ffma", 0),        # tiniest products stay on the CUDA cores
    (64, 64, 64, 0, "tf32x3", 3),      # from 2^14 useful multiply-adds: tensor cores, single SM
    (128, 128, 64, 0, "tf32x3", 4),    # from 2^20: SM pairs
    (512, 512, 512, 0, "tf32x3", 4),
    (768, 768, 1024, 0, "tf32x3", 4),
    (2048, 3072, 4096, 0, "tf32x3", 4),
    (200, 4096, 4096, 0, "tf32x3", 4),  # thin products too
    (300, 300, 301, 1, "tf32x3", 1),    # rows not 16-byte aligned, small: per-thread loads
    (1023, 1025, 1301, 1, "tf32x3", 4),  # from 1.25 * 2^30: aligned copies, then SM pairs
])
def test_auto_dispatch(lib, M, N, K, lda_pad, variant, tc):
    """AUTO's choice of variant and tensor-core kernel (SGEMM_TUNE_LAST_TC_KERNEL)
    at the switch points measured on GB300, and a correct result there."""
    _apply(lib, ("auto", 0, 0, 0))
    A, B = wl.make_pair(M, N, K, "normal", 61)
    C, flat, rc = run_sgemm(A, B, lda=K + lda_pad if lda_pad else None)
    assert rc == 0
    assert lib.variant_name(lib.last_variant_used()) == variant
    if variant == "tf32x3":
        assert lib.get_tuning(lib.SGEMM_TUNE_LAST_TC_KERNEL) == tc
    r, c = wl.sample_positions(M, N, 500, seed=3)
    assert sampled_error(C, A, B, r, c) <= TOL
