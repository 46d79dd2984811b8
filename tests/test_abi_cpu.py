"""The C-ABI library without a GPU: it loads, exports every declared symbol,
and rejects bad arguments before touching a device."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    with open(os.path.join(ROOT, "include", "sgemm.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sgemm_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def binding():
    from dense_fp32_matrix_major_gb300 import _build

    _build.build()
    from dense_fp32_matrix_major_gb300 import sgemm

    return sgemm


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("sgemm_f32", "sgemm_set_variant", "sgemm_get_variant", "sgemm_variant_name",
                     "sgemm_last_variant_used", "sgemm_strerror"):
        assert required in names


def test_library_exports_every_declared_symbol(binding):
    lib = ctypes.CDLL(binding.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    # The binding wraps exactly the declared set.
    assert set(binding.SIGNATURES) == set(_declared_functions())


def test_status_and_variant_names(binding):
    assert binding.strerror(0) == "success"
    assert "invalid" in binding.strerror(1)
    assert binding.strerror(99) == "unknown status"
    assert [binding.variant_name(v) for v in (0, 1, 2, 7)] == ["auto", "ffma", "tf32x3", "unknown"]
    assert binding.version().count(".") == 2


def test_variant_selector_roundtrip(binding):
    old = binding.get_variant()
    try:
        for v in (1, 2, 0):
            binding.set_variant(v)
            assert binding.get_variant() == v
        with pytest.raises(binding.SgemmError):
            binding.set_variant(5)
        assert binding.get_variant() == 0
    finally:
        binding.set_variant(old)


def test_watchdog_selftest_rejects_bad_limits(binding):
    # Range checks run before any device work.
    assert binding.lib.sgemm_watchdog_selftest(0, None) == binding.SGEMM_ERR_INVALID_ARG
    assert binding.lib.sgemm_watchdog_selftest(60001, None) == binding.SGEMM_ERR_INVALID_ARG


def test_tuning_keys(binding):
    assert binding.get_tuning(99) == -1
    binding.set_tuning(binding.SGEMM_TUNE_FFMA_TILE, 2)
    assert binding.get_tuning(binding.SGEMM_TUNE_FFMA_TILE) == 2
    binding.set_tuning(binding.SGEMM_TUNE_FFMA_TILE, 0)
    with pytest.raises(binding.SgemmError):
        binding.set_tuning(binding.SGEMM_TUNE_STREAM_K, 9)
    with pytest.raises(binding.SgemmError):
        binding.set_tuning(binding.SGEMM_TUNE_WATCHDOG_MS, 0)
    assert binding.get_tuning(binding.SGEMM_TUNE_WATCHDOG_MS) == 2000


@pytest.mark.parametrize(
    "args",
    [
        (-1, 4, 4, 0x1000, 4, 0x2000, 4, 0x3000, 4),  # negative M
        (4, 4, 4, 0x1000, 3, 0x2000, 4, 0x3000, 4),  # lda < K
        (4, 4, 4, 0x1000, 4, 0x2000, 3, 0x3000, 4),  # ldb < N
        (4, 4, 4, 0x1000, 4, 0x2000, 4, 0x3000, 3),  # ldc < N
        (4, 4, 4, 0, 4, 0x2000, 4, 0x3000, 4),  # NULL A with elements
        (4, 4, 4, 0x1000, 4, 0, 4, 0x3000, 4),  # NULL B with elements
        (4, 4, 4, 0x1000, 4, 0x2000, 4, 0, 4),  # NULL C with elements
        (4, 4, 4, 0x1000, 4, 0x2000, 4, 0x1008, 4),  # C overlaps A
        (4, 4, 4, 0x1000, 4, 0x2000, 4, 0x1FF0, 4),  # C overlaps B (ends inside B)
    ],
)
def test_invalid_arguments_rejected_without_device(binding, args):
    # Argument checks run before any CUDA call, so these work on a CPU-only host;
    # the fixed-scratch entry point takes the same arguments and checks.
    assert binding.sgemm_f32_raw(*args, 0) == binding.SGEMM_ERR_INVALID_ARG
    assert binding.sgemm_f32_noalloc_raw(*args, 0) == binding.SGEMM_ERR_INVALID_ARG


def test_noalloc_status_and_limit(binding):
    assert "scratch" in binding.strerror(binding.SGEMM_ERR_SCRATCH)
    assert binding.SGEMM_NOALLOC_SCRATCH_BYTES == 64 << 20


def _header_enums():
    with open(os.path.join(ROOT, "include", "sgemm.h")) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return {name: int(value) for name, value in re.findall(r"\b(SGEMM_[A-Z0-9_]+)\s*=\s*(-?\d+)", text)}


def test_binding_constants_match_the_header(binding):
    """Every enumerator of sgemm.h has the same value in the Python binding,
    and the binding's name maps use those values."""
    enums = _header_enums()
    assert len(enums) >= 20
    for name, value in enums.items():
        assert getattr(binding, name) == value, name
    assert binding.BIAS_KINDS["col"] == enums["SGEMM_BIAS_PER_COL"]
    assert binding.BIAS_KINDS["row"] == enums["SGEMM_BIAS_PER_ROW"]
    assert binding.ACTIVATIONS["gelu"] == enums["SGEMM_ACT_GELU"]
    assert binding.ACTIVATIONS["silu"] == enums["SGEMM_ACT_SILU"]
    assert binding.ACTIVATIONS["relu"] == enums["SGEMM_ACT_RELU"]
