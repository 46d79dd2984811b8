"""The tensor-core kernels' persistent schedules, checked on the CPU: a host
program built with nvcc calls make_schedule, sk_share_start and
for_each_unit_of (the code the kernels run) over a grid of tile counts,
k-block counts, slot counts, stream-K modes, K caps and switch costs, and
checks exact coverage, unit bounds and the order of the shares."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dense_fp32_matrix_major_gb300", "csrc")


def test_schedules_cover_every_k_block_once(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = tmp_path / "schedule_check"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O1", "--expt-relaxed-constexpr",
                    "-I", os.path.join(ROOT, "include"), "-I", CSRC,
                    os.path.join(ROOT, "tests", "schedule_check.cu"), "-o", str(exe)],
                   check=True, capture_output=True, text=True, timeout=600)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert "failures 0" in r.stdout
