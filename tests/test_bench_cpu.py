"""The bench's reference arm (the CPU oracle timed on a bounded sample) and
its command-line contract, on the CPU: the JSON line's keys, its metric and
unit (the same as the GPU arm's), zero host-device bytes for a CPU program,
silence on ranks other than 0, and the warm-up floor."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BENCH = os.path.join(ROOT, "bench.py")


def _run(args, env_extra=None, timeout=300):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, BENCH] + args, capture_output=True, text=True, cwd=ROOT, env=env,
                          timeout=timeout)


@pytest.fixture(scope="module")
def bench_module():
    sys.path.insert(0, ROOT)
    import bench

    return bench


def test_reference_arm_line(bench_module):
    r = _run(["--impl", "reference", "--steps", "3", "--warmup", "3", "--ref-step-seconds", "0.2",
              "--workload", "sq512_normal_s0"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["metric"] == bench_module.METRIC and d["unit"] == bench_module.UNIT
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"]["workload"] == "sq512_normal_s0"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert isinstance(cb["sample"], str) and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    r = _run(["--impl", "reference", "--steps", "3", "--warmup", "3", "--ref-step-seconds", "0.2",
              "--workload", "sq512_normal_s0"], {"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_warmup_below_three_is_refused():
    r = _run(["--impl", "reference", "--steps", "3", "--warmup", "2"])
    assert r.returncode != 0
    assert "warmup" in r.stderr
