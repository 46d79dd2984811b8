#!/usr/bin/env python3
"""Benchmark of the GB300 SGEMM: GFLOP/s (2MNK / time) and the roofline fraction.

One step = one C = A * B over the workload's seeded synthetic inputs, already
resident in HBM. Default workload: M = 2048, K = 4096, N = 3072, N(0, 1)
entries, seed 4 (the benchmark shape of "CUDA算子优化(4)：矩阵乘法"). Its
inputs and output (109 MB) fit in the 129 MB L2, so a 256 MiB buffer is
written between timed steps to flush L2; only the product is inside the
CUDA events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--variant auto|ffma|tf32x3] [--workload NAME] [--no-extras]
                    [--batched] [--fused]

Prints the headline JSON line first (rank 0): every output of the timed
product is compared with the CPU oracle, ``cpu_baseline`` is the oracle's
float loop (i-k-j order, bit-identical to the pages' i-j-k loop) on all host
cores over a bounded row sample, and ``e2e`` goes through host buffers. With
one GPU further lines follow (unless --no-extras): one per other benchmark
configuration (every output checked), the pages' single-thread CPU loop at
512^3 and 1024^3 and the 1024^2 all-ones product end to end, each beside the
figure the pages print for their own hardware. With N > 1 (torchrun, one
process per GPU) every rank runs its own replica of the workload: the product
does not shard with a data-path exchange, so there is no collective beyond
the timing barrier and the max-over-ranks reduction. ``--impl reference``
times the CPU oracle (the pages' float loop, threaded) on a bounded row
sample instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dense_fp32_matrix_major_gb300 import workloads as wl  # noqa: E402

METRIC = "SGEMM GFLOP/s (2MNK/s) on 1 GB300 and % of FP32 roofline peak"
UNIT = "GFLOP/s"
L2_FLUSH_BYTES = 256 << 20
# FP32 lanes per SM and the maximum SM clock of a GB300 (the profiling
# recipe's unit counts): the FFMA peak is SMs x 128 x 2 flops x clock.
FP32_LANES_PER_SM = 128
GB300_MAX_SM_MHZ = 2070.0
# Fallback denominators (no measured-peaks file): dense bf16 1.9 PFLOP/s burst,
# HBM 6.8 TB/s; TF32 runs at 1.1 / 2.25 of the bf16 rate (nominal ratio).
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
TF32_OVER_BF16 = 1.1 / 2.25
# Tensor-pipe rate of kind::tf32 MMAs on GB300 read from the ncu pipe counters
# (and matched by a microbenchmark of back-to-back 256 x 256 x 8 and 256 x 128
# x 8 tcgen05.mma: 1936 multiply-adds per cycle per SM at the nominal 2.07 GHz,
# i.e. 2048 at the clock the events saw): the ceiling at the sampled clock.
TF32_MACS_PER_CLK_PER_SM = 2048
# The pages' own numbers, quoted beside ours (other hardware, context only):
# "CUDA内存优化入门：从Naive到Tiled矩阵乘法" section 四, the CPU triple loop on an
# i7: ~450 ms at 512^3 and ~3600 ms at 1024^3; "CUDA 性能优化实战笔记 + C++示例
# 代码（第七章重点）" section 一, the 1024^2 all-ones program timed end to end
# (copies included) on an RTX 2060: 47.33 ms Debug, 33.37 ms Release.
PAGE_CPU_MS = {512: 450.0, 1024: 3600.0}
PAGE_E2E_MS_1024 = 33.37


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------- ranks (N > 1)


def max_over_ranks(ms: float, dist, device) -> float:
    """The slowest rank's step time (ms itself when the job has one rank)."""
    if dist is None:
        return ms
    import torch

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gflops(ws: int, flops_per_rank: float, ms_max: float) -> float:
    """Whole-job GFLOP/s: the units every rank processed over the slowest
    rank's time (each rank runs its own replica of the workload)."""
    return ws * flops_per_rank / (ms_max * 1e-3) / 1e9


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self._thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._thread:
            self._thread.join(timeout=2)

    def summary(self, t0=None, t1=None):
        """Median SM clock and throttle reasons of the samples read in [t0, t1]."""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in self.lines:
            if (t0 is not None and t < t0) or (t1 is not None and t > t1):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- peaks


def _measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


def _tf32x3_peak_tflops():
    """fp32-equivalent ceiling of the three-product TF32 path: TF32 dense / 3."""
    peaks = _measured_peaks()
    if peaks and peaks.get("bf16_tflops"):
        return float(peaks["bf16_tflops"]) * TF32_OVER_BF16 / 3.0, "measured bf16 x 1.1/2.25 / 3"
    return FALLBACK_BF16_TFLOPS * TF32_OVER_BF16 / 3.0, "fallback bf16 1.9 PF x 1.1/2.25 / 3"


def _tf32x3_pipe_ceiling(sm_count: int, sm_mhz: float):
    """fp32-equivalent ceiling from the measured tensor-pipe rate at the sampled clock."""
    tflops = sm_count * TF32_MACS_PER_CLK_PER_SM * 2 * sm_mhz * 1e6 / 1e12 / 3.0
    return tflops, (f"{sm_count} SMs x {TF32_MACS_PER_CLK_PER_SM} tf32 MAC/clk (ncu pipe counters) x 2 x "
                    f"{sm_mhz:.0f} MHz sampled / 3 products")


def _hbm_peak_gbs():
    peaks = _measured_peaks()
    if peaks and peaks.get("hbm_gbs"):
        return float(peaks["hbm_gbs"]), "measured copy bandwidth"
    return FALLBACK_HBM_GBS, "fallback 6.8 TB/s"


def _traffic_record(kernel_key: str):
    """Per-launch DRAM bytes from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            recs = json.load(f)
    except (OSError, ValueError):
        return None
    rec = recs.get(kernel_key)
    if not rec:
        return None
    h = hashlib.sha256()
    try:
        for rel in rec["sources"]:
            with open(os.path.join(ROOT, rel), "rb") as f:
                h.update(f.read())
    except OSError:
        return None
    return rec["dram_bytes_per_launch"] if h.hexdigest()[:16] == rec["sources_sha256_16"] else None


# Kernel names by the library's SGEMM_TUNE_LAST_TC_KERNEL value.
TC_KERNELS = {1: "tf32x3_kernel", 2: "tf32x3_tma_kernel", 3: "tf32x3_tmem_kernel", 4: "tf32x3_pair_kernel"}


# -------------------------------------------------------------- our arm


def _device_inputs(w, torch, device):
    A, B = _host_inputs(w)
    dA = torch.from_numpy(np.ascontiguousarray(A)).to(device)
    dB = torch.from_numpy(np.ascontiguousarray(B)).to(device)
    dC = torch.empty((w.M, w.N), dtype=torch.float32, device=device)
    return A, B, dA, dB, dC


def run_ours(args, w, torch, dist, full_parity: bool = False, with_e2e: bool = True):
    """Time sgemm_f32 on workload w (inputs resident in HBM, L2 flushed
    between steps) and check its output against the oracle: every output
    when full_parity, else seeded samples."""
    from dense_fp32_matrix_major_gb300 import sgemm

    ws, rank, local = _dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    sgemm.set_variant(args.variant)
    if args.tc_kernel is not None:
        sgemm.set_tuning(sgemm.SGEMM_TUNE_TF32X3_KERNEL, args.tc_kernel)
    A, B, dA, dB, dC = _device_inputs(w, torch, device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    def step():
        rc = sgemm.sgemm_f32_raw(w.M, w.N, w.K, dA.data_ptr(), w.K, dB.data_ptr(), w.N,
                                 dC.data_ptr(), w.N, sh)
        if rc:
            raise sgemm.SgemmError(rc, "sgemm_f32")

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    variant_used = sgemm.variant_name(sgemm.last_variant_used())
    launches_per_step = sgemm.last_launch_count()
    tc_kernel = TC_KERNELS.get(sgemm.get_tuning(sgemm.SGEMM_TUNE_LAST_TC_KERNEL), "tf32x3")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()  # L2 flush between timed steps, outside the events
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    wall1 = time.perf_counter()
    wall = wall1 - wall0
    time.sleep(0.15)  # the sample covering the end of the region is printed a little later
    sampler.stop()
    per_step = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(per_step) / len(per_step)
    ms_max = max_over_ranks(ms, dist, device)
    value = job_gflops(ws, w.flops, ms_max)

    # Parity check of the timed output (not timed): every output against the
    # threaded double oracle, or seeded samples.
    import oracle  # test infrastructure: used here only to check the result
    Cgot = dC.cpu().numpy()
    if full_parity:
        C64, S = oracle.sgemm_f64_rows(np.ascontiguousarray(A), np.ascontiguousarray(B))
        err = oracle.normalized_error(Cgot, C64, S)
        parity = {"err": err, "compared": "every output", "bound": 1e-5}
        if w.dist == "ones":
            parity["all_equal_K"] = bool(np.all(Cgot == np.float32(w.K)))
    else:
        r, c = wl.sample_positions(w.M, w.N, 64, seed=99)
        c64, s = oracle.sgemm_f64_at(A, B, r, c)
        err = oracle.normalized_error(Cgot[r, c], c64, s)
        parity = {"err": err, "compared": f"{len(r)} sampled outputs", "bound": 1e-5}

    # End to end: host buffers through the C ABI, copies inside the timed region.
    e2e = run_e2e(args, w, torch, sgemm, A, B, device, dist, ws) if with_e2e else None

    clocks = sampler.summary(wall0, wall1 + 0.12)
    sm_max = clocks["sm_max_mhz"] or GB300_MAX_SM_MHZ
    sm_count = torch.cuda.get_device_properties(device).multi_processor_count
    pipe = None
    if variant_used == "tf32x3":
        peak, peak_src = _tf32x3_peak_tflops()
        bound = "tensor"
        kernel_key = tc_kernel
        clk = clocks["sm_mhz"] or GB300_MAX_SM_MHZ
        pipe_peak, pipe_src = _tf32x3_pipe_ceiling(sm_count, clk)
    else:
        peak = sm_count * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
        peak_src = f"{sm_count} SMs x 128 FP32 lanes x 2 x {sm_max:.0f} MHz (recipe unit counts)"
        bound = "alu"
        kernel_key = "ffma_kernel"
    achieved = w.flops / (ms * 1e-3) / 1e12
    if variant_used == "tf32x3":
        pipe = {"peak": round(pipe_peak, 3), "frac": round(achieved / pipe_peak, 4), "unit": "TFLOP/s",
                "peak_source": pipe_src}
    traffic = _traffic_record(kernel_key)
    hbm_peak, hbm_src = _hbm_peak_gbs()
    algo_gbs = w.algorithmic_bytes / (ms * 1e-3) / 1e9
    hbm = {"algorithmic_gbs": round(algo_gbs, 1),
           "dram_gbs": round(traffic / (ms * 1e-3) / 1e9, 1) if traffic else None,
           "peak_gbs": hbm_peak, "peak_source": hbm_src,
           "frac": round((traffic / (ms * 1e-3) / 1e9 if traffic else algo_gbs) / hbm_peak, 4),
           "note": "compute-bound: intensity 2MNK / 4(MK+KN+MN) is far above the ridge point"}
    # The headline metric's denominator: the FP32 FFMA (CUDA-core) peak, which
    # the tensor-core variant exceeds because it does not run on that pipe.
    ffma_peak = sm_count * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
    fp32_ffma = {"peak": round(ffma_peak, 3), "frac": round(achieved / ffma_peak, 4), "unit": "TFLOP/s",
                 "peak_source": f"{sm_count} SMs x 128 FP32 lanes x 2 x {sm_max:.0f} MHz (recipe unit counts)"}
    roofline = {
        "bound": bound, "achieved": round(achieved, 3), "peak": round(peak, 3), "unit": "TFLOP/s",
        "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": kernel_key, "hbm": hbm,
        "fp32_ffma_peak": fp32_ffma,
        "tensor_pipe_ceiling": pipe,
        "peak_source": peak_src,
        "algorithmic_flops_per_launch": w.flops,
        "timing": "CUDA events around each sgemm_f32 call on its stream (includes the small "
                  "zeroing kernel when stream-K tiles exist), mean over the timed steps",
    }
    return {
        "value": value, "ms_per_step": ms_max, "wall_s": wall, "variant": variant_used,
        "launches_per_step": launches_per_step, "per_step_ms_min": min(per_step),
        "per_step_ms_median": statistics.median(per_step), "roofline": roofline, "e2e": e2e,
        "clocks": clocks, "parity": parity, "kernel": kernel_key,
    }


def run_batched_bench(args, bw, torch):
    """GFLOP/s of one strided-batched call over packed items (inputs resident,
    L2 flushed between steps), with a sampled parity check of a few items."""
    from dense_fp32_matrix_major_gb300 import sgemm
    import oracle  # test infrastructure: spot check only

    _, _, local = _dist_env()
    device = torch.device("cuda", local)
    sgemm.set_variant(args.variant)
    A, B = wl.make_batched(bw)
    dA = torch.from_numpy(A).to(device)
    dB = torch.from_numpy(B).to(device)
    dC = torch.empty((bw.batch, bw.M, bw.N), dtype=torch.float32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush.zero_()
        sgemm.gemm_batched(dA, dB, dC)
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 500))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in ev:
        flush.zero_()
        e0.record(stream)
        sgemm.gemm_batched(dA, dB, dC)
        e1.record(stream)
    torch.cuda.synchronize()
    ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps
    C = dC.cpu().numpy()
    err = 0.0
    for b in (0, bw.batch // 2, bw.batch - 1):
        r, c = wl.sample_positions(bw.M, bw.N, 32, seed=b)
        c64, s = oracle.sgemm_f64_at(A[b], B[b], r, c)
        err = max(err, oracle.normalized_error(C[b][r, c], c64, s))
    return {"workload": bw.name, "batch": bw.batch, "value": round(bw.flops / (ms * 1e-3) / 1e9, 2),
            "unit": UNIT, "ms_per_step": round(ms, 5), "variant": sgemm.variant_name(sgemm.last_variant_used()),
            "launches_per_step": sgemm.last_launch_count(), "parity_sampled_err": err}


def run_fused_bench(args, w, torch, plain_ms):
    """GFLOP/s of the fused product act(A B + bias) at workload w, one line per
    (bias kind, activation), against the plain product's time; sampled parity
    against the oracle's product followed by its epilogue."""
    from dense_fp32_matrix_major_gb300 import sgemm
    import oracle  # test infrastructure: spot check only

    _, _, local = _dist_env()
    device = torch.device("cuda", local)
    sgemm.set_variant(args.variant)
    A, B, dA, dB, dC = _device_inputs(w, torch, device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()
    out = []
    for kind, act in (("col", "gelu"), ("col", "relu"), ("row", "silu")):
        bias = (np.random.default_rng(17).standard_normal(w.N if kind == "col" else w.M)).astype(np.float32)
        dbias = torch.from_numpy(bias).to(device)
        for _ in range(args.warmup):
            flush.zero_()
            sgemm.gemm_fused(dA, dB, dC, bias=dbias, bias_kind=kind, act=act)
        torch.cuda.synchronize()
        steps = max(3, min(args.steps, 500))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            sgemm.gemm_fused(dA, dB, dC, bias=dbias, bias_kind=kind, act=act)
            e1.record(stream)
        torch.cuda.synchronize()
        ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps
        r, c = wl.sample_positions(w.M, w.N, 64, seed=7)
        c64, sc = oracle.sgemm_f64_at(A, B, r, c)
        e64, es = oracle.epilogue_f64(c64, sc, bias=bias, bias_kind=kind, act=act, rows=r, cols=c,
                                      shape=(w.M, w.N))
        err = oracle.normalized_error(dC.cpu().numpy()[r, c], e64, es)
        out.append({"workload": w.name, "epilogue": f"bias per {kind} + {act}",
                    "value": round(w.flops / (ms * 1e-3) / 1e9, 2), "unit": UNIT, "ms_per_step": round(ms, 5),
                    "plain_ms_per_step": round(plain_ms, 5), "overhead": round(ms / plain_ms - 1.0, 4),
                    "variant": sgemm.variant_name(sgemm.last_variant_used()),
                    "launches_per_step": sgemm.last_launch_count(), "parity_sampled_err": err})
    return out


def run_e2e(args, w, torch, sgemm, A, B, device, dist, ws):
    Ah = torch.from_numpy(np.ascontiguousarray(A)).pin_memory()
    Bh = torch.from_numpy(np.ascontiguousarray(B)).pin_memory()
    Ch = torch.empty((w.M, w.N), dtype=torch.float32).pin_memory()
    dA = torch.empty_like(Ah, device=device)
    dB = torch.empty_like(Bh, device=device)
    dC = torch.empty_like(Ch, device=device)
    stream = torch.cuda.current_stream()
    steps = max(3, min(args.steps, args.e2e_steps))
    for _ in range(2):
        sgemm.sgemm_f32_from_host(Ah, Bh, Ch, dA, dB, dC, stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        sgemm.sgemm_f32_from_host(Ah, Bh, Ch, dA, dB, dC, stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / steps, dist, device)
    return {
        "value": round(job_gflops(ws, w.flops, ms), 2), "unit": UNIT,
        "h2d_bytes_per_step": 4 * (w.M * w.K + w.K * w.N), "d2h_bytes_per_step": 4 * w.M * w.N,
        "ms_per_step": round(ms, 4), "steps": steps,
        "path": "sgemm_f32_from_host: pinned host A, B -> device, product, device C -> pinned host",
    }


# ------------------------------------------------------------ CPU oracle


_INPUT_CACHE = {}


def _host_inputs(w):
    if w.name not in _INPUT_CACHE:
        _INPUT_CACHE[w.name] = wl.make_inputs(w)
    return _INPUT_CACHE[w.name]


def cpu_oracle_sample(w, budget_s: float):
    """Time the oracle's float twin (the pages' loop arithmetic in i-k-j order,
    threaded by rows, bit-identical to their i-j-k loop) on all host cores,
    on the first rows of the workload, about budget_s seconds of work."""
    import oracle  # test infrastructure: timed here as the CPU baseline

    A, B = _host_inputs(w)
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    cores = os.cpu_count() or 1
    rows = min(w.M, cores)
    t0 = time.perf_counter()
    oracle.sgemm_f32_rows(A, B, 0, rows, nthreads=cores)
    t1 = time.perf_counter() - t0
    rows = int(max(1, min(w.M, rows * budget_s / max(t1, 1e-6))))
    t0 = time.perf_counter()
    oracle.sgemm_f32_rows(A, B, 0, rows, nthreads=cores)
    secs = time.perf_counter() - t0
    flops = 2 * rows * w.N * w.K
    return {
        "value": round(flops / secs / 1e9, 4), "unit": UNIT, "cores": min(cores, rows), "kind": "oracle",
        "sample": f"rows 0..{rows - 1} of A ({rows} x {w.K}) times all of B ({w.K} x {w.N}): the float "
                  f"loop in i-k-j order (bit-identical to the i-j-k loop), {min(cores, rows)} threads, "
                  f"{secs:.1f} s",
        "seconds": round(secs, 2),
    }


def cpu_pages_loop(n: int):
    """The pages' single-thread i-j-k float loop over a whole n^3 product (as
    their section 四 times it on an i7), for comparison with their figure."""
    import oracle  # test infrastructure: timed here as the pages' CPU loop

    A, B = wl.make_pair(n, n, n, "uniform01", 0)
    t0 = time.perf_counter()
    oracle.sgemm_f32(A, B)
    ms = (time.perf_counter() - t0) * 1e3
    return {"line": "pages_cpu_loop", "workload": f"sq{n}_uniform01", "ms": round(ms, 1),
            "value": round(2.0 * n ** 3 / (ms * 1e-3) / 1e9, 4), "unit": UNIT, "cores": 1,
            "kind": "oracle (float i-j-k loop, one thread)",
            "page_ms": PAGE_CPU_MS[n], "page_hardware": "Intel i7 (\"CUDA内存优化入门\" section 四)"}


def run_reference(args, w):
    ws, rank, _ = _dist_env()
    if rank != 0:
        return None
    budget = args.ref_step_seconds
    for _ in range(args.warmup):
        cpu_oracle_sample(w, budget / 4)
    vals, secs = [], 0.0
    for _ in range(args.steps):
        r = cpu_oracle_sample(w, budget)
        vals.append(r["value"])
        secs += r["seconds"]
    value = statistics.mean(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(2 * w.M * w.N * w.K / (value * 1e9) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": _config(w, "oracle"),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                         "sample": r["sample"]},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "the CPU oracle (the source pages' float loop, in i-k-j order and threaded by rows, "
                "bit-identical to their i-j-k loop), timed on a bounded row sample each step on all host "
                "cores; ms_per_step is the full workload extrapolated from the rate",
    }


def _config(w, variant):
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dist": w.dist, "seed": w.seed,
            "layout": "row-major fp32, lda=K, ldb=N, ldc=N", "variant": variant,
            "l2": "flushed between timed steps (256 MiB write); inputs+output 109 MB < 129 MB L2",
            "parallelism": "replicas (one independent product per GPU)"}


def print_extras(args, headline, torch):
    """One line per other benchmark configuration (every output checked), the
    pages' single-thread CPU loop at 512^3 and 1024^3, and the 1024^2 all-ones
    product end to end beside the pages' figure."""
    from dense_fp32_matrix_major_gb300 import sgemm

    for other in wl.ALL:
        if other is headline:
            continue
        sub = argparse.Namespace(**vars(args))
        sub.steps = min(args.steps, 200)
        r = run_ours(sub, other, torch, None, full_parity=True, with_e2e=False)
        roof = r["roofline"]
        print(json.dumps({
            "line": "config", "workload": other.name, "config": _config(other, r["variant"]),
            "value": round(r["value"], 2), "unit": UNIT, "ms_per_step": round(r["ms_per_step"], 5),
            "variant": r["variant"], "kernel": r["kernel"], "launches_per_step": r["launches_per_step"],
            "roofline_frac": roof["frac"], "roofline_peak": roof["peak"],
            "tensor_pipe_frac": roof["tensor_pipe_ceiling"]["frac"] if roof["tensor_pipe_ceiling"] else None,
            "fp32_ffma_frac": roof["fp32_ffma_peak"]["frac"], "parity": r["parity"],
            "clocks": r["clocks"]}), flush=True)
    for n in (512, 1024):
        print(json.dumps(cpu_pages_loop(n)), flush=True)
    # The all-ones 1024^2 product through host buffers, copies included, as the
    # pages time their program end to end.
    ones = wl.C2_ONES
    A, B = _host_inputs(ones)
    device = torch.device("cuda", torch.cuda.current_device())
    sub = argparse.Namespace(**vars(args))
    sgemm.set_variant(args.variant)
    e = run_e2e(sub, ones, torch, sgemm, A, B, device, None, 1)
    print(json.dumps({"line": "pages_e2e", "workload": ones.name, "ms": e["ms_per_step"], "value": e["value"],
                      "unit": UNIT, "h2d_bytes_per_step": e["h2d_bytes_per_step"],
                      "d2h_bytes_per_step": e["d2h_bytes_per_step"], "path": e["path"],
                      "page_ms": PAGE_E2E_MS_1024,
                      "page_hardware": "RTX 2060 (\"CUDA 性能优化实战笔记\" section 一, Release build)"}),
          flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--variant", default="auto", choices=["auto", "ffma", "tf32x3"])
    ap.add_argument("--workload", default=wl.C5_HEAD.name, choices=sorted(wl.BY_NAME))
    ap.add_argument("--tc-kernel", type=int, default=None, choices=[0, 1, 2, 3, 4, 5],
                    help="tensor-core kernel for 16-byte-aligned operands (library tuning key)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-step-seconds", type=float, default=4.0)
    ap.add_argument("--no-extras", action="store_true",
                    help="print only the headline line (by default, with one GPU, one more line per "
                         "benchmark configuration, the pages' CPU loop at 512^3 and 1024^3, and the "
                         "1024^2 all-ones product end to end follow it)")
    ap.add_argument("--all-configs", action="store_true", help=argparse.SUPPRESS)  # the default now
    ap.add_argument("--batched", action="store_true",
                    help="also print one extra line per strided-batched workload")
    ap.add_argument("--fused", action="store_true",
                    help="also print one extra line per fused epilogue (bias + activation) at the workload")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = wl.BY_NAME[args.workload]
    ws, rank, local = _dist_env()

    if args.impl == "reference":
        res = run_reference(args, w)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    import torch

    dist = None
    if ws > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    res = run_ours(args, w, torch, dist, full_parity=(ws == 1))
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(res["value"], 2), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["ms_per_step"], 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded numpy PCG64, N(0,1))",
            "config": _config(w, res["variant"]),
            "roofline": res["roofline"],
            "e2e": res["e2e"],
            "gpu_launches": res["launches_per_step"] * args.steps,
            "clocks": res["clocks"],
            "per_step_ms": {"mean": round(res["ms_per_step"], 5), "min": round(res["per_step_ms_min"], 5),
                            "median": round(res["per_step_ms_median"], 5)},
            "parity": res["parity"],
        }
        line["cpu_baseline"] = cpu_oracle_sample(w, args.cpu_seconds) if ws == 1 else None
        print(json.dumps(line), flush=True)
        if ws == 1 and not args.no_extras:
            print_extras(args, w, torch)
        if args.batched:
            for bw in wl.BATCHED:
                print(json.dumps(run_batched_bench(args, bw, torch)), flush=True)
        if args.fused:
            for line in run_fused_bench(args, w, torch, res["ms_per_step"]):
                print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
