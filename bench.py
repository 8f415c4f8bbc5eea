#!/usr/bin/env python3
"""Benchmark of the GB300 Ozaki-II FP64 GEMM.

Metric: effective FP64 TFLOPS = 2pqr / time of one ozaki2_dgemm call, on the
n = 8192, s = 14, fast workload (the study's headline configuration), with
the per-stage milliseconds of the same calls.  One step = one full call
(scaling, residues, the s modular GEMMs, CRT) on inputs already in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--s S] [--mode M]
    python bench.py --impl reference ...   # the native CPU oracle on a bounded sample
    python bench.py --sweep                # ms per call and per stage over s, n and mode

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the method has no exchange step on one problem; weak scaling); the timed
region is bracketed by barriers and the slowest rank's time is reported.
One JSON line is printed by rank 0.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import HEADLINE, WORKLOADS, make_workload  # noqa: E402

METRIC = "effective FP64 TFLOPS (2pqr/time), Ozaki-II n=8192 s=14 fast; per-stage ms"
# the committed ncu summary that gives the GEMM stage's DRAM traffic covers this workload only
GEMM_PROFILE_WORKLOAD = "n8192_s14_fast"


def metric_name(workload) -> str:
    """The headline metric string; other workloads name their own shape and mode."""
    w = WORKLOADS[workload] if isinstance(workload, str) else workload
    if w == WORKLOADS[HEADLINE]:
        return METRIC
    return (f"effective FP64 TFLOPS (2pqr/time), Ozaki-II p={w.p} q={w.q} r={w.r} s={w.s} {w.mode}; "
            "per-stage ms")
UNIT = "TFLOP/s"
# Published number for this metric and workload: GH200, fast-14, n=8192
# ("Ozaki II supplement: INT8 range conditions and paper performance results", §3.1 Table 3).
PAGES_BASELINE = {"n8192_s14_fast": 72.1}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_PROFILE = os.path.join(ROOT, "profiles", "oz2_gemm_kernel_n8192_s14_fast.md")
# the GEMM kernel's source files, hashed in this order against the summary's source_sha256
GEMM_SOURCES = [os.path.join(ROOT, "emulated_fp64_gemm_gb300", "csrc", f)
                for f in ("oz2_gemm.cu", "oz2_tcgen05.cuh")]
# rows of A and columns of B in each step of the reference arm's bounded sample
REF_SAMPLE = 2048
# sampled outputs of the accuracy report
ACCURACY_SAMPLES = 4096
# the native oracle's exact integer products (the C loops or an exact float64 BLAS product)
ORACLE_PRODUCTS = "blas"
# bytes per stored residue: the planes are fp16 (integer residues, exact in fp16)
PLANE_BYTES = 2
# the library's one-read kernels: A's statistics and residues together for q <= 2048,
# B's for q <= 8192 (fast mode); a stage's algorithmic bytes follow what it runs
ROWS_FUSED_MAX_Q, COLS_FUSED_MAX_Q = 2048, 8192
SWEEP_S = (2, 4, 6, 8, 10, 12, 14, 16, 18, 20)
SWEEP_N = (1024, 2048, 8192)


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--s", type=int, default=None, help="number of moduli (overrides the workload's)")
    ap.add_argument("--mode", choices=["fast", "accu"], default=None, help="bound mode (overrides the workload's)")
    ap.add_argument("--sweep", action="store_true",
                    help="time every s in %s at n in %s, fast and accu (one JSON line each)" % (SWEEP_S, SWEEP_N))
    ap.add_argument("--sweep-n", type=str, default=None,
                    help="comma-separated n for --sweep (default %s)" % ",".join(map(str, SWEEP_N)))
    ap.add_argument("--sweep-s", type=str, default=None,
                    help="comma-separated s for --sweep (default %s)" % ",".join(map(str, SWEEP_S)))
    ap.add_argument("--stages-once", action="store_true",
                    help="one call of the stage-timed entry point (each stage alone), e.g. under a profiler")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-context", action="store_true",
                    help="skip the native cuBLAS DGEMM timing reported as context")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------- helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def gemm_source_sha256():
    h = hashlib.sha256()
    for path in GEMM_SOURCES:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def gemm_traffic_per_unit():
    """DRAM bytes of the GEMM stage of one call (all its GEMM launches) from the
    committed ncu summary, or None when the kernel source changed since the
    counters were taken."""
    try:
        text = open(GEMM_PROFILE).read()
        src = gemm_source_sha256()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_call:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not m or not h or h.group(1) != src:
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.seek(0)
        mhz, maxes, reasons = [], [], set()
        for line in self.out.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(mhz)}


def cublas_emulated_dgemm_ms(dA, dB, dC, p, q, r, stream, reps):
    """Time cuBLAS's own fixed-point FP64 emulation (compute type
    CUBLAS_COMPUTE_64F_EMULATED_FIXEDPOINT, emulation math mode, eager
    strategy) on the same column-major operands, as context.  A library call
    through ctypes; returns (ms per call, None) or (None, reason)."""
    import ctypes

    import torch
    cb = None
    for name in ("libcublas.so.13", "/usr/local/cuda/lib64/libcublas.so.13"):
        try:
            cb = ctypes.CDLL(name)
            break
        except OSError:
            continue
    if cb is None:
        return None, "libcublas.so.13 not found"
    vp, ci = ctypes.c_void_p, ctypes.c_int
    h = vp()
    if cb.cublasCreate_v2(ctypes.byref(h)) != 0:
        return None, "cublasCreate failed"
    try:
        cb.cublasGemmEx.argtypes = [vp, ci, ci, ci, ci, ci, vp, vp, ci, ci, vp, ci, ci, vp, vp, ci, ci, ci, ci]
        one, zero = ctypes.c_double(1.0), ctypes.c_double(0.0)
        CUDA_R_64F, COMPUTE_64F_EMULATED_FIXEDPOINT, FP64_EMULATED_FIXEDPOINT_MATH, EAGER = 1, 79, 8, 2
        if (cb.cublasSetStream_v2(h, vp(stream.cuda_stream)) != 0
                or cb.cublasSetMathMode(h, FP64_EMULATED_FIXEDPOINT_MATH) != 0
                or cb.cublasSetEmulationStrategy(h, EAGER) != 0):
            return None, "cuBLAS emulation settings refused"

        def call():
            return cb.cublasGemmEx(h, 0, 0, p, r, q, ctypes.cast(ctypes.byref(one), vp), vp(dA.data_ptr()),
                                   CUDA_R_64F, p, vp(dB.data_ptr()), CUDA_R_64F, q,
                                   ctypes.cast(ctypes.byref(zero), vp), vp(dC.data_ptr()), CUDA_R_64F, p,
                                   COMPUTE_64F_EMULATED_FIXEDPOINT, -1)
        if call() != 0:
            return None, "cublasGemmEx with the emulated compute type failed"
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(reps):
            call()
        c1.record(stream)
        torch.cuda.synchronize()
        return c0.elapsed_time(c1) / reps, None
    finally:
        cb.cublasDestroy_v2(h)


def dist_setup():
    """(rank, world, local_rank); initialises torch.distributed under torchrun."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate_max(x: float) -> float:
    """Max of x over ranks (identity without torch.distributed)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def resolve_workload(args):
    """The named workload, with --s / --mode applied (a new name when they change it)."""
    w = WORKLOADS[args.workload]
    s = args.s if args.s is not None else w.s
    mode = args.mode if args.mode is not None else w.mode
    if (s, mode) == (w.s, w.mode):
        return w
    base = w.name.rsplit("_s", 1)[0]
    return dataclasses.replace(w, name=f"{base}_s{s}_{mode}", s=s, mode=mode)


def result_line(*, value, n_gpus, steps, warmup, ms_per_step, workload, extra):
    w = WORKLOADS[workload] if isinstance(workload, str) else workload
    base = PAGES_BASELINE.get(w.name) if w == WORKLOADS.get(w.name) else None
    out = {
        "metric": metric_name(w),
        "value": value,
        "unit": UNIT,
        "n_gpus": n_gpus,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": (value / base) if base else None,
        "dtype": "f16",
        "data": "synthetic",
        "config": {
            "workload": w.name, "p": w.p, "q": w.q, "r": w.r, "s": w.s, "mode": w.mode,
            "phi": w.phi, "seed": w.seed, "io_dtype": "f64",
            "tensor_path": "tcgen05.mma kind::f16 on integer residues, fp32 TMEM accumulation",
            "l2": "inputs larger than L2 (A+B = %.2f GB vs 129 MB)" % (8e-9 * (w.p * w.q + w.q * w.r)),
            "parallelism": f"replicas{n_gpus}",
            "vs_baseline_ref": "GH200 fast-14 n=8192, 72.1 TFLOPS (Ozaki II supplement, §3.1 Table 3)" if base else None,
        },
    }
    out.update(extra)
    return out


# ----------------------------------------------------------------------------- stage rooflines
def stage_work(w):
    """Algorithmic work of each stage of the stage-timed (sequential) pass.

    HBM stages count the bytes the method must move: every input double read
    once (8 B), every residue written once (PLANE_BYTES per residue, s per
    input element), every CRT coefficient byte read once and every output
    double written once ((s + 8) B per output).  In fast mode the one-read
    kernels make A's (q <= 2048) and B's (q <= 8192) residue planes in the
    statistics stage, so those planes count there.  Accu's quantisation
    stage reads A and B and writes the fp16 bound planes.  The GEMM stages
    count 2pqr (bound) and 2 s pqr (modular) flops."""
    pq, qr, pr = w.p * w.q, w.q * w.r, w.p * w.r
    res_a = (8 + PLANE_BYTES * w.s) * pq
    res_b = (8 + PLANE_BYTES * w.s) * qr
    if w.mode == "fast":
        fused_a, fused_b = w.q <= ROWS_FUSED_MAX_Q, w.q <= COLS_FUSED_MAX_Q
        scale = (res_a if fused_a else 8 * pq) + (res_b if fused_b else 8 * qr)
        residues = (0 if fused_a else res_a) + (0 if fused_b else res_b)
        bound_flops = 0.0
    else:
        scale = (8 + PLANE_BYTES) * (pq + qr)
        residues = res_a + res_b
        bound_flops = 2.0 * pq * w.r
    return {"scale": ("hbm", float(scale)), "bound_gemm": ("tensor", bound_flops),
            "residues": ("hbm", float(residues)), "gemm_mod": ("tensor", 2.0 * w.s * pq * w.r),
            "crt": ("hbm", float((w.s + 8) * pr))}


def stage_roofline(w, stage_ms, hbm_gbs, tensor_tflops):
    """Each stage's achieved rate (its algorithmic work / its time) against its
    roofline; 'suspect' marks a fraction above 1.2, which would mean the
    timing does not cover the work."""
    out = {}
    for name, (bound, work) in stage_work(w).items():
        ms = stage_ms.get(name, 0.0)
        if work <= 0 or ms <= 0:
            continue
        if bound == "hbm":
            rate = work / (ms * 1e-3) / 1e9
            e = {"bound": "hbm", "ms": ms, "bytes": work, "GBps": rate, "peak_GBps": hbm_gbs,
                 "frac": rate / hbm_gbs}
        else:
            rate = work / (ms * 1e-3) / 1e12
            e = {"bound": "tensor", "ms": ms, "flops": work, "TFLOPs": rate, "peak_TFLOPs": tensor_tflops,
                 "frac": rate / tensor_tflops}
        e["suspect"] = e["frac"] > 1.2
        out[name] = e
    return out


# ----------------------------------------------------------------------------- CPU oracle
def oracle_full(A, B, w):
    """The native oracle on the whole problem, every stage, on all host cores: (C, seconds)."""
    from oracle import native

    t0 = time.perf_counter()
    C = native.dgemm(A, B, w.s, w.mode, want=("C",), products=ORACLE_PRODUCTS)["C"]
    return C, time.perf_counter() - t0


def oracle_sample(A, B, w, n):
    """Time the native oracle on the leading n x q x n block: (TFLOP/s, seconds)."""
    from oracle import native

    a = A[:n, :]
    b = B[:, :n]
    t0 = time.perf_counter()
    native.dgemm(a, b, w.s, w.mode, want=("C",), products=ORACLE_PRODUCTS)
    dt = time.perf_counter() - t0
    return 2.0 * a.shape[0] * w.q * b.shape[1] / dt / 1e12, dt


def cpu_cores():
    from oracle import native

    return native.threads()


def accuracy_report(A, B, w, C_gpu, C_oracle=None):
    """Normwise and componentwise errors of the GPU's and the oracle's C against
    the exact product, on ACCURACY_SAMPLES seeded sampled outputs."""
    import numpy as np

    from oracle import native

    rng = np.random.default_rng(4242)
    n = min(ACCURACY_SAMPLES, w.p * w.r)
    ii = rng.integers(0, w.p, n)
    jj = rng.integers(0, w.r, n)
    if C_oracle is not None:
        co = np.asarray(C_oracle)[ii, jj]
    else:
        al, be = native.exponents(A, B, w.s, w.mode)
        co = native.entries(A, B, w.s, al, be, ii, jj)["C"]
    rep = native.accuracy_at(A, B, ii, jj, {"gpu": np.asarray(C_gpu)[ii, jj], "oracle": co})
    rep["not_worse_than_oracle"] = bool(rep["gpu"]["normwise"] <= rep["oracle"]["normwise"] and
                                        rep["gpu"]["componentwise"] <= rep["oracle"]["componentwise"])
    rep["against"] = "exact products (fixed-point accumulator of the native oracle), sampled outputs"
    return rep


def run_reference(args, rank):
    if rank != 0:
        return 0
    w = resolve_workload(args)
    A, B = make_workload(w)
    n = min(REF_SAMPLE, w.p, w.r)
    for _ in range(args.warmup):
        oracle_sample(A, B, w, n)
    times = []
    for _ in range(args.steps):
        times.append(oracle_sample(A, B, w, n)[1])
    total = sum(times)
    value = args.steps * 2.0 * n * w.q * n / total / 1e12
    sample = (f"leading {n}x{w.q}x{n} block of the {w.name} workload per step; the native oracle "
              f"(every stage; exact products as a float64 BLAS product) on {cpu_cores()} host threads")
    line = result_line(value=value, n_gpus=args.gpus, steps=args.steps, warmup=args.warmup,
                       ms_per_step=1e3 * total / args.steps, workload=w, extra={
                           "impl": "reference",
                           "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(),
                                            "kind": "oracle", "sample": sample},
                           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                                   "d2h_bytes_per_step": 0},
                           "gpu_launches": 0,
                       })
    line["dtype"] = "int64"
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- our arm
def time_calls(oz2, torch, dA, dB, C, w, steps, stream):
    """Device time (ms) of `steps` back-to-back ozaki2_dgemm calls, CUDA events on `stream`."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        oz2.dgemm(dA, dB, w.s, w.mode, out=C)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def sequential_stages(oz2, torch, dA, dB, C, w, reps):
    """Mean per-stage ms over `reps` calls of the stage-timed entry point, whose
    stages run one after another (the kernels of each stage alone on the GPU)."""
    acc = {}
    for _ in range(reps):
        _, ms = oz2.dgemm_stages(dA, dB, w.s, w.mode, out=C)
        for k, v in ms.items():
            acc[k] = acc.get(k, 0.0) + v
    return {k: v / reps for k, v in acc.items()}


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    import __graft_entry__ as entry

    entry.build()
    import emulated_fp64_gemm_gb300 as oz2

    torch.cuda.set_device(local)
    w = resolve_workload(args)
    A, B = make_workload(w)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    C = torch.empty((w.r, w.p), dtype=torch.float64, device="cuda").t()
    stream = torch.cuda.current_stream()

    args.warmup = max(args.warmup, 3)  # at least 3 untimed warm-up steps
    for _ in range(args.warmup):
        oz2.dgemm(dA, dB, w.s, w.mode, out=C)
    torch.cuda.synchronize()

    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_index = int(vis.split(",")[local])
        except (ValueError, IndexError):
            gpu_index = local
    clocks = ClockSampler(gpu_index)

    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.25)  # let the sampler take its first reading
    n0 = oz2.launch_count()
    local_ms = time_calls(oz2, torch, dA, dB, C, w, args.steps, stream)
    launches = oz2.launch_count() - n0
    barrier()
    clk = clocks.stop()

    # the GEMM span of the same calls comes from a second, instrumented pass
    # (events at the stage boundaries of the overlapped schedule); its own time
    # gives the overhead of instrumenting, which the clean pass above does not carry
    oz2.profile_begin(args.steps)
    instrumented_ms = time_calls(oz2, torch, dA, dB, C, w, args.steps, stream) / args.steps
    ncalls, stage_sum = oz2.profile_end()
    max_ms = aggregate_max(local_ms)
    # per-stage rooflines: the stage-timed entry point runs the stages one after another
    seq = sequential_stages(oz2, torch, dA, dB, C, w, reps=3)
    status = oz2.last_error()
    if status != 0:
        raise RuntimeError(f"device-side error word set: {status}")

    ms_per_step = max_ms / args.steps
    value = world * args.steps * w.flops / (max_ms * 1e-3) / 1e12
    stages = {k: v / max(ncalls, 1) for k, v in stage_sum.items()}

    # roofline of the dominant kernel: the s modular GEMMs (a dense contraction)
    peaks, how = measured_peaks()
    gemm_flops = 2.0 * w.s * w.p * w.q * w.r
    achieved = gemm_flops / (stages["gemm_mod"] * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    roofline = {"bound": "tensor", "kernel": "oz2_gemm2sm_kernel (CTA-pair tcgen05, mod epilogue)",
                "unit_of_work": "the GEMM stage of one call (all its GEMM launches)", "achieved": achieved,
                "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": gemm_traffic_per_unit() if w.name == GEMM_PROFILE_WORKLOAD else None,
                "peak_source": f"{how} bf16 dense burst (f16 kind::f16 runs at the bf16 rate)",
                "algorithmic": "2*s*p*q*r flops per launch"}
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    extra = {"impl": "ours", "roofline": roofline, "stages_ms": stages,
             "stages_note": ("from a second, instrumented pass of the same calls; overlapped schedule: "
                             "residues = residue time before the first GEMM, gemm_mod = span of the GEMM "
                             "launches, crt = CRT time after the last GEMM"),
             "instrumented_ms_per_step": instrumented_ms,
             "instrumenting_overhead": instrumented_ms / ms_per_step - 1.0,
             "stage_roofline": {"pass": "ozaki2_dgemm_stages (stages one after another), mean of 3 calls",
                                "peak_source": f"{how} HBM copy and bf16 dense burst",
                                "total_ms": seq.get("total"),
                                "stages": stage_roofline(w, seq, hbm, peak)},
             "gpu_launches": launches}
    if clk is not None:
        extra["clocks"] = {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"],
                           "reasons": clk["reasons"], "samples": clk["samples"]}

    # context: native FP64 GEMM (cuBLAS DGEMM through torch.matmul, a library call) on the
    # same device-resident operands, the comparison the pages' tables make
    if not args.no_context:
        ref = torch.matmul(dA, dB)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 3
        c0.record(stream)
        for _ in range(reps):
            torch.matmul(dA, dB, out=ref)
        c1.record(stream)
        torch.cuda.synchronize()
        dg_ms = c0.elapsed_time(c1) / reps
        extra["context"] = {"cublas_dgemm_tflops": w.flops / dg_ms / 1e9, "cublas_dgemm_ms": dg_ms,
                            "note": "native FP64 GEMM on the same operands (torch.matmul, float64)"}
        # cuBLAS's fixed-point FP64 emulation on the same operands (C column-major, ldc = p)
        dCe = torch.empty((w.r, w.p), dtype=torch.float64, device=dA.device).t()
        em_ms, why = cublas_emulated_dgemm_ms(dA, dB, dCe, w.p, w.q, w.r, stream, reps)
        if em_ms is None:
            extra["context"]["cublas_fp64_emulated"] = {"unavailable": why}
        else:
            extra["context"]["cublas_fp64_emulated"] = {
                "tflops": w.flops / em_ms / 1e9, "ms": em_ms,
                "note": ("cublasGemmEx, CUBLAS_COMPUTE_64F_EMULATED_FIXEDPOINT, emulation math mode, "
                         "eager strategy; a rate equal to the native DGEMM's means the emulation "
                         "did not engage on this device")}
        del ref, dCe

    # end to end through the host-memory entry point: H2D of A and B, D2H of C
    e_in = w.p * w.q + w.q * w.r
    if not args.no_e2e:
        hA = torch.from_numpy(A).pin_memory()
        hB = torch.from_numpy(B).pin_memory()
        hC = torch.empty((w.r, w.p), dtype=torch.float64).pin_memory().t()
        for _ in range(max(1, args.warmup)):  # the first call sizes the staging workspace
            oz2.dgemm_host(hA, hB, w.s, w.mode, out=hC)
        barrier()
        t0 = time.perf_counter()
        per_call = []
        for _ in range(args.steps):
            tc = time.perf_counter()
            oz2.dgemm_host(hA, hB, w.s, w.mode, out=hC)
            per_call.append(time.perf_counter() - tc)
        e2e_s = aggregate_max(time.perf_counter() - t0)
        # value: all timed calls (the mean); the median call shows the rate between the
        # occasional long stalls of the host link (tens of ms) that some calls meet
        extra["e2e"] = {"value": world * args.steps * w.flops / e2e_s / 1e12, "unit": UNIT,
                        "h2d_bytes_per_step": 8 * e_in, "d2h_bytes_per_step": 8 * w.p * w.r,
                        "median_ms_per_call": 1e3 * statistics.median(per_call),
                        "max_ms_per_call": 1e3 * max(per_call)}
        got = hC.numpy()
        if not np.array_equal(got, C.cpu().numpy()):
            raise RuntimeError("host entry point disagrees with the device entry point")
        del hA, hB, hC

    C_gpu = C.cpu().numpy()
    del dA, dB, C
    torch.cuda.empty_cache()
    C_oracle = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        C_oracle, dt = oracle_full(A, B, w)
        v = w.flops / dt / 1e12
        extra["cpu_baseline"] = {
            "value": v, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": (f"full problem ({w.p}x{w.q}x{w.r}, s={w.s}, {w.mode}), {dt:.1f} s: the native oracle, "
                       f"every stage on {cpu_cores()} host threads, exact products as a float64 BLAS product")}
        # the oracle's C for the whole problem doubles as a full elementwise check of the timed output
        extra["full_parity"] = {"entries": int(C_gpu.size), "identical": bool(np.array_equal(C_gpu, C_oracle)),
                                "max_ulp": entry.ulp_distance(C_gpu, C_oracle), "tolerance_ulp": 2}
    if rank == 0:
        extra["accuracy"] = accuracy_report(A, B, w, C_gpu, C_oracle)
        print(json.dumps(result_line(value=value, n_gpus=world, steps=args.steps,
                                     warmup=args.warmup, ms_per_step=ms_per_step,
                                     workload=w, extra=extra)), flush=True)
    return 0


def sweep_sets(args):
    """(n values, s values) of --sweep: --sweep-n / --sweep-s, else SWEEP_N / SWEEP_S."""
    ns = tuple(int(x) for x in args.sweep_n.split(",")) if args.sweep_n else SWEEP_N
    ss = tuple(int(x) for x in args.sweep_s.split(",")) if args.sweep_s else SWEEP_S
    for s in ss:
        if not 2 <= s <= 20:
            raise SystemExit(f"--sweep-s: s = {s} outside 2..20")
    for n in ns:
        if n < 1:
            raise SystemExit(f"--sweep-n: n = {n} must be positive")
    return ns, ss


def run_sweep(args):
    """ms per call (clean pass) and per stage (stage-timed pass) for every s in
    SWEEP_S at n in SWEEP_N (or --sweep-s / --sweep-n), fast and accu,
    phi = 0.5, seed 123456: one JSON line per configuration."""
    import torch

    import __graft_entry__ as entry
    from workloads import Workload, make_matrices

    entry.build()
    import emulated_fp64_gemm_gb300 as oz2

    stream = torch.cuda.current_stream()
    sweep_n, sweep_s = sweep_sets(args)
    for n in sweep_n:
        A, B = make_matrices(n, n, n, 0.5, 123456)
        dA = torch.from_numpy(A).cuda()
        dB = torch.from_numpy(B).cuda()
        C = torch.empty((n, n), dtype=torch.float64, device="cuda").t()
        steps = max(3, min(args.steps, 30))
        for mode in ("fast", "accu"):
            for s in sweep_s:
                w = Workload(f"n{n}_s{s}_{mode}", n, n, n, s, mode, 0.5, 123456)
                for _ in range(3):
                    oz2.dgemm(dA, dB, s, mode, out=C)
                torch.cuda.synchronize()
                ms = time_calls(oz2, torch, dA, dB, C, w, steps, stream) / steps
                seq = sequential_stages(oz2, torch, dA, dB, C, w, reps=3)
                print(json.dumps({"sweep": True, "n": n, "s": s, "mode": mode, "steps": steps,
                                  "ms_per_call": ms, "tflops": w.flops / ms / 1e9,
                                  "sequential_stages_ms": seq}), flush=True)
        del dA, dB, C
        torch.cuda.empty_cache()
    return 0


def run_stages_once(args):
    """One ozaki2_dgemm_stages call on the workload (stages one after another)."""
    import torch

    import __graft_entry__ as entry

    entry.build()
    import emulated_fp64_gemm_gb300 as oz2

    w = resolve_workload(args)
    A, B = make_workload(w)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    _, ms = oz2.dgemm_stages(dA, dB, w.s, w.mode)
    torch.cuda.synchronize()
    status = oz2.last_error()
    print(json.dumps({"workload": w.name, "stages_ms": ms, "last_error": status}), flush=True)
    return 0 if status == 0 else 1


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_setup()
    if args.stages_once:
        rc = run_stages_once(args) if rank == 0 else 0
    elif args.sweep:
        rc = run_sweep(args) if rank == 0 else 0
    elif args.impl == "reference":
        rc = run_reference(args, rank)
    else:
        rc = run_ours(args, rank, world, local)
    try:
        import torch.distributed as dist

        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()
    except Exception:
        pass
    return rc


if __name__ == "__main__":
    sys.exit(main())
