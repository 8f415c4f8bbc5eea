#!/usr/bin/env python3
"""Benchmark of the GB300 Ozaki-II FP64 GEMM.

Metric: effective FP64 TFLOPS = 2pqr / time of one ozaki2_dgemm call, on the
n = 8192, s = 14, fast workload (the study's headline configuration), with
the per-stage milliseconds of the same calls.  One step = one full call
(scaling, residues, the s modular GEMMs, CRT) on inputs already in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the method has no exchange step on one problem; weak scaling); the timed
region is bracketed by barriers and the slowest rank's time is reported.
One JSON line is printed by rank 0.
"""
from __future__ import annotations

import argparse
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


def metric_name(workload: str) -> str:
    """The headline metric string; other workloads name their own shape and mode."""
    if workload == HEADLINE:
        return METRIC
    w = WORKLOADS[workload]
    return (f"effective FP64 TFLOPS (2pqr/time), Ozaki-II p={w.p} q={w.q} r={w.r} s={w.s} {w.mode}; "
            "per-stage ms")
UNIT = "TFLOP/s"
# The pages' number for this metric and workload: GH200, fast-14, n=8192 (paper Table 3).
PAGES_BASELINE = {"n8192_s14_fast": 72.1}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_PROFILE = os.path.join(ROOT, "profiles", "oz2_gemm_kernel_n8192_s14_fast.md")
# the GEMM kernel's source files, hashed in this order against the summary's source_sha256
GEMM_SOURCES = [os.path.join(ROOT, "emulated_fp64_gemm_gb300", "csrc", f)
                for f in ("oz2_gemm.cu", "oz2_tcgen05.cuh")]
CPU_SAMPLE = 512  # rows of A and columns of B in the oracle's bounded sample


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
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


def result_line(*, value, n_gpus, steps, warmup, ms_per_step, workload, extra):
    w = WORKLOADS[workload]
    base = PAGES_BASELINE.get(workload)
    out = {
        "metric": metric_name(workload),
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
            "workload": workload, "p": w.p, "q": w.q, "r": w.r, "s": w.s, "mode": w.mode,
            "phi": w.phi, "seed": w.seed, "io_dtype": "f64",
            "tensor_path": "tcgen05.mma kind::f16 on integer residues, fp32 TMEM accumulation",
            "l2": "inputs larger than L2 (A+B = %.2f GB vs 129 MB)" % (8e-9 * (w.p * w.q + w.q * w.r)),
            "parallelism": f"replicas{n_gpus}",
            "vs_baseline_ref": "GH200 fast-14 n=8192, 72.1 TFLOPS (paper Table 3)" if base else None,
        },
    }
    out.update(extra)
    return out


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(A, B, w, n):
    """Time the oracle on the leading n x q x n block of the workload."""
    from oracle import ozaki2_oracle as oracle

    a = A[:n, :]
    b = B[:, :n]
    t0 = time.perf_counter()
    oracle.oracle_dgemm(a, b, w.s, w.mode)
    dt = time.perf_counter() - t0
    return 2.0 * n * w.q * n / dt / 1e12, dt


def cpu_cores():
    return os.cpu_count() or 1


def run_reference(args, rank):
    if rank != 0:
        return 0
    w = WORKLOADS[args.workload]
    A, B = make_workload(w)
    n = 256
    for _ in range(args.warmup):
        oracle_sample(A, B, w, n)
    times = []
    for _ in range(args.steps):
        times.append(oracle_sample(A, B, w, n)[1])
    total = sum(times)
    value = args.steps * 2.0 * n * w.q * n / total / 1e12
    sample = f"leading {n}x{w.q}x{n} block of the {args.workload} workload per step"
    line = result_line(value=value, n_gpus=args.gpus, steps=args.steps, warmup=args.warmup,
                       ms_per_step=1e3 * total / args.steps, workload=args.workload, extra={
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
def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    import __graft_entry__ as entry

    entry.build()
    import emulated_fp64_gemm_gb300 as oz2

    torch.cuda.set_device(local)
    w = WORKLOADS[args.workload]
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

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.25)  # let the sampler take its first reading
    n0 = oz2.launch_count()
    e0.record(stream)
    for _ in range(args.steps):
        oz2.dgemm(dA, dB, w.s, w.mode, out=C)
    e1.record(stream)
    torch.cuda.synchronize()
    launches = oz2.launch_count() - n0
    barrier()
    clk = clocks.stop()
    local_ms = e0.elapsed_time(e1)

    # the per-stage split comes from a second, instrumented pass of the same
    # calls (events at the stage boundaries); its own time gives the overhead
    # of instrumenting, which the clean pass above does not carry
    oz2.profile_begin(args.steps)
    e0.record(stream)
    for _ in range(args.steps):
        oz2.dgemm(dA, dB, w.s, w.mode, out=C)
    e1.record(stream)
    torch.cuda.synchronize()
    ncalls, stage_sum = oz2.profile_end()
    instrumented_ms = e0.elapsed_time(e1) / args.steps
    max_ms = aggregate_max(local_ms)
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
                "traffic": gemm_traffic_per_unit() if args.workload == GEMM_PROFILE_WORKLOAD else None,
                "peak_source": f"{how} bf16 dense burst (f16 kind::f16 runs at the bf16 rate)",
                "algorithmic": "2*s*p*q*r flops per launch"}
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    e_in = w.p * w.q + w.q * w.r
    stage_roofline = {
        "scale_GBps": 2 * 8 * e_in / (stages["scale"] * 1e-3) / 1e9 if stages["scale"] > 0 else None,
        "residues_GBps": (8 + 2 * w.s) * e_in / (stages["residues"] * 1e-3) / 1e9,
        "crt_GBps": (w.s + 8) * w.p * w.r / (stages["crt"] * 1e-3) / 1e9,
        "hbm_peak_GBps": hbm,
    }
    extra = {"impl": "ours", "roofline": roofline, "stages_ms": stages,
             "stages_note": ("from a second, instrumented pass of the same calls; overlapped schedule: "
                             "residues = residue time before the first GEMM, gemm_mod = span of the GEMM "
                             "launches, crt = CRT time after the last GEMM"),
             "instrumented_ms_per_step": instrumented_ms,
             "instrumenting_overhead": instrumented_ms / ms_per_step - 1.0,
             "stage_bandwidth": stage_roofline, "gpu_launches": launches}
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
        dev_c = C.cpu().numpy()
        if not np.array_equal(got, dev_c):
            raise RuntimeError("host entry point disagrees with the device entry point")

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt = oracle_sample(A, B, w, CPU_SAMPLE)
        extra["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                                 "sample": f"leading {CPU_SAMPLE}x{w.q}x{CPU_SAMPLE} block, "
                                           f"{dt:.1f} s; BLAS products on all cores, the rest on one"}
    if rank == 0:
        print(json.dumps(result_line(value=value, n_gpus=world, steps=args.steps,
                                     warmup=args.warmup, ms_per_step=ms_per_step,
                                     workload=args.workload, extra=extra)), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_setup()
    if args.impl == "reference":
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
