"""bench.py host logic without a GPU: the JSON line, clock parsing and the
max-over-ranks aggregation across two gloo ranks."""
import json
import os
import socket

import pytest

import bench


def test_result_line_has_the_contract_keys():
    line = bench.result_line(value=100.0, n_gpus=1, steps=30, warmup=3, ms_per_step=11.0,
                             workload="n8192_s14_fast", extra={"impl": "ours"})
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert k in line
    assert line["config"]["workload"] == "n8192_s14_fast"
    assert abs(line["vs_baseline"] - 100.0 / 72.1) < 1e-12
    json.dumps(line)
    other = bench.result_line(value=1.0, n_gpus=1, steps=1, warmup=3, ms_per_step=1.0,
                              workload="n4096_s14_accu", extra={})
    assert other["vs_baseline"] is None


def test_metric_names_the_workload_and_traffic_is_tied_to_the_profiled_source():
    # the headline keeps the contract's metric string; other workloads name their shape and mode
    assert bench.metric_name(bench.HEADLINE) == bench.METRIC
    other = bench.metric_name("n4096_s14_accu")
    assert "p=4096 q=4096 r=4096 s=14 accu" in other and other != bench.METRIC
    line = bench.result_line(value=1.0, n_gpus=1, steps=1, warmup=3, ms_per_step=1.0,
                             workload="n4096_s14_accu", extra={})
    assert line["metric"] == other
    # the GEMM traffic comes from the committed profile only while its recorded
    # source hash matches the kernel source; otherwise it is reported as null
    assert bench.GEMM_PROFILE_WORKLOAD == bench.HEADLINE
    import re
    text = open(bench.GEMM_PROFILE).read()
    recorded = re.search(r"source_sha256:\s*([0-9a-f]{64})", text).group(1)
    t = bench.gemm_traffic_per_unit()
    if recorded == bench.gemm_source_sha256():
        assert t is not None and t > 0
    else:
        assert t is None


def test_clock_sampler_without_nvidia_smi_returns_none():
    c = bench.ClockSampler(0)
    c.start()
    assert c.stop() is None or isinstance(c.stop(), dict)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier()
    v = bench.aggregate_max(10.0 + rank * 5.0)
    out.put((rank, v))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 15.0), (1, 15.0)]


def test_stage_work_counts_what_each_stage_runs():
    w = bench.WORKLOADS["n8192_s14_fast"]
    n2 = 8192 * 8192
    work = bench.stage_work(w)
    # q = 8192: A's statistics read A once; B's one-read kernel makes B's planes in this stage
    assert work["scale"] == ("hbm", float(8 * n2 + (8 + 2 * 14) * n2))
    assert work["residues"] == ("hbm", float((8 + 2 * 14) * n2))
    assert work["crt"] == ("hbm", float((14 + 8) * n2))
    assert work["gemm_mod"] == ("tensor", 2.0 * 14 * n2 * 8192)
    assert work["bound_gemm"][1] == 0.0
    small = bench.dataclasses.replace(w, p=1024, q=1024, r=1024)  # both one-read kernels
    ws = bench.stage_work(small)
    assert ws["residues"][1] == 0.0 and ws["scale"][1] == float((8 + 28) * 2 * 1024 * 1024)
    acc = bench.WORKLOADS["n4096_s14_accu"]
    wa = bench.stage_work(acc)
    assert wa["scale"][1] == float(10 * 2 * 4096 * 4096) and wa["bound_gemm"][1] == 2.0 * 4096**3


def test_stage_roofline_flags_rates_above_the_peak():
    w = bench.WORKLOADS["n8192_s14_fast"]
    work = bench.stage_work(w)
    ms_ok = {"scale": work["scale"][1] / 5e9 * 1e3 / 1e3, "residues": 0.2, "gemm_mod": 9.0, "crt": 0.5}
    out = bench.stage_roofline(w, ms_ok, 6792.1, 1898.6)
    assert set(out) == {"scale", "residues", "gemm_mod", "crt"}
    assert abs(out["scale"]["GBps"] - 5000.0) < 1e-6 and not out["scale"]["suspect"]
    assert abs(out["crt"]["frac"] - (22 * 8192**2 / 0.5e-3 / 1e9) / 6792.1) < 1e-12
    fast = bench.stage_roofline(w, {"crt": 0.05}, 6792.1, 1898.6)
    assert fast["crt"]["suspect"]  # 29 TB/s: the timing cannot cover the work


def test_s_and_mode_overrides_rename_the_workload():
    args = bench.parse_args(["--workload", "n8192_s14_fast", "--s", "18", "--mode", "accu"])
    w = bench.resolve_workload(args)
    assert (w.name, w.s, w.mode, w.p) == ("n8192_s18_accu", 18, "accu", 8192)
    line = bench.result_line(value=1.0, n_gpus=1, steps=1, warmup=3, ms_per_step=1.0, workload=w, extra={})
    assert line["config"]["workload"] == "n8192_s18_accu" and "s=18 accu" in line["metric"]
    assert line["vs_baseline"] is None
    same = bench.resolve_workload(bench.parse_args([]))
    assert same is bench.WORKLOADS["n8192_s14_fast"]


def test_sweep_sets_default_and_override():
    args = bench.parse_args(["--sweep"])
    assert bench.sweep_sets(args) == (bench.SWEEP_N, bench.SWEEP_S)
    args = bench.parse_args(["--sweep", "--sweep-n", "2048,16384", "--sweep-s", "14,15,18"])
    assert bench.sweep_sets(args) == ((2048, 16384), (14, 15, 18))
    with pytest.raises(SystemExit):
        bench.sweep_sets(bench.parse_args(["--sweep", "--sweep-s", "21"]))
