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
