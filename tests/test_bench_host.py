"""Host-side logic of bench.py without a GPU: the work model, the launch count,
the kernel-code hash that ties the traffic summaries to the kernel, and the max-over-ranks
aggregation across two gloo processes."""
import datetime
import os
import socket
import time

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from moe_token_dispatch_route_gb300 import workloads


def test_algorithmic_work_mixtral():
    wl = workloads.WORKLOADS["mixtral"]
    flops, nbytes, scatter = bench.algorithmic_work(wl, touched_experts=8)
    assert flops == 2 * 8192 * 2 * 4096 * 14336
    # x read, receive rows written and read back, Y written, 8 experts' weights read
    assert nbytes == 8192 * 4096 * 2 + 2 * 16384 * 4096 * 2 + 16384 * 14336 * 4 + 8 * 4096 * 14336 * 2
    assert scatter == 8192 * 4096 * 2 + 16384 * 4096 * 2
    # tensor-bound: far above the ridge of ~280 FLOP/B
    assert flops / nbytes > 800


def test_scatter_report_rate_only_without_background():
    on = bench.scatter_report(100_000, 1e9, 6758.0, {"background_scatter": 152})
    off = bench.scatter_report(100_000, 1e9, 6758.0, {"background_scatter": 0})
    assert on["background"] and "frac_hbm" not in on
    assert not off["background"] and abs(off["frac_hbm"] - 1e4 / 6758.0) < 1e-12
    assert on["gbs"] == off["gbs"] == 1e4 and on["window_ms"] == 0.1


def test_launches_per_step():
    assert bench.launches_per_step(workloads.WORKLOADS["mixtral"]) == 3
    assert bench.launches_per_step(workloads.WORKLOADS["decode"]) == 2


def test_kernel_code_hash_ignores_comments_only(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("int f(int x) {\n    return x + 1;  // one\n}\n")
    b = tmp_path / "b.cu"
    b.write_text("/* header */\n// f adds one\nint f(int x) {\n\n    return x + 1;\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) {\n    return x + 2;\n}\n")
    assert bench.kernel_code_hash(str(a)) == bench.kernel_code_hash(str(b))
    assert bench.kernel_code_hash(str(a)) != bench.kernel_code_hash(str(c))


def _smi_line(t, mhz, power_cap):
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{stamp}, {mhz}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {power_cap}"


def test_clock_summary_keeps_only_samples_inside_the_timed_region():
    c = bench.ClockSampler(0)
    c.t0 = time.time()
    c.t1 = c.t0 + 0.3
    c.lines = [_smi_line(c.t0 - 0.4, 1000, "Not Active"),   # before the region (idle)
               _smi_line(c.t0 + 0.05, 2070, "Not Active"),
               _smi_line(c.t0 + 0.15, 1900, "Active"),
               _smi_line(c.t0 + 0.25, 1950, "Not Active"),
               _smi_line(c.t0 + 0.9, 800, "Not Active")]    # after it
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 1950.0 and s["window"] == "timed region"
    assert s["reasons"] == ["sw_power_cap"] and s["sm_max_mhz"] == 2070.0


def test_clock_summary_without_a_sample_inside_takes_the_nearest():
    c = bench.ClockSampler(0)
    c.t0 = time.time()
    c.t1 = c.t0 + 0.01
    c.lines = [_smi_line(c.t0 - 0.5, 1200, "Not Active"), _smi_line(c.t1 + 0.1, 2000, "Not Active")]
    s = c.summary()
    assert s["samples"] == 1 and s["sm_mhz"] == 2000.0 and s["window"] == "nearest sample"


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(1.5 + rank, world)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_processes():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_clock_summary_from_nvml_samples():
    """NVML samples (time, SM MHz, reasons): only those inside the timed region count."""
    import types
    c = bench.ClockSampler(0)
    c.t0 = time.time()
    c.t1 = c.t0 + 0.02
    c.nvml = types.SimpleNamespace(max_mhz=2070.0, rows=[
        (c.t0 - 0.5, 900.0, []),                       # before the region
        (c.t0 + 0.002, 2070.0, []), (c.t0 + 0.004, 1980.0, ["sw_power_cap"]),
        (c.t0 + 0.006, 2010.0, []), (c.t0 + 5.0, 700.0, ["hw_slowdown"])])  # after it
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2010.0 and s["sm_mhz_min"] == 1980.0
    assert s["reasons"] == ["sw_power_cap"] and s["sm_max_mhz"] == 2070.0 and s["source"] == "nvml"
