#!/usr/bin/env python3
"""Benchmark of the whole hot path: routing + fused dispatch/grouped GEMM.

One step = moe_route (top-k, histogram, prefix sum, permutation) followed by
moe_dispatch_gemm (scatter into the rank receive buffers + per-expert GEMM)
over one batch of synthetic inputs already resident in HBM.  The default
workload is the Mixtral-shaped layer (T=8192, d=4096, E=8, top-2, N=14336).

Prints one JSON line (rank 0).  `value` is TFLOP/s of the whole step
(2*T*k*d*N FLOPs / step time); `e2e` is the same metric through the same C
ABI with the step's inputs copied from pinned host memory and Y copied back
inside the timed region.  `--impl reference` times the CPU oracle instead.

Multi-GPU (torchrun, one rank per GPU): the path has no multi-GPU exchange
in this library, so every rank runs an independent replica (weak scaling);
the timed region is bracketed by barriers and the max over ranks is used.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused dispatch+grouped-GEMM TFLOP/s and tokens/s at 1 GB300; % of bf16 peak"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 512 << 20
L2_BYTES = 126 << 20  # GB300 L2
KERNEL_SRC = os.path.join(ROOT, "moe_token_dispatch_route_gb300", "csrc", "dispatch_gemm.cu")


def _args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixtral")
    ap.add_argument("--shape", default="", help="custom workload T,d,E,k,N[,R] (overrides --workload)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tile-n", type=int, default=0)
    ap.add_argument("--tile-m", type=int, default=0, help="128 (one CTA per tile), 256 (CTA pairs), 0 auto")
    ap.add_argument("--l2", choices=["flush", "none"], default="flush",
                    help="between timed steps: flush L2 (default) or rely on inputs larger than L2")
    ap.add_argument("--producer-ctas", type=int, default=0)
    ap.add_argument("--workloads", default="others",
                    help="other configurations measured in the same run: 'others' (every other "
                         "workload), 'none', or a comma-separated list")
    ap.add_argument("--kernel-only", choices=["fused", "grouped", "gather"], default=None,
                    help="profiling case: after the warm-up, run only `--steps` launches of the fused "
                         "kernel (moe_dispatch_gemm), of the GEMM alone on the receive rows in place "
                         "(moe_grouped_gemm) or of the direct gather (moe_gather_gemm), L2 flushed "
                         "between them, print their median and exit")
    ap.add_argument("--ffn", choices=["auto", "on", "off"], default="auto",
                    help="also time the gated (SwiGLU) expert FFN with F = N (auto: Mixtral-shaped only)")
    return ap.parse_args(argv)


def _peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, source)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]),
                float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured")
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_code_hash(path: str = KERNEL_SRC) -> str:
    """First 16 hex digits of the SHA-256 of the fused kernel's source with its
    comments and blank lines removed: a comment edit keeps a capture valid, any
    code change invalidates it."""
    src = open(path, encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    lines = []
    for line in src.splitlines():
        code = line.split("//", 1)[0].rstrip()
        if code.strip():
            lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def _traffic_per_launch(workload: str):
    """DRAM bytes per launch of the fused kernel from the committed ncu summary,
    or None when absent or when the kernel source changed since the capture."""
    path = os.path.join(ROOT, "profiles", f"dispatch_gemm_{workload}_traffic.txt")
    try:
        vals = {}
        with open(path) as f:
            for line in f:
                if ":" in line:
                    key, val = line.split(":", 1)
                    vals[key.strip()] = val.strip()
        if vals.get("kernel_code_sha256_16") != kernel_code_hash():
            return None
        return float(vals["traffic_bytes_per_launch"])
    except Exception:
        return None


class NvmlClocks:
    """Read-only NVML queries (libnvidia-ml through ctypes) of one GPU's SM clock and
    clock-event reasons, polled by a thread of its own every PERIOD_S.  Nothing is set:
    only nvmlInit, handle lookups, nvmlDeviceGet*Clock* and nvmlShutdown are called."""

    PERIOD_S = 0.002
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown"}

    def __init__(self, index: int, uuid: str | None = None):
        import ctypes
        import threading

        self.ct = ctypes
        self.rows = []
        self._stop = threading.Event()
        self._thread = None
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        ok = False
        if uuid:
            ok = self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) == 0
        if not ok and self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.dev)) != 0:
            raise RuntimeError("no NVML handle")
        self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx)) == 0 \
            else None
        self.sample()  # one query now, so a failure shows before the timed region

    def sample(self):
        ct = self.ct
        mhz, rs = ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ct.byref(mhz)) != 0:  # NVML_CLOCK_SM
            raise RuntimeError("nvmlDeviceGetClockInfo failed")
        reasons = [n for b, n in self.REASON_BITS.items() if self._reasons(self.dev, ct.byref(rs)) == 0 and rs.value & b]
        self.rows.append((time.time(), float(mhz.value), reasons))

    def _run(self):
        while not self._stop.is_set():
            try:
                self.sample()
            except Exception:
                return
            time.sleep(self.PERIOD_S)

    def start(self):
        import threading
        self.rows = []
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=2.0)
        self.sample()  # the clock at the region's end
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clocks and clock-event reasons during the timed region: NVML polled every
    2 ms when libnvidia-ml can be loaded, else nvidia-smi every PERIOD_MS.

    The nvidia-smi sampler starts before the region (nvidia-smi takes a moment to
    report) and keeps only the samples whose own timestamps fall between entry and
    exit."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    STARTUP_S = 0.5
    PERIOD_MS = 50

    def __init__(self, index: int, use_nvml: bool = True):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None
        self.nvml = None
        self.use_nvml = use_nvml

    def __enter__(self):
        if self.use_nvml:
            try:
                uuid = None
                try:
                    import torch
                    uuid = "GPU-" + str(torch.cuda.get_device_properties(self.index).uuid)
                except Exception:
                    pass
                self.nvml = NvmlClocks(self.index, uuid)
                self.t0 = time.time()
                self.nvml.start()
                return self
            except Exception:
                self.nvml = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(self.STARTUP_S)
        except Exception:
            self.proc = None
        self.t0 = time.time()
        return self

    def __exit__(self, *exc):
        self.t1 = time.time()
        self.lines = []
        if self.nvml is not None:
            self.nvml.stop()
            return
        if self.proc is not None:
            time.sleep(2 * self.PERIOD_MS / 1000.0)  # the sample that covers the region's end
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    @staticmethod
    def _stamp(text: str):
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self):
        if self.nvml is not None:
            inside = [r for r in self.nvml.rows if self.t0 <= r[0] <= self.t1 + 0.01]
            if not inside:
                return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": "nvml"}
            return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": self.nvml.max_mhz,
                    "sm_mhz_min": min(r[1] for r in inside),
                    "reasons": sorted({n for r in inside for n in r[2]}), "samples": len(inside),
                    "window": "timed region", "period_ms": 1000 * NvmlClocks.PERIOD_S, "source": "nvml"}
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            t = self._stamp(parts[0])
            try:
                rows.append((t, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if r[0] is not None and self.t0 is not None
                  and self.t0 <= r[0] <= self.t1 + self.PERIOD_MS / 1000.0]
        window = "timed region"
        if not inside and rows:  # no sample inside a very short region: the one nearest its end
            stamped = [r for r in rows if r[0] is not None]
            inside = [min(stamped, key=lambda r: abs(r[0] - self.t1))] if stamped else rows[-1:]
            window = "nearest sample"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = {n for r in inside for n, v in zip(names, r[3]) if v.lower() == "active"}
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside), "window": window,
                "period_ms": self.PERIOD_MS}


def algorithmic_work(wl, touched_experts: int):
    """FLOPs and DRAM bytes one pass of the fused kernel must move at least:
    read x once (T*d*2), write and re-read the receive rows (2*S*d*2), write Y
    (S*N*4), read each touched expert's weights once (d*N*2 each)."""
    flops = wl.flops
    nbytes = (wl.T * wl.d * 2 + 2 * wl.S * wl.d * 2 + wl.S * wl.N * 4
              + touched_experts * wl.d * wl.N * 2)
    scatter_bytes = wl.T * wl.d * 2 + wl.S * wl.d * 2
    return flops, nbytes, scatter_bytes


def launches_per_step(wl) -> int:
    """Kernels of this library per step: routing select (+ permutation when
    T*k > 8192; smaller batches permute inside the routing kernel) + the fused
    dispatch/grouped-GEMM kernel."""
    return 2 + (1 if wl.T * wl.k > 8192 else 0)


LATENCY_BOUND_US = 10.0  # below this ideal time (HBM or tensor) a launch is latency-bound


def roofline_of(wl, touched: int, fused_avg_s: float, plan_info: dict, peaks) -> dict:
    """Roofline of the fused kernel from its algorithmic work (algorithmic_work) and its
    average launch time: "tensor" when the FLOP per byte exceed the measured ridge,
    "hbm" otherwise, "latency" when both ideal times are below LATENCY_BOUND_US."""
    hbm_peak, tf_peak, tf_sustained, peak_src = peaks
    flops, alg_bytes, _ = algorithmic_work(wl, touched)
    ridge = tf_peak * 1e12 / (hbm_peak * 1e9)
    t_tensor_us = flops / (tf_peak * 1e12) * 1e6
    t_hbm_us = alg_bytes / (hbm_peak * 1e9) * 1e6
    if flops / alg_bytes >= ridge:
        roof = {"bound": "tensor", "achieved": flops / fused_avg_s / 1e12, "peak": tf_peak,
                "unit": "TFLOP/s", "peak_source": f"{peak_src} (bf16 burst)"}
    else:
        roof = {"bound": "hbm", "achieved": alg_bytes / fused_avg_s / 1e9, "peak": hbm_peak,
                "unit": "GB/s", "peak_source": f"{peak_src} (copy bandwidth)"}
    if max(t_tensor_us, t_hbm_us) < LATENCY_BOUND_US:
        roof["bound"] = "latency"
        roof["note"] = (f"ideal times {t_hbm_us:.2f} us (HBM) and {t_tensor_us:.2f} us (tensor) are far "
                        f"below the launch and pipeline latency; achieved/frac against "
                        f"{'HBM' if roof['unit'] == 'GB/s' else 'bf16'} for reference")
    roof["frac"] = roof["achieved"] / roof["peak"]
    if roof["bound"] == "tensor":  # the same kernel against the power-capped sustained peak
        roof["peak_sustained"] = tf_sustained
        roof["frac_sustained"] = roof["achieved"] / tf_sustained
    roof["traffic"] = _traffic_per_launch(wl.name)
    tile = f"{plan_info['tile_m']}x{plan_info['tile_n']} tiles"
    roof["kernel"] = (f"dispatch_gemm_pair_kernel (CTA pairs, {tile})"
                      if plan_info["tile_m"] == 256 else f"dispatch_gemm_kernel ({tile})")
    roof["algorithmic_flops"] = flops
    roof["algorithmic_bytes"] = alg_bytes
    return roof


def scatter_report(scatter_ns: int, scatter_bytes: float, hbm_peak: float, plan_info: dict) -> dict:
    """The scatter window of the last timed call (first scatter start to last scatter end,
    from the workspace header) and its rate.  With the background scatter (CTA pairs on wide
    layers) the window ends when warp 3's copies beside the GEMM end, so its rate says how
    far ahead of the GEMM they ran, not what HBM can do."""
    bg = int(plan_info.get("background_scatter", 0)) > 0
    gbs = scatter_bytes / max(scatter_ns, 1)
    out = {"window_ms": scatter_ns / 1e6, "bytes": scatter_bytes, "gbs": gbs, "background": bg}
    if bg:
        out["note"] = ("all warps copy the first experts' rows (the first two waves of pair tiles), then "
                       "warp 3 of every CTA copies the rest beside the GEMM; the window ends with those "
                       "copies, so its rate is not an HBM rate")
    else:
        out["frac_hbm"] = gbs / hbm_peak
        out["note"] = "first scatter CTA start to last scatter CTA end, last timed call"
    return out


def trace_summary(tr, num_ctas: int, fields) -> dict:
    """Per-CTA trace records of one launch (rows of kTraceWords int64) -> [median, max]
    over CTAs of each phase stamp, in us from the first CTA's start."""
    tr = tr.view(-1, len(fields))[:num_ctas].cpu().double()
    fi = {n: i for i, n in enumerate(fields)}
    t0 = tr[:, fi["start"]].min()
    us = lambda col, rows=slice(None): ((tr[rows, fi[col]] - t0) / 1e3)
    loaded = tr[:, fi["tiles"]] > 0  # CTAs that loaded at least one tile
    scattered = tr[:, fi["scatter_end"]] > 0
    med_max = lambda v: [float(v.median()), float(v.max())] if v.numel() else None
    return {
        "scatter_end_us": med_max(us("scatter_end", scattered)),
        "first_tile_us": med_max(us("first_tile", loaded)),
        "flag_wait_us": med_max(tr[loaded, fi["flag_wait_ns"]] / 1e3),
        "end_us": med_max(us("end")),
        "ctas_with_tiles": int(loaded.sum()),
        "note": "one traced launch of the fused kernel, per-CTA global-timer stamps from the first CTA's "
                "start: [median, max] over CTAs",
    }


def measure_workload(wl, K: int, warmup: int, dev, stream, flush, l2: str = "flush") -> dict:
    """The whole path (route + fused dispatch/grouped GEMM) of one workload in the plan's
    own launch configuration: K timed steps (CUDA events on the launching stream, L2
    flushed between steps), nvidia-smi clocks during the timed region, the roofline of
    the fused kernel, the scatter window and one traced launch.  Used for every
    configuration besides the headline one."""
    import torch

    from moe_token_dispatch_route_gb300 import binding, workloads

    inp = workloads.make_inputs(wl, seed=0, w_device=dev)
    x, W, logits = inp["x"].to(dev), inp["W"], inp["logits"].to(dev)
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, num_ranks=wl.R, device=dev.index)
    bufs = binding.MoeBuffers(plan, dev)
    for _ in range(max(3, warmup)):
        binding.forward(plan, logits, x, W, bufs, stream)
    rc, st = binding.moe_read_status(bufs.status, stream)
    if rc != 0:
        raise SystemExit(f"{wl.name}: device status after warm-up: {st}")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        for i in range(K):
            if l2 == "flush":
                flush.fill_(float(i))
            e0, e1, e2 = ev[i]
            e0.record(stream)
            binding.route(plan, logits, bufs, stream)
            e1.record(stream)
            binding.dispatch_gemm(plan, x, W, bufs, stream)
            e2.record(stream)
        torch.cuda.synchronize(dev)
    rc, st = binding.moe_read_status(bufs.status, stream)
    if rc != 0:
        raise SystemExit(f"{wl.name}: device status after timed steps: {st}")
    hdr = bufs.workspace[:64].cpu().numpy().view("uint64")
    scatter_ns = int(hdr[25]) - int(hdr[24])
    touched = int((bufs.counts > 0).sum().item())
    step_ms = [a.elapsed_time(c) for a, _, c in ev]
    dg_ms = [b.elapsed_time(c) for _, b, c in ev]
    trace = torch.zeros(plan.info["sm_count"] * binding.TRACE_WORDS, dtype=torch.int64, device=dev)
    binding.moe_set_trace(plan, trace)
    flush.fill_(2.0)
    binding.dispatch_gemm(plan, x, W, bufs, stream)
    torch.cuda.synchronize(dev)
    binding.moe_set_trace(plan, None)
    tr = trace_summary(trace, plan.info["num_ctas"], binding.TRACE_FIELDS)

    def median_ms(fn, n=10):
        for _ in range(2):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a_, b_ in evs:
            flush.fill_(1.0)
            a_.record(stream)
            fn()
            b_.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.median(a_.elapsed_time(b_) for a_, b_ in evs)

    # the step after the path: moe_combine on Y, and the combine fused into the epilogue
    comb_out = torch.empty(wl.T, wl.N, dtype=torch.float32, device=dev)
    combine_ms = median_ms(lambda: binding.moe_combine(plan, bufs.Y, bufs.topk_w, bufs.dest, comb_out, stream))
    fused_comb_ms = median_ms(lambda: binding.dispatch_gemm_combine(plan, x, W, bufs, comb_out, stream))
    rc, st = binding.moe_read_status(bufs.status, stream)
    if rc != 0:
        raise SystemExit(f"{wl.name}: device status after the combine timing: {st}")
    del comb_out
    # the direct gather on the same plan (no receive buffers, the same bits)
    gather_ms = median_ms(lambda: binding.gather_gemm(plan, x, W, bufs, stream))
    rc, st = binding.moe_read_status(bufs.status, stream)
    if rc != 0:
        raise SystemExit(f"{wl.name}: device status after the gather timing: {st}")
    _, _, scatter_bytes = algorithmic_work(wl, touched)
    peaks = _peaks()
    # the gather's own algorithmic bytes: x once, the touched weights, Y (no receive rows)
    gather_bytes = wl.T * wl.d * 2 + touched * wl.d * wl.N * 2 + wl.S * wl.N * 4
    roof = roofline_of(wl, touched, statistics.mean(dg_ms) / 1000.0, plan.info, peaks)
    out = {
        "config": {**wl.describe(), "tile_m": plan.info["tile_m"], "tile_n": plan.info["tile_n"],
                   "num_ctas": plan.info["num_ctas"], "producer_ctas": plan.info["producer_ctas"]},
        "steps": K,
        "step_ms": statistics.median(step_ms),
        "route_ms": statistics.median([a.elapsed_time(b) for a, b, _ in ev]),
        "fused_ms": statistics.median(dg_ms),
        "fused_mean_ms": statistics.mean(dg_ms),
        "tflops": wl.flops / (statistics.median(step_ms) * 1e9),
        "tokens_per_s": wl.T / (statistics.median(step_ms) / 1000.0),
        "roofline": roof,
        "scatter": scatter_report(scatter_ns, scatter_bytes, peaks[0], plan.info),
        "touched_experts": touched,
        "trace": tr,
        "combine": {"unfused_ms": statistics.median(dg_ms) + combine_ms, "combine_ms": combine_ms,
                    "fused_ms": fused_comb_ms,
                    "note": "fused kernel + moe_combine against moe_dispatch_gemm_combine; 10 launches "
                            "each, L2 flushed; not in step_ms"},
        "direct_gather": {"ms": gather_ms, "tflops": wl.flops / (gather_ms * 1e9),
                          "frac_bf16_peak": wl.flops / (gather_ms * 1e9) / peaks[1],
                          "gbs": gather_bytes / (gather_ms * 1e6),
                          "frac_hbm": gather_bytes / (gather_ms * 1e6) / peaks[0],
                          "speedup_vs_dispatch": statistics.median(dg_ms) / gather_ms,
                          "note": "moe_gather_gemm on the same plan (A rows copied from x, no receive "
                                  "buffers, Y bit-identical); 10 launches, L2 flushed; not in step_ms"},
        "clocks": clk.summary(),
        "gpu_launches": launches_per_step(wl) * K,
    }
    del bufs, W, x, inp
    torch.cuda.empty_cache()
    return out


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float across the process group (identity when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


MULTICORE_WORKLOADS = ("mixtral", "finegrained", "deepseek_v3")  # oracle split over all host cores


def oracle_threads(wl) -> int:
    """Host threads of the oracle's timed GEMM: all cores on the Mixtral-, fine-grained-
    and DeepSeek-V3-shaped layers, one on the tiny and decode layers."""
    return max(1, os.cpu_count() or 1) if wl.name in MULTICORE_WORKLOADS else 1


class OracleSample:
    """The CPU oracle, as it stands, on a bounded sample of one workload.

    One sample = routing of all T tokens (top-k, histogram, permutation), then
    gather + fp64 grouped GEMM of the first `rows` destination rows, the GEMM's
    output rows split over `threads` host threads (each the single-threaded oracle
    on its own rows; the result is bitwise the single-threaded one).  Inputs and the
    weight slice those rows need are prepared once, outside any timing."""

    def __init__(self, wl, max_rows=512):
        import numpy as np

        import oracle
        from moe_token_dispatch_route_gb300 import workloads

        self.wl = wl
        self.oracle = oracle
        inp = workloads.make_inputs(wl, seed=0, with_weights=False)
        self.L = inp["logits"].numpy()
        self.xb = workloads.bf16_bits(inp["x"])
        ref = oracle.route(self.L, wl.k)
        rows = min(max_rows, wl.S)
        self.n_exp = oracle.expert_of_row(ref["offsets"], rows - 1) + 1
        W = workloads.make_weights(workloads.custom("w", wl.T, wl.d, self.n_exp, 1, wl.N), seed=0)
        self.Wb = workloads.bf16_bits(W)
        self.np = np

    def run(self, rows, threads=1):
        """Time one sample; returns (seconds, GEMM FLOPs of the sample)."""
        o, np = self.oracle, self.np
        rows = min(rows, self.wl.S)
        t0 = time.perf_counter()
        ref = o.route(self.L, self.wl.k)
        a_rows = o.gather(self.xb, ref["perm"][:rows], self.wl.k)
        off = np.minimum(ref["offsets"][: self.n_exp + 1], rows).astype(np.int32)
        if threads > 1:
            o.grouped_gemm_parallel(a_rows, self.Wb[: self.n_exp], off, threads)
        else:
            o.grouped_gemm(a_rows, self.Wb[: self.n_exp], off)
        secs = time.perf_counter() - t0
        return secs, 2.0 * rows * self.wl.d * self.wl.N

    def describe(self, rows, secs, threads=1):
        return {"sample": f"routing of all {self.wl.T} tokens + gather and fp64 GEMM of the first "
                          f"{rows} destination rows (output rows split over {threads} host threads), "
                          f"{secs:.2f} s; TFLOP/s = sampled GEMM FLOPs / sample time",
                "cores": threads, "kind": "oracle"}


def _oracle_rows(wl, threads: int, seconds: float) -> int:
    """Destination rows of an oracle sample that takes about `seconds` on `threads`
    host threads, from a timed 8-row single-thread calibration."""
    cal = OracleSample(wl, max_rows=8)
    secs8, _ = cal.run(8)
    per_row = max(secs8, 1e-4) / 8
    return max(1, min(wl.S, int(threads * seconds / per_row)))


def cpu_baseline(wl, seconds=15.0):
    """The oracle timed once on about `seconds` of work on the host cores (all of
    them on the three large layers); returns (TFLOP/s, info, seconds)."""
    threads = oracle_threads(wl)
    rows = _oracle_rows(wl, threads, seconds)
    s = OracleSample(wl, max_rows=rows)
    secs, flops = s.run(rows, threads)
    return flops / secs / 1e12, s.describe(rows, secs, threads), secs


def run_reference(args, wl):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    # each step is one oracle sample, sized so that warm-up + timed steps take about two minutes
    threads = oracle_threads(wl)
    per_step = max(0.2, 120.0 / max(1, args.steps + args.warmup))
    rows = _oracle_rows(wl, threads, per_step)
    sample = OracleSample(wl, max_rows=rows)
    for _ in range(args.warmup):
        sample.run(rows, threads)
    times = []
    flops = 0.0
    for _ in range(args.steps):
        secs, flops = sample.run(rows, threads)
        times.append(secs)
    total = sum(times)
    value = len(times) * flops / total / 1e12
    info = sample.describe(rows, statistics.median(times), threads)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {**wl.describe(), "sample_rows_per_step": rows},
            "cpu_baseline": {"value": value, "unit": UNIT, **info},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def time_swiglu_ffn(wl, inp, x, logits, dev, stream, flush, reps=20):
    """The whole gated expert FFN of the workload's shape with F = N, timed on its
    own: route -> fused dispatch + gated up-projection (W1 [E, d, 2F]) -> grouped
    down projection (W2 [E, F, d]) -> combine.  Per-kernel medians over `reps`
    steps, L2 flushed between steps."""
    import torch

    from moe_token_dispatch_route_gb300 import binding, workloads

    F = wl.N
    W1, W2 = workloads.make_ffn_weights(wl, F, seed=0, device=dev)
    up = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, 2 * F, num_ranks=wl.R, device=dev.index)
    bu = binding.MoeBuffers(up, dev, out="H")
    down = binding.moe_plan(wl.T, F, wl.E, wl.k, wl.d, device=dev.index)
    ws = torch.zeros(down.workspace_bytes // 4 + 64, dtype=torch.int32, device=dev)
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    Y2 = torch.empty(wl.S, wl.d, dtype=torch.float32, device=dev)
    out = torch.empty(wl.T, wl.d, dtype=torch.float32, device=dev)

    def step(evs=None):
        rec = (lambda i: evs[i].record(stream)) if evs else (lambda i: None)
        rec(0)
        binding.route(up, logits, bu, stream)
        rec(1)
        binding.dispatch_gemm_swiglu(up, x, W1, bu, stream)
        rec(2)
        binding.moe_grouped_gemm(down, bu.H, bu.offsets, W2, Y2, ws, st, stream)
        rec(3)
        binding.moe_combine(down, Y2, bu.topk_w, bu.dest, out, stream)
        rec(4)

    for _ in range(3):
        step()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(reps)]
    for i in range(reps):
        flush.fill_(float(i))
        step(ev[i])
    torch.cuda.synchronize(dev)
    for s_ in (bu.status, st):
        rc, status = binding.moe_read_status(s_, stream)
        if rc != 0:
            raise SystemExit(f"device status in the FFN timing: {status}")
    med = [statistics.median(e[j].elapsed_time(e[j + 1]) for e in ev) for j in range(4)]
    total = statistics.median(e[0].elapsed_time(e[4]) for e in ev)
    up_flops = 2.0 * wl.S * wl.d * 2 * F
    down_flops = 2.0 * wl.S * F * wl.d
    _, tf_peak, _, peak_src = _peaks()
    res = {"F": F, "ms": total, "route_ms": med[0], "up_ms": med[1], "down_ms": med[2],
           "combine_ms": med[3],
           "up_tflops": up_flops / (med[1] * 1e9), "down_tflops": down_flops / (med[2] * 1e9),
           "layer_tflops": (up_flops + down_flops) / (total * 1e9),
           "note": "gated expert FFN with F = N: route -> dispatch + SwiGLU up-projection "
                   "(bf16 H) -> grouped down projection -> combine; timed separately, not in value"}
    res["up_frac"] = res["up_tflops"] / tf_peak
    res["down_frac"] = res["down_tflops"] / tf_peak
    res["peak_source"] = f"{peak_src} (bf16 burst)"
    res["tile_m"] = [up.info["tile_m"], down.info["tile_m"]]
    del W1, W2, bu, Y2, out
    return res


def run_kernel_only(args, wl):
    """A short run for profilers: route once, warm up, then `args.steps` launches of one
    kernel with L2 flushed between them; prints one JSON line with their median."""
    import torch

    from moe_token_dispatch_route_gb300 import binding, build as _build, workloads

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _build.build()
    inp = workloads.make_inputs(wl, seed=0, w_device=dev)
    x, W, logits = inp["x"].to(dev), inp["W"], inp["logits"].to(dev)
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, num_ranks=wl.R, tile_n=args.tile_n,
                            tile_m=args.tile_m, producer_ctas=args.producer_ctas, device=0)
    bufs = binding.MoeBuffers(plan, dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    binding.forward(plan, logits, x, W, bufs, stream)  # routing + receive rows in place
    ws = torch.zeros(plan.workspace_bytes // 4 + 64, dtype=torch.int32, device=dev)
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    if args.kernel_only == "fused":
        launch = lambda: binding.dispatch_gemm(plan, x, W, bufs, stream)
    elif args.kernel_only == "gather":
        launch = lambda: binding.gather_gemm(plan, x, W, bufs, stream)
    else:
        if wl.R != 1:
            raise SystemExit("--kernel-only grouped needs one rank buffer (R = 1)")
        launch = lambda: binding.moe_grouped_gemm(plan, bufs.recv[0], bufs.offsets, W, bufs.Y, ws, st, stream)
    for _ in range(args.warmup):
        flush.fill_(1.0)
        launch()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a_, b_ in evs:
        flush.fill_(1.0)
        a_.record(stream)
        launch()
        b_.record(stream)
    torch.cuda.synchronize(dev)
    for s_ in (bufs.status, st):
        rc, words = binding.moe_read_status(s_, stream)
        if rc != 0:
            raise SystemExit(f"device status: {words}")
    print(json.dumps({"kernel_only": args.kernel_only, "config": wl.describe(), "launches": args.steps,
                      "ms": statistics.median(a_.elapsed_time(b_) for a_, b_ in evs),
                      "tile_m": plan.info["tile_m"], "tile_n": plan.info["tile_n"]}), flush=True)
    return 0


def run_ours(args, wl):
    import torch

    from moe_token_dispatch_route_gb300 import binding, workloads

    world, rank, local = _dist()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the CUDA library has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    from moe_token_dispatch_route_gb300 import build as _build
    _build.build()

    inp = workloads.make_inputs(wl, seed=0, w_device=dev)
    x = inp["x"].to(dev)
    W = inp["W"]
    logits = inp["logits"].to(dev)
    plan = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, num_ranks=wl.R, tile_n=args.tile_n, tile_m=args.tile_m,
                            producer_ctas=args.producer_ctas, device=local)
    bufs = binding.MoeBuffers(plan, dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(max(3, args.warmup)):
        binding.forward(plan, logits, x, W, bufs, stream)
    rc, st = binding.moe_read_status(bufs.status, stream)
    if rc != 0:
        raise SystemExit(f"device status after warm-up: {st}")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        for i in range(K):
            if args.l2 == "flush":
                flush.fill_(float(i))  # evict L2 between steps (outside the events)
            e0, e1, e2 = ev[i]
            e0.record(stream)
            binding.route(plan, logits, bufs, stream)
            e1.record(stream)
            binding.dispatch_gemm(plan, x, W, bufs, stream)
            e2.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    rc, st = binding.moe_read_status(bufs.status, stream)
    if rc != 0:
        raise SystemExit(f"device status after timed steps: {st}")
    hdr = bufs.workspace[:64].cpu().numpy().view("uint64")
    scatter_ns = int(hdr[25]) - int(hdr[24])  # last call's scatter window (words 48..51)
    touched = int((bufs.counts > 0).sum().item())
    step_ms = [a.elapsed_time(c) for a, _, c in ev]
    route_ms = [a.elapsed_time(b) for a, b, _ in ev]
    dg_ms = [b.elapsed_time(c) for _, b, c in ev]
    total_s = sum(step_ms) / 1000.0
    total_s = max_over_ranks(total_s, world, dev)

    # the step after the path (combine), timed on its own: reads Y, writes [T, N]
    comb_out = torch.empty(wl.T, wl.N, dtype=torch.float32, device=dev)
    for _ in range(3):
        binding.moe_combine(plan, bufs.Y, bufs.topk_w, bufs.dest, comb_out, stream)
    cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
    for a_, b_ in cev:
        flush.fill_(1.0)
        a_.record(stream)
        binding.moe_combine(plan, bufs.Y, bufs.topk_w, bufs.dest, comb_out, stream)
        b_.record(stream)
    torch.cuda.synchronize(dev)
    combine_ms = statistics.median(a_.elapsed_time(b_) for a_, b_ in cev)
    del comb_out

    # the step before the path (GPU router logits), timed on its own: reads x and W_r
    W_r = inp["W_r"].to(dev)
    bias_d = inp["bias"].to(dev) if wl.bias != "none" else None
    L_gpu = torch.empty_like(logits)
    for _ in range(3):
        binding.moe_router_logits(plan, x, W_r, bias_d, L_gpu, stream)
    rev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
    for a_, b_ in rev:
        flush.fill_(1.0)
        a_.record(stream)
        binding.moe_router_logits(plan, x, W_r, bias_d, L_gpu, stream)
        b_.record(stream)
    torch.cuda.synchronize(dev)
    router_ms = statistics.median(a_.elapsed_time(b_) for a_, b_ in rev)
    del L_gpu

    # one traced launch: where the fused kernel's time goes, per CTA (moe_set_trace)
    trace = torch.zeros(plan.info["sm_count"] * binding.TRACE_WORDS, dtype=torch.int64, device=dev)
    binding.moe_set_trace(plan, trace)
    flush.fill_(2.0)
    binding.dispatch_gemm(plan, x, W, bufs, stream)
    torch.cuda.synchronize(dev)
    binding.moe_set_trace(plan, None)
    trace_info = trace_summary(trace, plan.info["num_ctas"], binding.TRACE_FIELDS)
    del trace

    # the same step captured once in a CUDA graph and replayed (launch overhead removed)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        binding.forward(plan, logits, x, W, bufs)
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        binding.forward(plan, logits, x, W, bufs)
    for _ in range(3):
        graph.replay()
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
    for a_, b_ in gev:
        flush.fill_(1.0)
        a_.record(stream)
        graph.replay()
        b_.record(stream)
    torch.cuda.synchronize(dev)
    rc, st = binding.moe_read_status(bufs.status, stream)
    if rc != 0:
        raise SystemExit(f"device status after the graph timing: {st}")
    graph_ms = statistics.median(a_.elapsed_time(b_) for a_, b_ in gev)
    del graph

    # the direct-gather variant of the fused kernel (no receive buffers), timed on its own
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
    for _ in range(3):
        binding.gather_gemm(plan, x, W, bufs, stream)
    for a_, b_ in gev:
        flush.fill_(1.0)
        a_.record(stream)
        binding.gather_gemm(plan, x, W, bufs, stream)
        b_.record(stream)
    torch.cuda.synchronize(dev)
    rc, st = binding.moe_read_status(bufs.status, stream)
    if rc != 0:
        raise SystemExit(f"device status after the gather timing: {st}")
    gather_ms = statistics.median(a_.elapsed_time(b_) for a_, b_ in gev)
    binding.dispatch_gemm(plan, x, W, bufs, stream)  # leave Y as the path computes it

    # the fused kernel with a bf16 Y (MOE_OUT_BF16), timed on its own
    plan_b = binding.moe_plan(wl.T, wl.d, wl.E, wl.k, wl.N, num_ranks=wl.R, tile_n=args.tile_n, tile_m=args.tile_m,
                              producer_ctas=args.producer_ctas, out_dtype=binding.MOE_OUT_BF16,
                              device=local)
    bufs_b = binding.MoeBuffers(plan_b, dev)
    binding.route(plan_b, logits, bufs_b, stream)
    for _ in range(3):
        binding.dispatch_gemm(plan_b, x, W, bufs_b, stream)
    bev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
    for a_, b_ in bev:
        flush.fill_(1.0)
        a_.record(stream)
        binding.dispatch_gemm(plan_b, x, W, bufs_b, stream)
        b_.record(stream)
    torch.cuda.synchronize(dev)
    rc, st = binding.moe_read_status(bufs_b.status, stream)
    if rc != 0:
        raise SystemExit(f"device status after the bf16-output timing: {st}")
    ybf16_ms = statistics.median(a_.elapsed_time(b_) for a_, b_ in bev)
    del bufs_b, plan_b

    # the combine fused into the GEMM epilogue: one launch, against the unfused chain (the
    # fused kernel writing Y + moe_combine reading it)
    fused_combine = None
    if True:
        comb_out = torch.empty(wl.T, wl.N, dtype=torch.float32, device=dev)
        for _ in range(3):
            binding.dispatch_gemm_combine(plan, x, W, bufs, comb_out, stream)
        fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
        for a_, b_ in fev:
            flush.fill_(1.0)
            a_.record(stream)
            binding.dispatch_gemm_combine(plan, x, W, bufs, comb_out, stream)
            b_.record(stream)
        torch.cuda.synchronize(dev)
        rc, st = binding.moe_read_status(bufs.status, stream)
        if rc != 0:
            raise SystemExit(f"device status after the fused-combine timing: {st}")
        fc_ms = statistics.median(a_.elapsed_time(b_) for a_, b_ in fev)
        unfused = statistics.median(dg_ms) + combine_ms
        fused_combine = {"ms": fc_ms, "unfused_ms": unfused, "speedup_vs_unfused": unfused / fc_ms,
                         "tflops": wl.flops / (fc_ms * 1e9),
                         "note": "moe_dispatch_gemm_combine: the fused kernel whose epilogue writes each "
                                 "gate-weighted row into its token's row of out [T, N] (stored by the "
                                 "token's lowest expert, then added in expert order), no Y; unfused = "
                                 "fused kernel (writes Y) + moe_combine; 20 launches, L2 flushed; not in value"}
        del comb_out
        binding.dispatch_gemm(plan, x, W, bufs, stream)  # leave Y as the path computes it

    ffn = None
    if args.ffn == "on" or (args.ffn == "auto" and wl.name == "mixtral"):
        ffn = time_swiglu_ffn(wl, inp, x, logits, dev, stream, flush)

    # end to end through the same ABI: every step copies its inputs in from pinned host
    # memory, runs the path and copies Y out to pinned host memory.  The steps are pipelined
    # over two buffer sets on three streams (copy in, compute, copy out), so step i's copies
    # overlap its neighbours' work.  When the weights fit in twice the L2, each step also
    # flushes L2 on the compute stream, inside the timed region; larger weights evict it.
    w_bytes = wl.E * wl.d * wl.N * 2
    e2e_flush = w_bytes < 2 * L2_BYTES
    x_h = inp["x"].pin_memory()
    l_h = inp["logits"].pin_memory()
    sets = []
    for j in range(2):
        b_j = bufs if j == 0 else binding.MoeBuffers(plan, dev)
        sets.append({"bufs": b_j, "x": torch.empty_like(x), "l": torch.empty_like(logits),
                     "y": torch.empty(b_j.Y.shape, dtype=b_j.Y.dtype).pin_memory()})
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    E2E = max(3, args.e2e_steps)

    def e2e_steps(n):
        ev = {key: [torch.cuda.Event() for _ in range(n)] for key in ("in", "comp", "out")}
        for i in range(n):
            st = sets[i % 2]
            if i >= 2:
                s_in.wait_event(ev["comp"][i - 2])  # step i-2 has read this set's inputs
            with torch.cuda.stream(s_in):
                st["x"].copy_(x_h, non_blocking=True)
                st["l"].copy_(l_h, non_blocking=True)
                ev["in"][i].record(s_in)
            stream.wait_event(ev["in"][i])
            if i >= 2:
                stream.wait_event(ev["out"][i - 2])  # this set's Y of step i-2 is out
            if e2e_flush:
                flush.fill_(float(i))
            binding.forward(plan, st["l"], st["x"], W, st["bufs"], stream)
            ev["comp"][i].record(stream)
            s_out.wait_event(ev["comp"][i])
            with torch.cuda.stream(s_out):
                st["y"].copy_(st["bufs"].Y, non_blocking=True)
                ev["out"][i].record(s_out)
        return ev

    e2e_steps(2)
    torch.cuda.synchronize(dev)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(s_in)
    e2e_steps(E2E)
    e_end.record(s_out)
    torch.cuda.synchronize(dev)
    for st in sets:
        rc, st_words = binding.moe_read_status(st["bufs"].status, stream)
        if rc != 0:
            raise SystemExit(f"device status after the end-to-end steps: {st_words}")
    e2e_s = max_over_ranks(e_start.elapsed_time(e_end) / 1000.0, world, dev)
    h2d = x_h.numel() * x_h.element_size() + l_h.numel() * l_h.element_size()
    d2h = sets[0]["y"].numel() * sets[0]["y"].element_size()

    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return 0

    # every other configuration of the benchmark, each in its own plan's launch
    # configuration, measured in the same run (rank 0 only)
    others = {}
    names = [] if args.workloads == "none" else (
        [n for n in workloads.WORKLOADS if n != wl.name] if args.workloads == "others"
        else [n for n in args.workloads.split(",") if n and n != wl.name])
    if names:
        del sets, bufs, W, x, logits, inp, flush
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        for name in names:
            others[name] = measure_workload(workloads.WORKLOADS[name], max(20, K), args.warmup, dev,
                                            stream, flush, args.l2)

    hbm_peak, tf_peak, tf_sustained, peak_src = _peaks()
    flops, alg_bytes, scatter_bytes = algorithmic_work(wl, touched)
    value = world * K * flops / total_s / 1e12
    dg_avg_s = statistics.mean(dg_ms) / 1000.0
    roof = roofline_of(wl, touched, dg_avg_s, plan.info, (hbm_peak, tf_peak, tf_sustained, peak_src))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": 1000.0 * total_s / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**wl.describe(), "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": (f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write)" if args.l2 == "flush"
                          else f"no flush: inputs larger than L2 (W {wl.E * wl.d * wl.N * 2 >> 20} MiB)"),
                   "tile_m": plan.info["tile_m"], "tile_n": plan.info["tile_n"],
                   "producer_ctas": plan.info["producer_ctas"],
                   "num_ctas": plan.info["num_ctas"], "stages": plan.info["stages"]},
        "tokens_per_s": world * K * wl.T / total_s,
        "pct_bf16_peak": 100.0 * value / world / tf_peak,
        "route_ms": statistics.median(route_ms),
        "dispatch_gemm_ms": statistics.median(dg_ms),
        "roofline": roof,
        "fused_tflops": flops / dg_avg_s / 1e12,
        "scatter": scatter_report(scatter_ns, scatter_bytes, hbm_peak, plan.info),
        "touched_experts": touched,
        "router": {"ms": router_ms, "flops": 2.0 * wl.T * wl.d * wl.E,
                   "tflops": 2.0 * wl.T * wl.d * wl.E / (router_ms * 1e9),
                   "note": "moe_router_logits (step before the path; fp32 CUDA-core FMAs in a fixed "
                           "order), timed separately; not in value"},
        "combine": {"ms": combine_ms, "bytes": wl.S * wl.N * 4 + wl.T * wl.N * 4,
                    "gbs": (wl.S * wl.N * 4 + wl.T * wl.N * 4) / (combine_ms * 1e6),
                    "frac_hbm": (wl.S * wl.N * 4 + wl.T * wl.N * 4) / (combine_ms * 1e6) / hbm_peak,
                    "note": "moe_combine (step after the path), timed separately; not in value"},
        "trace": trace_info,
        "cuda_graph": {"step_ms": graph_ms, "eager_step_ms": statistics.median(step_ms),
                       "note": "route + fused kernel captured in one CUDA graph and replayed; "
                               "20 replays, L2 flushed; not in value"},
        "direct_gather": {"ms": gather_ms, "tflops": flops / (gather_ms * 1e9),
                          "dispatch_gemm_ms": statistics.median(dg_ms),
                          "speedup_vs_dispatch": statistics.median(dg_ms) / gather_ms,
                          "frac_bf16_peak": flops / (gather_ms * 1e9) / _peaks()[1],
                          "note": "moe_gather_gemm on the same plan: A rows copied from x by perm straight "
                                  "into the GEMM's shared memory by cp.async warps, no receive buffers, no "
                                  "scatter phase, Y bit-identical to the dispatch; "
                                  "20 launches, L2 flushed; not in value"},
        "y_bf16": {"ms": ybf16_ms, "tflops": flops / (ybf16_ms * 1e9),
                   "note": "moe_dispatch_gemm with out_dtype = MOE_OUT_BF16 (Y rounded once to bf16, "
                           "half the Y bytes); 20 launches, L2 flushed; not in value"},
        "combine_fused": fused_combine,
        "swiglu_ffn": ffn,
        "e2e": {"value": world * E2E * flops / e2e_s / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": E2E,
                "note": "through the C ABI with pinned host buffers: every step copies x and the "
                        "logits in and Y out; steps pipelined over two buffer sets on three streams; "
                        + ("L2 flushed inside each step" if e2e_flush else
                           f"no flush: the weights ({w_bytes >> 20} MiB) exceed the L2")},
        "gpu_launches": launches_per_step(wl) * K,
        "clocks": clk.summary(),
        "workloads": others or None,
    }
    if not args.no_cpu_baseline:
        v, info, _ = cpu_baseline(wl)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, **info}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = _args(argv)
    from moe_token_dispatch_route_gb300 import workloads
    if args.shape:
        v = [int(t) for t in args.shape.split(",")]
        wl = workloads.custom("custom_" + "x".join(map(str, v)), *v)
    else:
        wl = workloads.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)
    if args.kernel_only:
        return run_kernel_only(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
