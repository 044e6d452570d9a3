#!/usr/bin/env python3
"""Throughput of the device-wide single-pass scan on GB300.

One step is one call of the C entry point dwp_scan_exclusive (u32 addition)
over n = 2^28 full-range values already resident in HBM: scratch clear plus
the single-pass scan kernel, i.e. every step of the plain scan's hot path.
The input (1 GiB) and output (1 GiB) are each larger than the 129 MB L2, so
no L2 flush is needed between steps.

Printed (rank 0, one JSON line): Gelem/s of the whole job, the roofline of the
scan kernel against the measured HBM copy bandwidth, the same metric end to
end from pinned host memory (copies inside the timed region), the oracle
timed on the host cores, SM clocks sampled during the timed region, and the
other scans, the segmented scan and the compaction measured the same way
under "secondary".

--impl reference times the sequential CPU oracle instead (the only other
place this script runs oracle code), on a bounded slice of the same input.
With torchrun (N > 1) every rank scans its own replica of the input (no
collective on the data path); rank 0 reports max-over-ranks time.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "u32 exclusive scan Gelem/s and HBM GB/s as % of peak at n=2^28; segscan Gelem/s"
N_FULL = 1 << 28
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "scan_u32_exclusive_2p28.md")
KERNEL_SOURCES = ["device_wide_prefix_gb300/csrc/scan.cu", "device_wide_prefix_gb300/csrc/device.cuh"]
CSRC = "device_wide_prefix_gb300/csrc/"
# ncu summary and kernel sources behind each secondary entry's traffic figure
SECONDARY_PROFILES = {
    "segscan_u32_exclusive": ("segscan_u32_skewed.md", [CSRC + "segscan.cu", CSRC + "device.cuh"]),
    "compact_16B_records": ("compact_16B_records.md", [CSRC + "compact.cu", CSRC + "device.cuh"]),
    "linear_recurrence_f32": ("recurrence_f32_2p28.md", [CSRC + "recurrence.cu", CSRC + "device.cuh"]),
    "segreduce_u32": ("segreduce_u32_skewed.md", [CSRC + "segreduce.cu", CSRC + "device.cuh"]),
    "u32_add_exclusive_2p20": ("scan_small_u32_2p20.md", [CSRC + "scan_small.cu", CSRC + "device.cuh"]),
}


def kernel_hash(paths=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def profiled_traffic(summary=PROFILE_SUMMARY, sources=KERNEL_SOURCES):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    if not os.path.exists(summary):
        return None
    fields = {}
    with open(summary) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_source_sha256_16") != kernel_hash(sources):
        return None
    try:
        return int(fields["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (100 ms) while running; summary of those inside a window."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    @staticmethod
    def _ts(s: str) -> float:
        s = s.strip()
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return time.mktime(time.strptime(s.split(".")[0], fmt.split(".")[0])) + (
                    float("0." + s.split(".")[1]) if "." in s else 0.0)
            except ValueError:
                continue
        return 0.0

    def summary(self, t0: float, t1: float) -> dict:
        rows = []
        for row in csv.reader(io.StringIO("\n".join(self.lines))):
            if len(row) < 10:
                continue
            try:
                rows.append({"t": self._ts(row[0]), "sm": float(row[2]), "max": float(row[3]),
                             "power": float(row[4]) if row[4].strip() not in ("[N/A]", "") else 0.0,
                             "hw_slowdown": row[6].strip(), "hw_thermal": row[7].strip(),
                             "sw_thermal": row[8].strip(), "sw_power_cap": row[9].strip()})
            except ValueError:
                continue
        inside = [r for r in rows if t0 - 0.05 <= r["t"] <= t1 + 0.05]
        used = inside if inside else rows[-3:]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "no nvidia-smi samples"}
        reasons = set()
        for r in used:
            for key, name in (("hw_slowdown", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"),
                              ("sw_power_cap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median([r["sm"] for r in used])),
                "sm_max_mhz": max(r["max"] for r in used), "reasons": sorted(reasons),
                "samples": len(used), "power_w_max": max(r["power"] for r in used),
                "window": "timed region" if inside else "last samples (timed region shorter than the sampling period)"}


class NvmlClockSampler:
    """SM clock, clock-event reasons and power read through NVML (ctypes) on a
    thread every `period` seconds: a timed region of a few milliseconds gets
    several samples, where nvidia-smi's 100 ms period gives one.  Reads only;
    nothing is set.  `ok` is False when NVML cannot be loaded."""

    # nvmlClocksEventReasons bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, period: float = 0.0005):
        import ctypes
        import threading
        self.ok = False
        self.period = period
        self.samples = []
        self._stop = threading.Event()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
                return
            reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint(0)
            nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))  # NVML_CLOCK_SM
        except (OSError, AttributeError):
            return
        self.max_mhz = float(mx.value)
        self.ok = True

        def run():
            clk, rs, mw = ctypes.c_uint(0), ctypes.c_ulonglong(0), ctypes.c_uint(0)
            while not self._stop.is_set():
                if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                        reasons(h, ctypes.byref(rs)) == 0:
                    nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
                    self.samples.append((time.time(), float(clk.value), int(rs.value), mw.value / 1e3))
                time.sleep(period)

        self._thread = threading.Thread(target=run, daemon=True)
        self._thread.start()

    def stop(self):
        if self.ok:
            self._stop.set()
            self._thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict | None:
        used = [s for s in self.samples if t0 <= s[0] <= t1]
        if not used:
            return None
        reasons = sorted({name for s in used for bit, name in self.REASONS.items() if s[2] & bit})
        return {"sm_mhz": float(np.median([s[1] for s in used])), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(used), "power_w_max": max(s[3] for s in used),
                "window": "timed region", "source": "NVML, %.1f ms period" % (self.period * 1e3)}


def clock_record(nvml, smi, t0: float, t1: float) -> dict | None:
    """The NVML samples of the timed region when there are any, else the
    nvidia-smi ones; the other source's summary rides along."""
    a = nvml.summary(t0, t1) if nvml is not None and nvml.ok else None
    b = smi.summary(t0, t1) if smi is not None else None
    if a is None:
        return b
    if b is not None:
        a["nvidia_smi"] = {k: b.get(k) for k in ("sm_mhz", "reasons", "samples")}
    return a


def max_over_ranks(dist, v: float, device) -> float:
    """The largest of every rank's v (a time), through one all-reduce on
    `device` (the GPU under NCCL; the CPU under gloo).  With dist None (one
    process) v itself."""
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(units_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput of `world` replicas, each processing
    units_per_rank, timed by the slowest rank: units per second / 1e9."""
    return world * units_per_rank / (ms_max * 1e-3) / 1e9


def host_cores() -> dict:
    """Host CPU cores: all of them, and those this process may run on."""
    try:
        usable = len(os.sched_getaffinity(0))
    except AttributeError:
        usable = os.cpu_count()
    return {"host_cores": os.cpu_count(), "usable_cores": usable}


# ---------------------------------------------------------------- reference arm

def run_reference(args, rank: int) -> None:
    if rank != 0:
        return
    import oracle
    ref = oracle.Oracle()
    x = synth.u32_full_values(N_FULL)
    # calibrate, then size each step so the whole run stays near 60 s
    t = time.perf_counter()
    ref.scan_u32_add(x[: 1 << 22], False)
    rate = (1 << 22) / max(time.perf_counter() - t, 1e-6)
    per_step = int(min(N_FULL, max(1 << 20, 60.0 * rate / max(args.steps + args.warmup, 1))))
    per_step -= per_step % 4
    sl = x[:per_step]
    for _ in range(args.warmup):
        ref.scan_u32_add(sl, False)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ref.scan_u32_add(sl, False)
    dt = time.perf_counter() - t0
    val = per_step * args.steps / dt / 1e9
    sample = "first %d elements of the n=2^28 full-range u32 input per step" % per_step
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "Gelem/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic (SplitMix64 seed 0xD3B00002)",
        "config": {"workload": "u32 exclusive sum scan, n=2^28, values uniform in [0, 2^32)",
                   "n": N_FULL, "sample_elements_per_step": per_step},
        "cpu_baseline": {"value": val, "unit": "Gelem/s", "cores": 1, "kind": "oracle",
                         "sample": sample, **host_cores()},
        "e2e": {"value": val, "unit": "Gelem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm

def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--only", default=None,
                    choices=["scan", "segscan", "compact", "recurrence", "segreduce", "compact_staged"],
                    help="time only this workload (at --log2n) and print its entry; for "
                         "profiler captures")
    ap.add_argument("--log2n", type=int, default=28,
                    help="problem size 2^k (default 28, the benchmarked workload; smaller "
                         "sizes are for profiler captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    args.steps = max(args.steps, 1)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.only:
        run_only(args)
        return

    import torch
    import device_wide_prefix_gb300 as dwp

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    lib = dwp.load()
    stream = torch.cuda.current_stream(dev)
    sptr = int(stream.cuda_stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    def ranks_max(v: float) -> float:
        return max_over_ranks(dist, v, dev)

    import ctypes
    n = 1 << args.log2n
    x_host = torch.from_numpy(synth.u32_full_values(n).view(np.int32)).pin_memory()
    wl = "u32 exclusive sum scan, n=2^%d, values uniform in [0, 2^32)" % args.log2n
    x = x_host.to(dev)
    y = torch.empty_like(x)
    need = dwp.scan_scratch_bytes(n)
    scratch = dwp.alloc_scratch(need, dev)
    sb = ctypes.c_size_t(need)
    f = lib.dwp_scan_exclusive
    a_in, a_out, a_s = ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(scratch.data_ptr())
    a_st = ctypes.c_void_p(sptr)

    def step():
        st = f(dwp.DWP_U32_ADD, a_in, a_out, n, a_s, ctypes.byref(sb), a_st)
        if st != 0:
            raise RuntimeError(dwp.status_string(st))

    clocks = ClockSampler(local_rank) if rank == 0 else None
    nvml_clocks = NvmlClockSampler(local_rank) if rank == 0 else None
    for _ in range(args.warmup):
        step()
    barrier()
    if dwp.read_status(scratch) != dwp.DWP_SUCCESS:
        raise RuntimeError("device status after warm-up: %s" % dwp.status_string(dwp.read_status(scratch)))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier()
    wall0 = time.time()
    e0.record(stream)
    for k in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    wall1 = time.time()
    st = dwp.read_status(scratch)
    if st != dwp.DWP_SUCCESS:
        raise RuntimeError("device status after timed steps: %s" % dwp.status_string(st))
    ms = ranks_max(e0.elapsed_time(e1) / args.steps)
    value = replica_value(n, world, ms)
    # median and minimum per step from a second, separate pass with an event
    # before every step.  Those events are kept out of the timed region
    # above: an event between two calls stops the next call's launch from
    # overlapping the previous call (programmatic dependent launch), so each
    # step would pay its launch in full.
    for k in range(args.steps):
        marks[k].record(stream)
        step()
    marks[args.steps].record(stream)
    barrier()
    per_step = sorted(marks[k].elapsed_time(marks[k + 1]) for k in range(args.steps))

    # end to end from pinned host memory through the same C entry point:
    # every step copies its input in, scans it and copies the result out.
    # Serially on one stream, and pipelined over two streams with their own
    # device buffers, so that one step's copy-out overlaps the next step's
    # copy-in (the two directions use separate copy engines).
    e2e_steps = max(3, min(args.steps, 20))
    y_host = [torch.empty(n, dtype=torch.int32).pin_memory() for _ in range(2)]
    for _ in range(2):
        x.copy_(x_host, non_blocking=True); step(); y_host[0].copy_(y, non_blocking=True)
    barrier()
    e0.record(stream)
    for _ in range(e2e_steps):
        x.copy_(x_host, non_blocking=True)
        step()
        y_host[0].copy_(y, non_blocking=True)
    e1.record(stream)
    barrier()
    e2e_serial_ms = ranks_max(e0.elapsed_time(e1) / e2e_steps)
    sides = [torch.cuda.Stream(dev) for _ in range(2)]
    xs, ys, scr2 = [x, torch.empty_like(x)], [y, torch.empty_like(y)], [scratch, dwp.alloc_scratch(need, dev)]

    # Copies in one direction go one after another: a step's copy-in waits
    # for the previous step's copy-in, its copy-out for the previous
    # copy-out.  Left free, the two streams could fall into step (both
    # copying in, then both copying out), and no copy-out would overlap a
    # copy-in; two copies in one direction only share the link anyway.
    done_in, done_out = {}, {}

    def e2e_step(k):
        j = k % 2
        s = sides[j]
        with torch.cuda.stream(s):
            if k - 1 in done_in:
                s.wait_event(done_in.pop(k - 1))
            xs[j].copy_(x_host, non_blocking=True)
            done_in[k] = torch.cuda.Event()
            done_in[k].record(s)
            st = f(dwp.DWP_U32_ADD, ctypes.c_void_p(xs[j].data_ptr()), ctypes.c_void_p(ys[j].data_ptr()), n,
                   ctypes.c_void_p(scr2[j].data_ptr()), ctypes.byref(sb), ctypes.c_void_p(int(s.cuda_stream)))
            if st != 0:
                raise RuntimeError(dwp.status_string(st))
            if k - 1 in done_out:
                s.wait_event(done_out.pop(k - 1))
            y_host[j].copy_(ys[j], non_blocking=True)
            done_out[k] = torch.cuda.Event()
            done_out[k].record(s)

    for k in range(2):
        e2e_step(k)
    barrier()
    done_in.clear()
    done_out.clear()
    e0.record(stream)
    for s in sides:
        s.wait_event(e0)
    for k in range(e2e_steps):
        e2e_step(k)
    for s in sides:
        stream.wait_stream(s)
    e1.record(stream)
    barrier()
    e2e_ms = ranks_max(e0.elapsed_time(e1) / e2e_steps)
    for j in range(2):
        if dwp.read_status(scr2[j]) != dwp.DWP_SUCCESS:
            raise RuntimeError("device status after the end-to-end steps")
    del xs, ys, scr2
    if clocks is not None:
        clocks.stop()
    if nvml_clocks is not None:
        nvml_clocks.stop()

    peaks = measured_peaks()
    alg_bytes = 8 * n
    achieved = alg_bytes / (ms * 1e-3) / 1e9

    secondary = {}
    if not args.no_secondary and rank == 0:
        secondary = measure_secondary(dwp, lib, dev, stream, peaks, x, y, scratch, need)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    # the oracle reads a pageable copy, as the reference arm does
    cpu = cpu_baseline(x_host.numpy().view(np.uint32).copy(), args.cpu_budget_s)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "Gelem/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "ms_median": per_step[len(per_step) // 2],
        "ms_min": per_step[0],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u32",
        "data": "synthetic (SplitMix64 seed 0xD3B00002, values uniform in [0, 2^32))",
        "config": {"workload": wl,
                   "n": n, "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (1 GiB in + 1 GiB out vs 129 MB L2); no flush"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "timing": "CUDA events over the whole C call (scratch-clear kernel + scan kernel)",
                     "traffic": profiled_traffic()},
        "cpu_baseline": cpu,
        "e2e": {"value": n / (e2e_ms * 1e-3) / 1e9, "unit": "Gelem/s",
                "h2d_bytes_per_step": 4 * n, "d2h_bytes_per_step": 4 * n,
                "ms_per_step": e2e_ms, "steps": e2e_steps,
                "how": "pinned host in and out, two steps in flight on two streams",
                "serial_one_stream_ms_per_step": e2e_serial_ms},
        "gpu_launches": 2 * args.steps,
        "clocks": clock_record(nvml_clocks, clocks, wall0, wall1),
        "secondary": secondary,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def cpu_baseline(x: np.ndarray, budget_s: float) -> dict:
    import oracle
    ref = oracle.Oracle()
    runs, t_total = 0, 0.0
    while t_total < budget_s or runs == 0:
        t = time.perf_counter()
        ref.scan_u32_add(x, False)
        t_total += time.perf_counter() - t
        runs += 1
        if runs >= 100:
            break
    return {"value": runs * x.size / t_total / 1e9, "unit": "Gelem/s", "cores": 1, "kind": "oracle",
            "sample": "%d full passes over the n=2^%d input (%.1f s), sequential C oracle on one host core"
                      % (runs, int(x.size).bit_length() - 1, t_total), **host_cores()}


def time_calls(fn, steps: int, warmup: int, stream, stats: dict | None = None) -> float:
    """Mean ms per call over `steps` back-to-back calls (one event pair
    around all of them); with `stats`, also the median and minimum of the
    per-call event pairs."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    mean = e0.elapsed_time(e1) / steps
    if stats is not None:
        # a second pass with an event between calls; an event breaks the
        # overlap of one call's launch with the previous call, so for short
        # calls these figures run above the mean of the back-to-back pass
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        for k in range(steps):
            marks[k].record(stream)
            fn()
        marks[steps].record(stream)
        torch.cuda.synchronize()
        per = sorted(marks[k].elapsed_time(marks[k + 1]) for k in range(steps))
        stats["ms_median"], stats["ms_min"] = per[len(per) // 2], per[0]
    return mean


def measure_secondary(dwp, lib, dev, stream, peaks, x, y, scratch, need) -> dict:
    import ctypes
    n = x.numel()
    out = {}
    sb = ctypes.c_size_t(need)
    st_ptr = ctypes.c_void_p(int(stream.cuda_stream))
    xf = None
    for name, entry, op in (("u32_add_inclusive", lib.dwp_scan_inclusive, dwp.DWP_U32_ADD),
                            ("u32_max_exclusive", lib.dwp_scan_exclusive, dwp.DWP_U32_MAX),
                            ("u32_max_inclusive", lib.dwp_scan_inclusive, dwp.DWP_U32_MAX),
                            ("f32_add_inclusive", lib.dwp_scan_inclusive, dwp.DWP_F32_ADD)):
        src = x
        if op == dwp.DWP_F32_ADD:
            import torch
            xf = torch.from_numpy(synth.f32_values(n)).to(dev)
            src = xf
        args = (op, ctypes.c_void_p(src.data_ptr()), ctypes.c_void_p(y.data_ptr()), n,
                ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb), st_ptr)
        stats = {}
        ms = time_calls(lambda: entry(*args), 200, 5, stream, stats)
        gbs = 8 * n / (ms * 1e-3) / 1e9
        out[name] = {"n": n, "ms": ms, **stats, "Gelem_s": n / (ms * 1e-3) / 1e9, "GB_s": gbs,
                     "frac": gbs / peaks["hbm_gbs"]}
    del xf
    out["u32_add_exclusive_2p20"] = measure_small(dwp, lib, dev, stream)
    out["single_pass_vs_two_level"] = measure_two_level(dwp, lib, dev, stream)
    out["fallback_one_silent_tile"] = measure_fallback(dwp, lib, stream, x, y, scratch, need)
    out["lookback_window_ablation"] = measure_window_ablation(dwp, lib, stream, x, y, scratch, need)
    out["segscan_u32_exclusive"] = measure_segscan(dwp, lib, dev, stream, peaks)
    out["compact_16B_records"] = measure_compact(dwp, lib, dev, stream, peaks)
    out["compact_staged_vs_fused"] = measure_compact_staged(dwp, lib, dev, stream, peaks)
    out["linear_recurrence_f32"] = measure_recurrence(dwp, lib, dev, stream, peaks)
    out["segreduce_u32"] = measure_segreduce(dwp, lib, dev, stream, peaks)
    for name, (summary, sources) in SECONDARY_PROFILES.items():
        if name in out:
            out[name]["traffic"] = profiled_traffic(os.path.join(ROOT, "profiles", summary), sources)
    return out


def measure_small(dwp, lib, dev, stream, log2n=20, steps=2000, warmup=20) -> dict:
    """The small case: u32 exclusive add over 2^20 values in [0, 16), L2-resident
    and launch-bound, so the figure is microseconds per call."""
    import ctypes
    import torch
    n = 1 << log2n
    x = torch.from_numpy(synth.u32_small_values(n).view(np.int32)).to(dev)
    y = torch.empty_like(x)
    sb = ctypes.c_size_t(0)
    lib.dwp_scan_exclusive(0, None, None, n, None, ctypes.byref(sb), None)
    scratch = torch.empty(sb.value, dtype=torch.uint8, device=dev)
    args = (dwp.DWP_U32_ADD, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()), n,
            ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb),
            ctypes.c_void_p(int(stream.cuda_stream)))
    stats = {}
    ms = time_calls(lambda: lib.dwp_scan_exclusive(*args), steps, warmup, stream, stats)
    return {"n": n, "us": ms * 1e3, "us_median": stats["ms_median"] * 1e3, "us_min": stats["ms_min"] * 1e3,
            "Gelem_s": n / (ms * 1e-3) / 1e9,
            "workload": "u32 exclusive sum scan, n=2^%d values in [0,16) (SplitMix64 seed 0xD3B00001), "
                        "L2-resident: launch-bound, not an HBM figure" % log2n}


def measure_two_level(dwp, lib, dev, stream, log2ns=(12, 14, 16, 18, 19, 20, 21, 22, 23, 24, 26), steps=500) -> dict:
    """u32 exclusive add by the single-pass look-back scan and by the
    two-level three-launch form, microseconds per call, back to back."""
    import ctypes
    import torch
    st_ptr = ctypes.c_void_p(int(stream.cuda_stream))
    res = {"unit": "us per call"}
    for lg in log2ns:
        n = 1 << lg
        x = torch.from_numpy(synth.u32_small_values(n).view(np.int32)).to(dev)
        y = torch.empty_like(x)
        row = {}
        for name, fn in (("single_pass", lib.dwp_scan_exclusive), ("two_level", lib.dwp_scan_two_level)):
            sb = ctypes.c_size_t(0)
            if name == "single_pass":
                fn(0, None, None, n, None, ctypes.byref(sb), None)
            else:
                fn(0, 0, None, None, n, None, ctypes.byref(sb), None)
            scratch = torch.empty(sb.value, dtype=torch.uint8, device=dev)
            common = (ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()), n,
                      ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb), st_ptr)
            args = (0,) + common if name == "single_pass" else (0, 0) + common
            row[name] = time_calls(lambda: fn(*args), max(20, steps >> max(0, lg - 20)), 5, stream) * 1e3
        res["2^%d" % lg] = row
    return res


def measure_fallback(dwp, lib, stream, x, y, scratch, need, silent=5, polls=64, steps=20) -> dict:
    """Cost of one Decoupled Fallback: the headline call with tile `silent`
    never publishing, its successors rescuing it after `polls` look-back polls."""
    import ctypes
    n = x.numel()
    sb = ctypes.c_size_t(need)
    st_ptr = ctypes.c_void_p(int(stream.cuda_stream))
    args = (dwp.DWP_U32_ADD, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()), n,
            ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb), st_ptr)
    healthy = time_calls(lambda: lib.dwp_scan_exclusive(*args), steps, 3, stream)
    try:
        lib.dwp_debug_set_fault(silent, 0, polls)
        ms = time_calls(lambda: lib.dwp_scan_exclusive(*args), steps, 3, stream)
        status = lib.dwp_read_status(ctypes.c_void_p(scratch.data_ptr()), st_ptr)
        fb = ctypes.c_uint32(0)
        lib.dwp_read_fallbacks(ctypes.c_void_p(scratch.data_ptr()), st_ptr, ctypes.byref(fb))
    finally:
        lib.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
    return {"n": n, "silent_tile": silent, "fallback_polls": polls, "ms": ms,
            "healthy_ms": healthy, "added_us": (ms - healthy) * 1e3, "fallbacks_last_call": fb.value,
            "status": dwp.dwp_status_string(status)}


def measure_window_ablation(dwp, lib, stream, x, y, scratch, need, steps=50,
                            windows=(0, 32, 128, 1024)) -> dict:
    """Bounded look-back window against the unbounded one on the headline call:
    healthy, and with tile 5 silent until a successor rescues it after 64
    polls (every later tile then folds a long chain of aggregates: the case a
    window bounds)."""
    import ctypes
    n = x.numel()
    sb = ctypes.c_size_t(need)
    st_ptr = ctypes.c_void_p(int(stream.cuda_stream))
    args = (dwp.DWP_U32_ADD, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()), n,
            ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb), st_ptr)
    res = {"n": n, "note": "window 0 = unbounded (the default); ms per call"}
    try:
        for w in windows:
            lib.dwp_set_lookback_window(w)
            healthy = time_calls(lambda: lib.dwp_scan_exclusive(*args), steps, 3, stream)
            lib.dwp_debug_set_fault(5, 0, 64)
            stalled = time_calls(lambda: lib.dwp_scan_exclusive(*args), steps, 3, stream)
            lib.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
            status = lib.dwp_read_status(ctypes.c_void_p(scratch.data_ptr()), st_ptr)
            res["window_%d" % w] = {"healthy_ms": healthy, "one_silent_tile_ms": stalled,
                                    "status": dwp.dwp_status_string(status)}
    finally:
        lib.dwp_set_lookback_window(0)
        lib.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
    return res


def run_only(args) -> None:
    """One workload alone, `args.steps` timed calls, for profiler captures."""
    import torch
    import device_wide_prefix_gb300 as dwp
    dev = torch.device("cuda", 0)
    lib = dwp.load()
    stream = torch.cuda.current_stream(dev)
    fn = {"scan": measure_scan_only, "segscan": measure_segscan, "compact": measure_compact,
          "recurrence": measure_recurrence, "segreduce": measure_segreduce,
          "compact_staged": measure_compact_staged}[args.only]
    r = fn(dwp, lib, dev, stream, measured_peaks(), log2n=args.log2n, steps=args.steps,
           warmup=args.warmup)
    print(json.dumps({"only": args.only, **r}), flush=True)


def measure_scan_only(dwp, lib, dev, stream, peaks, log2n=28, steps=100, warmup=5) -> dict:
    """u32 exclusive add scan of 2^log2n full-range values alone (the kernel
    the size picks: small-input up to 2^22, pipelined above)."""
    import ctypes
    import torch
    n = 1 << log2n
    x = torch.from_numpy(synth.u32_full_values(n).view(np.int32)).to(dev)
    y = torch.empty_like(x)
    need = dwp.scan_scratch_bytes(n)
    scratch = dwp.alloc_scratch(need, dev)
    sb = ctypes.c_size_t(need)
    args = (dwp.DWP_U32_ADD, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()), n,
            ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb), ctypes.c_void_p(int(stream.cuda_stream)))
    stats = {}
    ms = time_calls(lambda: lib.dwp_scan_exclusive(*args), steps, warmup, stream, stats)
    if dwp.read_status(scratch) != dwp.DWP_SUCCESS:
        raise RuntimeError("scan reported a device-side error")
    gbs = 8 * n / (ms * 1e-3) / 1e9
    return {"n": n, "ms": ms, **stats, "Gelem_s": n / (ms * 1e-3) / 1e9, "GB_s": gbs,
            "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": 8 * n}


def measure_compact(dwp, lib, dev, stream, peaks, log2n=26, steps=100, warmup=5) -> dict:
    """Stable compaction of 2^26 16-byte records {u32 id, 3 x f32 N(0,1)} by
    Bernoulli(0.3) byte flags."""
    import ctypes
    import torch
    n = 1 << log2n
    rec = torch.from_numpy(synth.records(n).view(np.int32)).to(dev)
    flags = torch.from_numpy(synth.keep_flags(n)).to(dev)
    out = torch.empty_like(rec)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    need = dwp.compact_scratch_bytes(n)
    scratch = dwp.alloc_scratch(need, dev)
    sb = ctypes.c_size_t(need)
    args = (ctypes.c_void_p(rec.data_ptr()), ctypes.c_void_p(flags.data_ptr()), n,
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(cnt.data_ptr()),
            ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb),
            ctypes.c_void_p(int(stream.cuda_stream)))
    stats = {}
    ms = time_calls(lambda: lib.dwp_compact_by_flags(*args), steps, warmup, stream, stats)
    if dwp.read_status(scratch) != dwp.DWP_SUCCESS:
        raise RuntimeError("compaction reported a device-side error")
    k = int(cnt.item())
    alg = 17 * n + 16 * k + 4
    gbs = alg / (ms * 1e-3) / 1e9
    return {"n": n, "kept": k, "ms": ms, **stats, "Gelem_s": n / (ms * 1e-3) / 1e9, "GB_s": gbs,
            "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": alg,
            "workload": "stable compaction of 2^%d 16-byte records, keep flag Bernoulli(0.3) "
                        "(SplitMix64 seed 0xD3B00004)" % log2n}


def kept_sector_bytes(flags: np.ndarray, unit: int = 32) -> int:
    """Bytes of the `unit`-byte pieces of the record array that hold at least
    one kept 16-byte record: what a compaction that reads only the kept
    records must read when memory moves `unit` bytes at a time (32 for an L2
    sector; about 128 for what DRAM moved in a probe of this workload)."""
    per = unit // 16
    f = flags != 0
    if f.size % per:
        f = np.concatenate([f, np.zeros(per - f.size % per, dtype=bool)])
    return int(f.reshape(-1, per).any(axis=1).sum()) * unit


def measure_compact_staged(dwp, lib, dev, stream, peaks, log2n=26, steps=50, warmup=5) -> dict:
    """Staged compaction (u32 flags and their exclusive scan written to
    memory, then a scatter: three launches and the scan's clear) against the
    fused single-pass kernel, on the compaction workload, with the bytes each
    moves.  Algorithmic bytes:
      fused         n flags + 16n records read, 16k written, 4 count
      staged        n flags read + 4n u32 flags written; the scan reads 4n and
                    writes 4n; the scatter reads 4n flags, 4n offsets and the
                    sectors holding kept records (S), writes 16k and the count
      lower bound   n flags + S + 16k + 4: a compaction that reads only the
                    sectors of kept records ("selective read")."""
    import ctypes
    import torch
    n = 1 << log2n
    rec = torch.from_numpy(synth.records(n).view(np.int32)).to(dev)
    flags_np = synth.keep_flags(n)
    flags = torch.from_numpy(flags_np).to(dev)
    out = torch.empty_like(rec)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    res = {"n": n}
    sector = kept_sector_bytes(flags_np)
    for name, fn, need in (("fused", lib.dwp_compact_by_flags, dwp.compact_scratch_bytes(n)),
                           ("staged", lib.dwp_compact_by_flags_staged, dwp.compact_staged_scratch_bytes(n))):
        scratch = dwp.alloc_scratch(need, dev)
        sb = ctypes.c_size_t(need)
        args = (ctypes.c_void_p(rec.data_ptr()), ctypes.c_void_p(flags.data_ptr()), n,
                ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(cnt.data_ptr()),
                ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb),
                ctypes.c_void_p(int(stream.cuda_stream)))
        stats = {}
        ms = time_calls(lambda: fn(*args), steps, warmup, stream, stats)
        if dwp.read_status(scratch) != dwp.DWP_SUCCESS:
            raise RuntimeError("%s compaction reported a device-side error" % name)
        k = int(cnt.item())
        alg = 17 * n + 16 * k + 4 if name == "fused" else 21 * n + sector + 16 * k + 4
        res[name] = {"ms": ms, **stats, "algorithmic_bytes": alg,
                     "GB_s": alg / (ms * 1e-3) / 1e9, "frac": alg / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}
        del scratch
    k = int(cnt.item())
    lower = n + sector + 16 * k + 4
    res["kept"] = k
    res["kept_sector_bytes"] = sector
    res["selective_read_lower_bound"] = {
        "bytes": lower, "ms_at_peak": lower / (peaks["hbm_gbs"] * 1e9) * 1e3,
        "fused_frac_of_it": lower / (res["fused"]["ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"]}
    # the same bound in 128-byte pieces: at p = 0.3 reading only the kept
    # records measured no faster than reading them all
    line = kept_sector_bytes(flags_np, 128)
    lower128 = n + line + 16 * k + 4
    res["selective_read_lower_bound_128B"] = {
        "bytes": lower128, "ms_at_peak": lower128 / (peaks["hbm_gbs"] * 1e9) * 1e3,
        "fused_frac_of_it": lower128 / (res["fused"]["ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"]}
    res["staged_over_fused"] = res["staged"]["ms"] / res["fused"]["ms"]
    res["extra_bytes_staged"] = res["staged"]["algorithmic_bytes"] - res["fused"]["algorithmic_bytes"]
    return res


def measure_segscan(dwp, lib, dev, stream, peaks, log2n=27, steps=200, warmup=5) -> dict:
    """Segmented exclusive u32 scan, n = 2^27 values in [0, 255], Zipf(1.2)
    segment lengths capped at 2^22 with 5% empty segments (CSR offsets)."""
    import ctypes
    import torch
    n = 1 << log2n
    off_np = synth.segment_offsets(n)
    nseg = off_np.size - 1
    v = torch.from_numpy(synth.u32_byte_values(n).view(np.int32)).to(dev)
    off = torch.from_numpy(off_np.view(np.int32)).to(dev)
    y = torch.empty_like(v)
    need = dwp.segmented_scan_scratch_bytes(n)
    scratch = dwp.alloc_scratch(need, dev)
    sb = ctypes.c_size_t(need)
    args = (ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(off.data_ptr()), nseg,
            ctypes.c_void_p(y.data_ptr()), n, dwp.DWP_EXCLUSIVE, ctypes.c_void_p(scratch.data_ptr()),
            ctypes.byref(sb), ctypes.c_void_p(int(stream.cuda_stream)))
    stats = {}
    ms = time_calls(lambda: lib.dwp_segmented_scan_u32(*args), steps, warmup, stream, stats)
    if dwp.read_status(scratch) != dwp.DWP_SUCCESS:
        raise RuntimeError("segmented scan reported a device-side error")
    alg = 8 * n + 4 * (nseg + 1)
    gbs = alg / (ms * 1e-3) / 1e9
    return {"n": n, "segments": nseg, "ms": ms, **stats, "Gelem_s": n / (ms * 1e-3) / 1e9, "GB_s": gbs,
            "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": alg,
            "workload": ("segmented exclusive u32 sum scan, n=2^%d values in [0,255], Zipf(1.2) " % log2n) +
                        "lengths capped at 2^22, 5% empty, CSR offsets (SplitMix64 seed 0xD3B00005)"}


def measure_segreduce(dwp, lib, dev, stream, peaks, log2n=27, steps=200, warmup=5) -> dict:
    """Segmented u32 reduction over the segmented scan's skewed offsets: n = 2^27
    values in [0, 255], Zipf(1.2) lengths capped at 2^22, 5% empty."""
    import ctypes
    import torch
    n = 1 << log2n
    off_np = synth.segment_offsets(n)
    nseg = off_np.size - 1
    v = torch.from_numpy(synth.u32_byte_values(n).view(np.int32)).to(dev)
    off = torch.from_numpy(off_np.view(np.int32)).to(dev)
    out = torch.empty(nseg, dtype=torch.int32, device=dev)
    need = dwp.segmented_reduce_scratch_bytes(n)
    scratch = dwp.alloc_scratch(need, dev)
    sb = ctypes.c_size_t(need)
    args = (ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(off.data_ptr()), nseg,
            ctypes.c_void_p(out.data_ptr()), n, ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb),
            ctypes.c_void_p(int(stream.cuda_stream)))
    stats = {}
    ms = time_calls(lambda: lib.dwp_segmented_reduce_u32(*args), steps, warmup, stream, stats)
    if dwp.read_status(scratch) != dwp.DWP_SUCCESS:
        raise RuntimeError("segmented reduction reported a device-side error")
    alg = 4 * n + 4 * (nseg + 1) + 4 * nseg
    gbs = alg / (ms * 1e-3) / 1e9
    return {"n": n, "segments": nseg, "ms": ms, **stats, "Gelem_s": n / (ms * 1e-3) / 1e9, "GB_s": gbs,
            "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": alg,
            "workload": ("segmented u32 sum reduction, n=2^%d values in [0,255], Zipf(1.2) " % log2n) +
                        "lengths capped at 2^22, 5% empty, CSR offsets (SplitMix64 seed 0xD3B00005)"}


def measure_recurrence(dwp, lib, dev, stream, peaks, log2n=28, steps=200, warmup=5) -> dict:
    """f32 linear recurrence h[t] = a[t] h[t-1] + b[t], inclusive, n = 2^28,
    a uniform in [0.5, 1), b uniform in [-1, 1)."""
    import ctypes
    import torch
    n = 1 << log2n
    a = torch.from_numpy(synth.decay_values(n)).to(dev)
    b = torch.from_numpy(synth.f32_values(n, seed=synth.SEED_RECURRENCE_B)).to(dev)
    h = torch.empty_like(b)
    need = dwp.linear_recurrence_scratch_bytes(n)
    scratch = dwp.alloc_scratch(need, dev)
    sb = ctypes.c_size_t(need)
    args = (ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()), ctypes.c_void_p(h.data_ptr()),
            n, dwp.DWP_INCLUSIVE, ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb),
            ctypes.c_void_p(int(stream.cuda_stream)))
    stats = {}
    ms = time_calls(lambda: lib.dwp_linear_recurrence_f32(*args), steps, warmup, stream, stats)
    if dwp.read_status(scratch) != dwp.DWP_SUCCESS:
        raise RuntimeError("linear recurrence reported a device-side error")
    alg = 12 * n
    gbs = alg / (ms * 1e-3) / 1e9
    return {"n": n, "ms": ms, **stats, "Gelem_s": n / (ms * 1e-3) / 1e9, "GB_s": gbs,
            "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": alg,
            "workload": "f32 linear recurrence h[t] = a[t] h[t-1] + b[t], inclusive, n=2^%d, "
                        "a uniform in [0.5,1), b uniform in [-1,1) (SplitMix64 seeds 0xD3B00006/7)"
                        % log2n}


if __name__ == "__main__":
    main()
