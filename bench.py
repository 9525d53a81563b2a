#!/usr/bin/env python3
"""Benchmark: device-wide scan and stream compaction on one GB300 (or N replicas).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--headline-only]

One step is one fp32 inclusive scan of n = 1e8 values ~ N(0,1) through the C ABI
(gb_scan_inclusive: status reset + the single-pass kernel), with the input already
in HBM.  The step is timed with CUDA events on the launching stream; the kernel alone
is timed through the library's profile-event hook.  Rank 0 prints ONE JSON line.

Besides the headline, the line carries the other workloads (int32/fp64/max scans,
compaction, packing, batched and large-element scans, the reduce-then-scan variant)
under "workloads", each as kernel time, GB/s and fraction of the HBM roofline, L2
flushed between repetitions.  --impl reference times the CPU oracle instead.

Multi-GPU: the scan does not shard here; N > 1 runs N independent replicas (one per
rank, no collective on the data path) and reports their aggregate throughput.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fp32 1e8 inclusive scan GB/s (% of HBM peak); compaction Gelem/s"
HEADLINE = "fp32_1e8"
N_HEAD = 100_000_000
BYTES_HEAD = 2 * N_HEAD * 4            # read once, write once (single pass)
# AcceleratedKernels.jl PR #208, RTX 5080, cumsum F32 1e8: 1388.2 us (context only).
PAGE_FP32_1E8_US = 1388.2
PAGE_FP32_1E8_GBS = BYTES_HEAD / (PAGE_FP32_1E8_US * 1e-6) / 1e9
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------- helpers ------

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy read+write)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s)"


# The source files each profiled kernel is compiled from: a capture stays valid
# while none of them changes.
KERNEL_SOURCES = {
    "scan_stash_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_stash.cuh"),
    "scan_rows_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_rows.cuh"),
    "scan_rows_chunk_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_rows.cuh"),
    "scan_seg_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_seg.cuh"),
    "scan_seg_chunk_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_seg.cuh"),
    "compact_seg_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_seg.cuh", "compact.cuh"),
    "compact_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_rows.cuh", "compact.cuh"),
    "partition_seg_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_seg.cuh", "compact.cuh", "partition.cuh"),
    "scan_lanes_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_lanes.cuh"),
    "pack_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_rows.cuh", "pack.cu"),
    "pack_seg_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_seg.cuh", "pack.cu"),
    "rts_scan_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_rows.cuh", "rts.cuh"),
    "stf_fan_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_rows.cuh", "rts.cuh"),
    "scan_segmented_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_seg.cuh", "segmented.cuh"),
    "lanes_rts_reduce_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_lanes.cuh", "scan_lanes_rts.cuh"),
    "lanes_rts_spine_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_lanes.cuh", "scan_lanes_rts.cuh"),
    "lanes_rts_scan_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_lanes.cuh", "scan_lanes_rts.cuh"),
    "scan_lanes_seg_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_seg.cuh", "scan_lanes_seg.cuh"),
    "scan_affine_seg_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_seg.cuh", "scan_affine.cuh"),
    "scan_affine_tile_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_seg.cuh", "scan_affine.cuh"),
    "scan_strips_kernel": ("common.cuh", "tile.cuh", "launch.h", "scan_strips.cuh"),
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the sources of `kernel` (its name up to the first '<')."""
    d = os.path.join(ROOT, "stream_compaction_decoupled_gb300", "csrc")
    files = KERNEL_SOURCES.get(kernel.split("<")[0], tuple(sorted(os.listdir(d))))
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel: str):
    """DRAM bytes per launch recorded by an ncu capture of this exact kernel source.

    The summaries under profiles/ carry 'kernel:', 'source_hash:' and
    'traffic_bytes_per_launch:' lines; a figure taken on older sources of the
    kernel is ignored.  `python bench.py --source-hash KERNEL` prints the hash.
    """
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return None
    src = kernel_source_hash(kernel)
    for f in sorted(os.listdir(d)):
        if not f.endswith(".md"):
            continue
        txt = open(os.path.join(d, f)).read()
        k = re.search(r"^kernel:\s*(\S+)", txt, re.M)
        h = re.search(r"^source_hash:\s*(\S+)", txt, re.M)
        t = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt, re.M)
        if k and h and t and k.group(1) == kernel and h.group(1) == src:
            return float(t.group(1))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms in the background."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "gbscan_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 10:
                        continue
                    try:
                        ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                        rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                    except ValueError:
                        continue
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "no samples (nvidia-smi unavailable)"}
        inside = [r for r in rows if t0 <= r[0] <= t1]
        window = "timed region"
        if not inside:  # the timed region was shorter than the sampling period
            inside = [r for r in rows if r[0] >= t0 - 2.0]
            window = "benchmark load around the timed region (timed region < sampling period)"
        if not inside:
            inside, window = rows, "whole run"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[3][i].lower() == "active"})
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


def dist_init():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist.get_rank(), ws, int(os.environ.get("LOCAL_RANK", "0"))
    return 0, 1, 0


def max_over_ranks(value: float, device=None) -> float:
    """Largest value over all ranks (1 rank: the value itself)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index] if device is not None else None)
        else:
            dist.barrier()


# ----------------------------------------------------------- GPU workloads -----

class L2Flush:
    """Writes a buffer of twice the L2 size between repetitions."""

    def __init__(self, device):
        import torch
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        self.buf = torch.empty(max(2 * l2, 64 << 20) // 4, dtype=torch.float32, device=device)

    def __call__(self):
        self.buf.fill_(1.0)


def time_call(fn, reps: int, flush, stream, kernel_events: bool):
    """Best and median kernel time (ms) of fn() over reps, L2 flushed before each."""
    import torch
    import stream_compaction_decoupled_gb300 as gb
    ks, steps = [], []
    for _ in range(reps):
        if flush:
            flush()
        # Keep the GPU busy while the host enqueues the call, so that the events time
        # device work, not the host's launch latency.
        torch.cuda._sleep(200_000)
        kb, ka = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sb, sa = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if kernel_events:
            gb.set_profile_events(kb, ka)
        sb.record(stream)
        fn()
        sa.record(stream)
        gb.set_profile_events(None, None)
        torch.cuda.synchronize()
        steps.append(sb.elapsed_time(sa))
        if kernel_events:
            ks.append(kb.elapsed_time(ka))
    k = ks if kernel_events else steps
    return {"kernel_ms_best": min(k), "kernel_ms_median": float(np.median(k)),
            "step_ms_median": float(np.median(steps))}


def workload_call(w, device):
    """The library call of workload `w` on device-resident synthetic inputs:
    (fn, algorithmic bytes, units, unit)."""
    import torch
    import stream_compaction_decoupled_gb300 as gb
    x = torch.from_numpy(w.make()).to(device)
    es = x.element_size()
    if w.kind == "scan":
        y = torch.empty_like(x)
        n_el = x.numel()
        if w.inclusive:
            fn = lambda: gb.scan_inclusive(x, w.op, lanes=w.lanes, out=y)  # noqa: E731
        else:
            fn = lambda: gb.scan_exclusive(x, w.op, lanes=w.lanes, out=y)  # noqa: E731
        return fn, 2 * n_el * es, n_el // w.lanes, "Gelem/s"
    if w.kind == "batched":
        rows, cols = w.shape
        xv = x.reshape(rows, cols, w.lanes)
        y = torch.empty_like(xv)
        fn = lambda: gb.scan_batched(xv, axis=w.axis, op=w.op, lanes=w.lanes, out=y)  # noqa: E731
        return fn, 2 * x.numel() * es, rows * cols, "Gelem/s"
    if w.kind == "compact":
        idx = torch.empty(x.numel(), dtype=torch.int32, device=device)
        cnt = torch.empty(1, dtype=torch.int32, device=device)
        p = w.extra["p"]
        fn = lambda: gb.compact(x, "lt", p, out_idx=idx, out_count=cnt)  # noqa: E731
        fn()
        torch.cuda.synchronize()
        m = int(cnt.item())
        return fn, 4 * x.numel() + 4 * m + 4, x.numel(), "Gelem/s"
    if w.kind == "segmented":  # values, one head flag byte per element, values out
        from stream_compaction_decoupled_gb300.workloads import head_flags
        fl = torch.from_numpy(head_flags(x.numel(), w.extra["p_head"], w.extra["flag_seed"])).to(device)
        y = torch.empty_like(x)
        fn = lambda: gb.scan_segmented(x, fl, w.op, out=y)  # noqa: E731
        return fn, 2 * x.numel() * es + x.numel(), x.numel(), "Gelem/s"
    if w.kind == "partition":  # values and their input indices
        out = torch.empty_like(x)
        idx = torch.empty(x.numel(), dtype=torch.int32, device=device)
        cnt = torch.empty(1, dtype=torch.int32, device=device)
        p = w.extra["p"]
        fn = lambda: gb.partition(x, "lt", p, out=out, out_idx=idx, out_count=cnt)  # noqa: E731
        return fn, 2 * x.numel() * es + 4 * x.numel() + 4, x.numel(), "Gelem/s"
    total = int(x.sum().item())  # pack
    recs = torch.empty(total, dtype=torch.int32, device=device)
    tot = torch.empty(1, dtype=torch.int32, device=device)
    fn = lambda: gb.pack_by_counts(x, total, offsets=True, out_records=recs, out_total=tot)  # noqa: E731
    return fn, 4 * x.numel() * 2 + 4 * total, x.numel(), "Gelem/s"


def profile_workload(name, reps):
    """--profile NAME: only that workload's call, 3 untimed calls then `reps` calls
    with L2 flushed before each, for ncu captures (skip 3 launches, capture 1-3)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from stream_compaction_decoupled_gb300 import workloads as W
    import stream_compaction_decoupled_gb300 as gb
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    comparators = {"fp32_1e8_reduce_then_scan": gb.scan_reduce_then_scan, "fp32_1e8_scan_then_fan": gb.scan_then_fan}
    if name in comparators:  # the comparison variants on the headline input
        xh = torch.from_numpy(W.BY_NAME[HEADLINE].make()).to(device)
        yh = torch.empty_like(xh)
        call = comparators[name]
        fn, nbytes = (lambda: call(xh, out=yh)), BYTES_HEAD
    else:
        fn, nbytes, units, unit = workload_call(W.BY_NAME[name], device)
    for _ in range(3):
        fn()
    t = time_call(fn, reps, L2Flush(device), torch.cuda.current_stream(device), kernel_events=True)
    ms = t["kernel_ms_best"]
    print(json.dumps({"profile_workload": name, "reps": reps, "call_us_best": round(ms * 1e3, 2),
                      "GB_s": round(nbytes / (ms * 1e-3) / 1e9, 1)}), flush=True)


def secondary_workloads(device, hbm_peak, reps=10, only=None):
    """Every other workload: kernel time, GB/s, fraction of the HBM roofline."""
    import torch
    import stream_compaction_decoupled_gb300 as gb
    from stream_compaction_decoupled_gb300 import workloads as W
    stream = torch.cuda.current_stream(device)
    flush = L2Flush(device)
    out = {}
    for w in W.WORKLOADS:
        if w.name == HEADLINE or (only and w.name not in only):
            continue
        fn, nbytes, units, unit = workload_call(w, device)
        for _ in range(3):
            fn()
        t = time_call(fn, reps, flush, stream, kernel_events=True)
        ms = t["kernel_ms_best"]
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[w.name] = {"kernel_us_best": round(ms * 1e3, 2), "kernel_us_median": round(t["kernel_ms_median"] * 1e3, 2),
                       "step_us_median": round(t["step_ms_median"] * 1e3, 2),
                       "GB_s": round(gbs, 1), "frac_hbm": round(gbs / hbm_peak, 4),
                       "throughput": round(units / (ms * 1e-3) / 1e9, 3), "throughput_unit": unit,
                       "algorithmic_bytes": int(nbytes), "l2": "flushed between repetitions"}
        del fn
    # The comparison variants on the headline workload: reduce-then-scan (3n element
    # transfers) and scan-then-fan (4n), each three launches.
    comparators = [("fp32_1e8_reduce_then_scan", gb.scan_reduce_then_scan, "3n"),
                   ("fp32_1e8_scan_then_fan", gb.scan_then_fan, "4n")]
    if only and not any(c[0] in only for c in comparators):
        return out
    xh = torch.from_numpy(W.BY_NAME[HEADLINE].make()).to(device)
    yh = torch.empty_like(xh)
    for name, call, traffic in comparators:
        if only and name not in only:
            continue
        fn = lambda: call(xh, out=yh)  # noqa: E731
        for _ in range(3):
            fn()
        t = time_call(fn, reps, None, stream, kernel_events=False)
        ms = t["kernel_ms_best"]
        out[name] = {
            "step_us_best": round(ms * 1e3, 2), "step_us_median": round(t["kernel_ms_median"] * 1e3, 2),
            "GB_s": round(BYTES_HEAD / (ms * 1e-3) / 1e9, 1),
            "frac_hbm": round(BYTES_HEAD / (ms * 1e-3) / 1e9 / hbm_peak, 4), "algorithmic_bytes": BYTES_HEAD,
            "note": "three launches; 2n-byte model, so %s traffic shows as a lower GB/s" % traffic}
    return out


# ------------------------------------------------------------ FP64 add rate ---

# A throughput probe of the FP64 adder (the bound of the fp64 scans on GB300), written
# out, built with nvcc and run by --fp64-add-rate.  Every thread runs 8 independent
# chains of dependent adds (one add per chain per iteration), so the adder, not the
# latency of one chain, is the limit; 8 CTAs of 256 threads per SM.  The result is
# written to memory so the adds are not removed.
_ADD_RATE_SRC = r"""
#include <cstdio>
template <class T> __global__ void chains(T* out, T step, int iters) {
  T c[8];
  for (int k = 0; k < 8; ++k) c[k] = (T)(threadIdx.x + k);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < 8; ++k) c[k] += step;
  }
  T s = 0;
  for (int k = 0; k < 8; ++k) s += c[k];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}
template <class T> void rate(const char* name) {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const int blocks = sms * 8, threads = 256, iters = 4096;
  T* out = nullptr;
  cudaMalloc(&out, sizeof(T) * blocks * threads);
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  float best = 1e30f;
  for (int r = 0; r < 7; ++r) {
    cudaEventRecord(a);
    chains<T><<<blocks, threads>>>(out, (T)1e-9, iters);
    cudaEventRecord(b);
    cudaEventSynchronize(b);
    float ms = 0;
    cudaEventElapsedTime(&ms, a, b);
    if (ms < best) best = ms;
  }
  const double adds = (double)blocks * threads * iters * 8;
  printf("%s %d %.6f %.1f %s\n", name, sms, best, adds, cudaGetErrorString(cudaGetLastError()));
  cudaFree(out);
}
int main() {
  rate<double>("fp64");
  rate<float>("fp32");
  return 0;
}
"""


def fp64_add_rate() -> dict:
    """Build and run the add-rate probe: adds per second and per clock per SM for
    fp64 and fp32 (best of 7 launches, CUDA events)."""
    import tempfile
    nvcc = os.environ.get("NVCC") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as tmp:
        src, exe = os.path.join(tmp, "add_rate.cu"), os.path.join(tmp, "add_rate")
        with open(src, "w") as f:
            f.write(_ADD_RATE_SRC)
        subprocess.run([nvcc, "-O3", "-gencode", "arch=compute_103a,code=sm_103a", src, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    peaks = {}
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    mhz = peaks.get("sm_max_mhz", 2070.0)
    res = {"sm_clock_mhz_assumed": mhz}
    for line in out.splitlines():
        name, sms, ms, adds, err = line.split(maxsplit=4)
        rate = float(adds) / (float(ms) * 1e-3)
        res[name] = {"adds_per_s": rate, "per_clock_per_sm": rate / (int(sms) * mhz * 1e6), "ms": float(ms),
                     "status": err}
    return res


# ---------------------------------------------------------------- CPU oracle ---

def host_cpu() -> dict:
    """The host the oracle runs on: its logical CPU count and CPU model (lscpu's
    "Model name", else /proc/cpuinfo's, else the machine type)."""
    import platform
    import subprocess
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"host_cpus": os.cpu_count(), "cpu_model": model or platform.machine()}


def cpu_oracle_leg(x_full: np.ndarray, steps: int, budget_s: float):
    """The oracle timed on the host: `steps` inclusive scans of a leading slice of the
    headline input, its length chosen so that all steps take about budget_s."""
    import oracle
    cal = x_full[:1_000_000]
    t0 = time.perf_counter()
    oracle.scan(cal)
    per_elem = max((time.perf_counter() - t0) / cal.size, 1e-10)
    n = int(min(x_full.size, max(1_000_000, budget_s / max(steps, 1) / per_elem)))
    x = x_full[:n]
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.scan(x)
        times.append(time.perf_counter() - t0)
    return n, times


def reference_arm(args, rank):
    """--impl reference: the CPU oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    from stream_compaction_decoupled_gb300 import workloads as W
    n, times = cpu_oracle_leg(W.BY_NAME[HEADLINE].make(), args.warmup + args.steps, budget_s=60.0)
    times = times[args.warmup:] or times
    t = float(np.mean(times))
    gbs = 2 * n * 4 / t / 1e9
    sample = ("fp32 inclusive scan of the first %d of the 1e8 N(0,1) seed-2 values, one thread, "
              "%d timed steps after %d warm-up" % (n, args.steps, args.warmup))
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 in, f64 accumulate",
            "data": "synthetic", "config": {"workload": "fp32_1e8 inclusive scan (sample, see cpu_baseline)"},
            "cpu_baseline": dict({"value": round(gbs, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                  "sample": sample}, **host_cpu()),
            "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm ------

def our_arm(args, rank, world, local_rank):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import stream_compaction_decoupled_gb300 as gb
    from stream_compaction_decoupled_gb300 import workloads as W

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    hbm_peak, peak_src = peaks()
    stream = torch.cuda.current_stream(device)

    n = args.n
    x_host = W.BY_NAME[HEADLINE].make() if n == N_HEAD else W.normal(n, np.float32, 2)
    nbytes = 2 * n * 4
    x = torch.from_numpy(x_host).to(device)
    y = torch.empty_like(x)
    temp = torch.empty(gb.temp_storage_bytes(gb.KIND_SCAN, gb.F32, 1, n), dtype=torch.uint8, device=device)
    step = lambda: gb.scan_inclusive(x, out=y, temp=temp)  # noqa: E731

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    sampler = ClockSampler(device.index if world == 1 else int(os.environ.get("LOCAL_RANK", "0")))
    if rank == 0:
        sampler.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(device)
    torch.cuda.synchronize()
    # The timed region: K calls back to back, events only at its two ends (an event
    # between a call's status clear and its kernel, or between calls, would stop the
    # programmatic dependent launches from overlapping).
    t_wall0 = time.time()
    # A device-side sleep queued ahead of the start event keeps the GPU busy while
    # the host enqueues the first steps, so the region opens on queued work: the
    # host's launch latency for the first call stays out of a short run's figure.
    torch.cuda._sleep(2_000_000)  # about 1 ms of clock cycles
    ev0.record(stream)
    for i in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(device)
    ms_total = ev0.elapsed_time(ev1)
    ms_total_max = max_over_ranks(ms_total, device)
    if gb.device_error() != gb.OK:
        raise RuntimeError("device-side error during the timed region")
    # Per-call device time through the library's profile events (status clear +
    # kernel of one call, not overlapped with the next): reported beside the
    # timed-region figure, on fewer calls.
    kcalls = max(3, min(args.steps, 200))
    k_before = [torch.cuda.Event(enable_timing=True) for _ in range(kcalls)]
    k_after = [torch.cuda.Event(enable_timing=True) for _ in range(kcalls)]
    for e in k_before + k_after:
        e.record(stream)
    torch.cuda.synchronize()
    for i in range(kcalls):
        gb.set_profile_events(k_before[i], k_after[i])
        step()
    gb.set_profile_events(None, None)
    torch.cuda.synchronize()
    call_ms_events = float(np.mean([b.elapsed_time(a) for b, a in zip(k_before, k_after)]))

    # End to end through the C ABI's host-buffer scan: pinned host input -> device ->
    # scan -> pinned host output, in chunks whose copies overlap the scans.
    xh = torch.from_numpy(x_host).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    work = torch.empty(gb.host_scan_work_bytes(torch.float32, n), dtype=torch.uint8, device=device)
    e2e_step = lambda: gb.scan_inclusive_host(xh, out=yh, work=work, stream=stream)  # noqa: E731
    e2e_steps = max(3, min(args.steps, 30))
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    a_h, a_d = yh[-1000:].numpy().astype(np.float64), y[-1000:].cpu().numpy().astype(np.float64)
    if not np.all(np.abs(a_h - a_d) <= 1e-4 * (1.0 + np.abs(a_d))) or gb.device_error() != gb.OK:
        raise RuntimeError("host-buffer scan disagrees with the device scan")  # different sum order: a tolerance
    barrier(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, device)
    barrier(device)

    extra = None
    if rank == 0 and not args.headline_only and world == 1 and (n == N_HEAD or args.workloads):
        extra = secondary_workloads(device, hbm_peak, only=set(args.workloads.split(",")) if args.workloads else None)
    if rank == 0:
        sampler.stop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and n == N_HEAD:
        n_s, times = cpu_oracle_leg(x_host, 3, budget_s=30.0)
        t = min(times)
        cpu = {"value": round(2 * n_s * 4 / t / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": "fp32 inclusive scan of %d of the headline's values (fp64 accumulation), best of 3, "
                         "one host thread" % n_s}
        cpu.update(host_cpu())  # the machine's cores and CPU model beside the one thread used

    if rank != 0:
        return
    ms_per_step = ms_total_max / args.steps
    value = world * nbytes / (ms_per_step * 1e-3) / 1e9
    # The dominant kernel runs once per step; its average launch duration over the
    # timed region is at most the region's time per step (which also holds the
    # overlapped status clears), so `achieved` is a lower bound on its rate.
    kernel_ms = ms_total / args.steps
    achieved = nbytes / (kernel_ms * 1e-3) / 1e9
    # The library runs the L2-resident persistent kernel for one long aligned row of
    # at least 152 SMs x 16 tiles of 4096 elements, the one-CTA-per-tile kernel below.
    kname = "scan_stash_kernel<float,add>" if n >= 152 * 16 * 4096 else "scan_rows_kernel<float,add>"
    traffic = traffic_from_profiles(kname)
    clocks = sampler.summary(t_wall0, t_wall1)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": round(value / world / PAGE_FP32_1E8_GBS, 3) if n == N_HEAD else None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": ("fp32_1e8: inclusive add scan of n=1e8 fp32 ~N(0,1), seed 2, 1-D contiguous"
                                if n == N_HEAD else "fp32 inclusive scan, n=%d (reduced size, not the headline)" % n),
                   "n": n, "l2": "inputs larger than L2 (%d MB in + %d MB out vs 129 MB L2), no flush"
                                 % (n * 4 >> 20, n * 4 >> 20),
                   "parallelism": "replicas" if world > 1 else "1 GPU",
                   "step": "gb_scan_inclusive = status clear kernel + one single-pass kernel, chained by "
                           "programmatic dependent launch"},
        "frac_of_hbm_peak": round(value / world / hbm_peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                     "kernel": kname, "kernel_us_mean": round(kernel_ms * 1e3, 2),
                     "kernel_time_source": "timed region / launches of the dominant kernel (one per step; "
                                           "includes the overlapped status clears)",
                     "call_us_profile_events": round(call_ms_events * 1e3, 2),
                     "algorithmic_bytes_per_launch": nbytes, "peak_source": peak_src},
        "e2e": {"value": round(world * nbytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": n * 4, "d2h_bytes_per_step": n * 4, "steps": e2e_steps,
                "ms_per_step": round(e2e_ms, 3),
                "call": "gb_scan_inclusive_host (pinned host buffers; 48 MiB chunks, copies in and out "
                        "overlapping the scans)"},
        "gpu_launches": 2 * args.steps, "launches_per_step": {"status clear": 1, kname: 1},
        "clocks": clocks,
        "compaction_headline": None,
        "cpu_baseline": cpu,
        "page_context": {"rtx5080_fp32_1e8_us": PAGE_FP32_1E8_US, "rtx5080_fp32_1e8_GB_s": round(PAGE_FP32_1E8_GBS, 1)},
    }
    if extra:
        line["workloads"] = extra
        c = extra.get("compact_p0.5")
        if c:
            line["compaction_headline"] = {"workload": "compact_p0.5 (fp32 1e7, x<0.5)",
                                           "value": c["throughput"], "unit": "Gelem/s",
                                           "by_selectivity": {
                                               k.split("_p")[1]: {"Gelem_s": extra[k]["throughput"],
                                                                  "kernel_us": extra[k]["kernel_us_best"],
                                                                  "frac_hbm": extra[k]["frac_hbm"]}
                                               for k in ("compact_p0.01", "compact_p0.5", "compact_p0.99")
                                               if k in extra}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workloads", default="",
                    help="comma-separated names of the other workloads to time (default: all)")
    ap.add_argument("--n", type=int, default=N_HEAD,
                    help="headline size (default 1e8); smaller values are for profiling runs only")
    ap.add_argument("--profile", metavar="WORKLOAD", default=None,
                    help="run only WORKLOAD's call (3 untimed, then --steps with L2 flushed) for ncu")
    ap.add_argument("--fp64-add-rate", action="store_true",
                    help="build and run the FP64 / FP32 add-rate probe (the fp64 scans' roofline), print it, exit")
    ap.add_argument("--source-hash", metavar="KERNEL", default=None,
                    help="print the source hash that profiles/ summaries of KERNEL record, and exit")
    args = ap.parse_args(argv)
    if args.fp64_add_rate:
        print(json.dumps(fp64_add_rate()))
        return
    if args.source_hash:
        print(kernel_source_hash(args.source_hash))
        return
    if args.profile:
        profile_workload(args.profile, args.steps)
        return
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    rank, world, local_rank = dist_init()
    if args.impl == "reference":
        reference_arm(args, rank)
    else:
        our_arm(args, rank, world, local_rank)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
