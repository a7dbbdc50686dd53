#!/usr/bin/env python3
"""Throughput of the fused row softmax on one GB300 (or N, as replicas).

One step = one softmax_rows call (the whole hot path: plan, persistent
schedule, row load, max, exp-sum, normalise-and-store) over the workload's
M x N matrix, inputs resident in HBM. The headline workload is the FP32
4096 x 4096 matrix with extreme rows (seed 1).

Cold-L2 lane (default): before every step a 512 MiB (>= 4x L2) buffer is READ
outside the event pair, evicting the L2 without leaving dirty lines that the
timed kernel would have to write back. Each step is timed with CUDA events
on the stream the kernel is launched on; value = algorithmic bytes
(2*M*N*elem_bytes per step, one read and one write of every element) over the
summed step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME|all]
                  [--lane cold|warm] [--impl ours|reference]

--impl reference times the CPU oracle (the plain FP64 C implementation) on the
host cores, on the same workload and metric. Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

NOMINAL_HBM_GBS = 8000.0  # the bar's denominator: ~8 TB/s HBM3e
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 512 << 20
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASON_NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=None,
                    help="one of %s; 'all' (those five) or 'wide' (%s)"
                         % (", ".join(synth.WORKLOADS), ", ".join(synth.WIDE_FEW)))
    ap.add_argument("--api", choices=("rows", "split", "masked", "backward", "rmsnorm"),
                    default="rows",
                    help="rows: softmax_rows / softmax_rows_ex; split: softmax_rows_split "
                         "with a device workspace (the split plan for few, wide rows); masked: "
                         "softmax_rows_masked with the workload's causal period (masked "
                         "entries are not read); backward: softmax_rows_backward_ex on the "
                         "backward shapes (%s); rmsnorm: rmsnorm_residual_rows_ex on the RMSNorm "
                         "shapes (%s); 'all' for every shape of the lane"
                         % (", ".join(synth.BACKWARD), ", ".join(synth.RMSNORM)))
    ap.add_argument("--lane", choices=("cold", "warm"), default="cold")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--plan", type=int, default=0, help="forced plan (0 = automatic)")
    ap.add_argument("--cpu-budget", type=float, default=6.0,
                    help="seconds of oracle time for the CPU baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--burst", type=float, default=1.0, help="seconds of load before timing")
    ap.add_argument("--rows", type=int, default=0,
                    help="use only the first ROWS rows (small cases for profiling)")
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


def recorded_traffic(workload: str, plan: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current sources of the kernel this plan runs (else None)."""
    from memory_bound_row_rows_gb300 import _build
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d.get(workload)
        files = _build.PLAN_SOURCES.get(plan)
        if rec and files and rec.get("plan") == plan and \
                rec.get("source_hash") == _build.source_hash(files):
            return rec.get("dram_bytes_per_launch"), rec
    except (OSError, ValueError, KeyError):
        pass
    return None, None


# ---- clocks --------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampled every 100 ms in the background while the GPU is loaded."""

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        cmd = ["nvidia-smi", "--query-gpu=" + CLOCK_FIELDS, "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return self

        def reader():
            for line in self.proc.stdout:
                self.lines.append(line.strip())
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(REASON_NAMES, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- CPU oracle leg (cpu_baseline and the reference arm) -------------------------

def oracle_pass(w, x, nthreads):
    import oracle
    t0 = time.perf_counter()
    y = oracle.softmax_rows(x.reshape(-1), w.M, w.N, w.ld_in, w.ld_out, w.dtype,
                            nthreads=nthreads)
    return time.perf_counter() - t0, y


def cpu_baseline(w, x, budget_s: float):
    """The oracle as it stands, on all host cores, repeated for about budget_s."""
    nthreads = synth.host_threads()
    times, y = [], None
    t_start = time.perf_counter()
    while True:
        dt, y = oracle_pass(w, x, nthreads)
        times.append(dt)
        if time.perf_counter() - t_start >= budget_s:
            break
    gbs = w.fused_bytes * len(times) / sum(times) / 1e9
    # The same oracle on one core, over the leading rows (about a tenth of the budget).
    import oracle
    rows = max(1, min(w.M, int(w.M * 0.1 * budget_s / max(1e-9, 16 * sum(times) / len(times)))))
    t0 = time.perf_counter()
    oracle.softmax_rows(x[:rows].reshape(-1), rows, w.N, w.ld_in, w.ld_out, w.dtype, nthreads=1)
    t1 = time.perf_counter() - t0
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": nthreads, "kind": "oracle",
            "sample": "whole %s matrix (%d x %d), %d pass(es) of the FP64 C oracle, %d threads"
                      % (w.name, w.M, w.N, len(times), nthreads),
            "rows_per_s": round(w.M * len(times) / sum(times), 1),
            "serial": {"value": round(2 * rows * w.N * w.elem_bytes / t1 / 1e9, 4), "unit": "GB/s",
                       "cores": 1, "sample": "first %d rows, one pass" % rows}}, y


# ---- GPU leg ----------------------------------------------------------------------

def gpu_uuid(device_index: int):
    import torch
    try:
        u = torch.cuda.get_device_properties(device_index).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


def step_stats(ms) -> dict:
    """Per-step time statistics in µs: median, p10/p90, MAD, min, max."""
    us = np.asarray(ms, dtype=np.float64) * 1e3
    med = float(np.median(us))
    return {"median_step_us": round(med, 3),
            "p10_p90_step_us": [round(float(np.percentile(us, 10)), 3),
                                round(float(np.percentile(us, 90)), 3)],
            "mad_step_us": round(float(np.median(np.abs(us - med))), 3),
            "min_max_step_us": [round(float(us.min()), 3), round(float(us.max()), 3)]}


def timed_steps(args, step, flush_l2, stream, rank, local_rank, world):
    """Warm-up, a burst of load, then exactly args.steps steps, each between a
    pair of CUDA events on `stream` (the L2 flush, if any, outside the pair),
    with nvidia-smi sampling the clocks throughout. Returns (ms list, clocks)."""
    import torch
    for _ in range(max(3, args.warmup)):
        flush_l2()
        step()
    torch.cuda.synchronize()
    clk = ClockSampler(gpu_uuid(local_rank) if rank == 0 else None)
    with clk:
        t_end = time.perf_counter() + args.burst
        while time.perf_counter() < t_end:
            for _ in range(20):
                flush_l2()
                step()
            torch.cuda.synchronize()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        for k in range(args.steps):
            flush_l2()
            starts[k].record(stream)
            step()
            ends[k].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)], clk.summary()


def run_ours(args, w, rank, local_rank, world):
    import torch

    import memory_bound_row_rows_gb300 as sr

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    lib = sr.load()
    x = w.generate()
    tdt = {synth.F32: torch.float32, synth.BF16: torch.bfloat16, synth.F16: torch.float16}[w.dtype]

    def host_tensor(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return t if w.dtype == synth.F32 else t.view(torch.int16).view(tdt)

    x_dev = host_tensor(x).to(dev)
    y_dev = torch.empty((w.M, w.ld_out), dtype=tdt, device=dev)
    ws, ws_bytes = None, 0
    if args.api == "split":
        ws_bytes = sr.softmax_rows_split_workspace_bytes(x_dev, y_dev, w.M, w.N, w.ld_in,
                                                         w.ld_out, w.dtype)
        ws = torch.empty(max(16, ws_bytes), dtype=torch.uint8, device=dev)
    # float32 so the reduction reads the buffer directly (an int32 sum would
    # first widen it to int64, writing 1 GiB and leaving dirty lines in L2).
    flush = torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    plan_used = sr.softmax_rows_plan(x_dev, y_dev, w.M, w.N, w.ld_in, w.ld_out, w.dtype) \
        if args.plan == 0 else args.plan

    def step():
        if args.api == "split":
            st = lib.softmax_rows_split(x_dev.data_ptr(), y_dev.data_ptr(), w.M, w.N, w.ld_in,
                                        w.ld_out, w.dtype, ws.data_ptr(), ws_bytes, sh)
        elif args.api == "masked":
            st = lib.softmax_rows_masked(x_dev.data_ptr(), y_dev.data_ptr(), w.M, w.N, w.ld_in,
                                         w.ld_out, w.dtype, None, w.causal_period, args.plan, sh)
        else:
            st = lib.softmax_rows_ex(x_dev.data_ptr(), y_dev.data_ptr(), w.M, w.N, w.ld_in,
                                     w.ld_out, w.dtype, args.plan, sh)
        if st != 0:
            raise RuntimeError("softmax_rows failed: %s" % sr.softmax_rows_strerror(st))

    def flush_l2():
        if args.lane == "cold":
            torch.sum(flush)  # reads 512 MiB: L2 now holds clean lines only

    ms, clocks = timed_steps(args, step, flush_l2, stream, rank, local_rank, world)
    assert sr.softmax_rows_last_device_error() == sr.SR_OK

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, x, dev, lib, host_tensor, tdt)
    if args.api == "split":
        plan_used = "split"
    elif args.api == "masked":
        plan_used = "masked-" + sr.PLAN_NAMES.get(plan_used, str(plan_used))
    return {"ms": ms, "clocks": clocks,
            "plan": plan_used if isinstance(plan_used, str) else sr.PLAN_NAMES.get(plan_used, str(plan_used)),
            "y_dev": y_dev, "e2e": e2e, "x": x}


def run_e2e(args, w, x, dev, lib, host_tensor, tdt):
    """Same metric through the C ABI with host buffers, timed around whole calls with the
    input in pinned host memory and the result landing back in pinned host memory. Two
    public entry points: softmax_rows_host_mapped (the kernel reads and writes the mapped
    host buffers itself, zero copy) and softmax_rows_host (staged through a device
    workspace, copy-in, compute and copy-out of chunks overlapped on three streams).
    The line reports the faster, and both figures."""
    import torch
    import memory_bound_row_rows_gb300 as sr
    x_pin = host_tensor(x).pin_memory()
    y_pin = torch.empty((w.M, w.ld_out), dtype=tdt).pin_memory()
    need = sr.softmax_rows_host_workspace_bytes(w.M, w.N, w.dtype)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def staged():
        st = lib.softmax_rows_host(x_pin.data_ptr(), y_pin.data_ptr(), w.M, w.N, w.ld_in,
                                   w.ld_out, w.dtype, ws.data_ptr(), need, stream.cuda_stream)
        if st != 0:
            raise RuntimeError("softmax_rows_host failed: %s" % sr.softmax_rows_strerror(st))

    def mapped():
        st = lib.softmax_rows_host_mapped(x_pin.data_ptr(), y_pin.data_ptr(), w.M, w.N, w.ld_in,
                                          w.ld_out, w.dtype, stream.cuda_stream)
        if st != 0:
            raise RuntimeError("softmax_rows_host_mapped failed: %s" % sr.softmax_rows_strerror(st))

    def timed(step):
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        k = max(3, min(args.steps, 20))
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(k):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / 1e3 / k, k

    sec_m, k = timed(mapped)
    sec_s, _ = timed(staged)
    eb = w.elem_bytes
    best_mapped = sec_m <= sec_s
    sec = sec_m if best_mapped else sec_s
    return {"value": round(w.fused_bytes / sec / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": w.M * w.N * eb, "d2h_bytes_per_step": w.M * w.N * eb,
            "ms_per_step": round(sec * 1e3, 4), "steps": k,
            "path": ("softmax_rows_host_mapped: the kernel reads pinned host input and writes "
                     "pinned host output over the host link (zero copy)") if best_mapped else
                    ("softmax_rows_host: pinned host -> device workspace -> pinned host, "
                     "chunks overlapped on three streams"),
            "mapped_gbs": round(w.fused_bytes / sec_m / 1e9, 2),
            "staged_gbs": round(w.fused_bytes / sec_s / 1e9, 2)}


def parity_vs_oracle(w, y_dev, y_ref, max_elements: int = 1 << 25):
    """Compare the GPU output with the CPU-baseline leg's oracle output.

    Every row when the matrix has at most ``max_elements`` entries, otherwise
    an evenly strided subset of rows (always including the first and last).
    """
    import torch
    step = max(1, -(-w.M * w.N // max_elements))
    rows = np.unique(np.concatenate([np.arange(0, w.M, step), [w.M - 1]]))
    y = y_dev[torch.from_numpy(rows).to(y_dev.device)].detach().cpu()
    if w.dtype != synth.F32:
        y = y.view(torch.int16)
    y = y.numpy()
    if w.dtype != synth.F32:
        y = y.view(np.uint16)
    g = synth.storage_to_float64(y[:, :w.N], w.dtype)
    r = synth.storage_to_float64(y_ref[rows, :w.N], w.dtype)
    atol = 1e-6 if w.dtype == synth.F32 else 4e-3
    bad = ~(np.abs(g - r) <= atol + atol * np.abs(r))
    bad &= ~(np.isnan(g) & np.isnan(r))
    return {"rows": int(rows.size), "of_rows": w.M, "elements": int(g.size),
            "outside_tolerance": int(bad.sum()), "atol": atol, "rtol": atol,
            "max_abs_err": float(np.nanmax(np.abs(g - r)))}


def algorithmic_bytes(w, api: str) -> int:
    """Bytes one call must move: every element read once and written once; with
    the causal mask applied in the kernel, only the valid entries are read."""
    if api == "masked" and w.causal_period > 0:
        P = w.causal_period
        full, rest = divmod(w.M, P)
        def valid_sum(rows):  # rows 0..rows-1 of one period
            return sum(min(w.N, q + 1) for q in range(rows))
        valid = full * valid_sum(P) + valid_sum(rest)
        return w.elem_bytes * (valid + w.M * w.N)
    return w.fused_bytes


def max_over_ranks(value: float, device="cpu") -> float:
    """The largest of every rank's value (identity without a process group)."""
    import torch
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(fused_bytes: int, steps: int, world: int, slowest_total_s: float) -> float:
    """Whole-job GB/s when every rank runs the full workload (weak scaling):
    all ranks' bytes over the slowest rank's time."""
    return world * fused_bytes * steps / slowest_total_s / 1e9


def bench_ours(args, w):
    import torch
    rank, local_rank, world = dist_env()
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl")
    from memory_bound_row_rows_gb300 import _build
    res = run_ours(args, w, rank, local_rank, world)
    ms = res["ms"]
    total_s = max_over_ranks(sum(ms) / 1e3, device="cuda" if world > 1 else "cpu")
    if rank != 0:
        return None
    steps = len(ms)
    mean_s = total_s / steps
    nbytes = algorithmic_bytes(w, args.api)
    value = replica_throughput(nbytes, steps, world, total_s)
    peaks = measured_peaks()
    src_hash = _build.source_hash(_build.PLAN_SOURCES.get(res["plan"]))
    traffic, rec = recorded_traffic(w.name, res["plan"])
    achieved = nbytes / (sum(ms) / 1e3 / steps) / 1e9
    line = {
        "metric": ("cold-L2 softmax GB/s (2*M*N*bytes/time)" if args.lane == "cold"
                   else "warm-L2 softmax GB/s (2*M*N*bytes/time)") if args.api != "masked"
        else "cold-L2 masked softmax GB/s ((valid reads + M*N writes)*bytes/time)",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": round(mean_s * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": synth.DTYPE_NAMES[w.dtype],
        "data": "synthetic: seeded SplitMix64/Box-Muller (seed %d), generated on the host" % w.seed,
        "config": {"workload": w.name, "M": w.M, "N": w.N, "ld_in": w.ld_in, "ld_out": w.ld_out,
                   "plan": res["plan"], "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": ("flushed: a 512 MiB device buffer is read before every step, outside "
                          "the event pair") if args.lane == "cold" else "warm (no flush)",
                   "inputs_resident_in_hbm": True},
        "pct_of_8000_gbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_hbm": round(100 * value / world / peaks["hbm_gbs"], 2),
        "rows_per_s": round(world * w.M * steps / total_s, 1),
        "bytes_per_step": nbytes,
        "dense_equivalent_gbs": round(world * w.fused_bytes * steps / total_s / 1e9, 2),
        **step_stats(ms),
        "gpu_launches": steps * (2 if res["plan"] == "split" else 1),
        "clocks": res["clocks"],
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": traffic,
                     "traffic_note": (rec or {}).get("note") if traffic else
                     "null: no ncu capture recorded for the current kernel sources"},
        "source_hash": src_hash,
    }
    if res["e2e"] is not None:
        line["e2e"] = res["e2e"]
    if world == 1:
        cpu, y_ref = cpu_baseline(w, res["x"], args.cpu_budget)
        line["cpu_baseline"] = cpu
        line["parity"] = parity_vs_oracle(w, res["y_dev"], y_ref)
    return line


# ---- row-pair lanes: softmax backward and residual RMSNorm ----------------------

def _ulp(r, dtype):
    mant = {synth.F32: 23, synth.BF16: 7, synth.F16: 10}[dtype]
    emin = {synth.F32: -126, synth.BF16: -126, synth.F16: -14}[dtype]
    a = np.abs(r)
    return np.exp2(np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), emin) - mant)


class BackwardLane:
    """dx = y * (dy - sum(y * dy)) per row: y ~ U[0, 2/N), dy ~ N(0, 1)."""
    api = "backward"
    catalog = synth.BACKWARD
    headline = synth.BACKWARD_HEADLINE
    label = "softmax backward"
    model = "3*M*N*bytes"

    def __init__(self, w):
        self.w = w
        self.mats = [w.y_rows(0, w.M), w.dy_rows(0, w.M)]
        self.vecs = []

    data = property(lambda self: "synthetic: y ~ U[0, 2/N), dy ~ N(0, 1), seeded SplitMix64 "
                                 "(seed %d)" % self.w.seed)

    def call(self, lib, dev_mats, dev_vecs, out, plan, stream):
        w = self.w
        return lib.softmax_rows_backward_ex(dev_mats[0].data_ptr(), dev_mats[1].data_ptr(),
                                            out.data_ptr(), w.M, w.N, w.ld, w.ld, w.N, w.dtype,
                                            plan, stream)

    def plan(self, sr, dev_mats, dev_vecs, out, plan):
        w = self.w
        return sr.softmax_rows_backward_plan(dev_mats[0], dev_mats[1], out, w.M, w.N, w.ld, w.ld,
                                             w.N, w.dtype, plan, 0)

    def oracle_rows(self, rows):
        import oracle
        w = self.w
        y, dy = (np.ascontiguousarray(m[rows]).reshape(-1) for m in self.mats)
        return oracle.load().softmax_backward(y, dy, len(rows), w.N, w.ld, w.ld, w.N, w.dtype)

    def outside_gate(self, g, r, rows):
        """|g - r| <= |y|(2^-17 S + 2^-22 |dy - d|) + 2^-22 |r| + 2 ulp(r), d = sum y*dy and
        S = sum |y*dy| per row (the FP32 dot product's error bound, one cast)."""
        dec = lambda a: synth.storage_to_float64(np.ascontiguousarray(a[:, :self.w.N]),
                                                 self.w.dtype)
        y, dy = dec(self.mats[0][rows]), dec(self.mats[1][rows])
        d = (y * dy).sum(axis=1, keepdims=True)
        S = np.abs(y * dy).sum(axis=1, keepdims=True)
        tol = (np.abs(y) * (2.0 ** -17 * S + 2.0 ** -22 * np.abs(dy - d)) + 2.0 ** -22 * np.abs(r)
               + 2 * _ulp(r, self.w.dtype))
        return int((~(np.abs(g - r) <= tol) & ~(np.isnan(g) & np.isnan(r))).sum())

    gate = "FP32 dot-product error bound plus 2 ulp of the dtype"


class RmsNormLane(BackwardLane):
    """y = dtype(h * w / sqrt(mean(h^2) + eps)), h = dtype(x + residual)."""
    api = "rmsnorm"
    catalog = synth.RMSNORM
    headline = synth.RMSNORM_HEADLINE
    label = "residual RMSNorm"
    model = "(3*M*N + N)*bytes"

    def __init__(self, w):
        self.w = w
        self.mats = [w.x_rows(0, w.M), w.residual_rows(0, w.M)]
        self.vecs = [w.weight()]

    data = property(lambda self: "synthetic: x, residual ~ N(0, 1), weight ~ U[0.5, 1.5), "
                                 "eps %g, seeded SplitMix64 (seed %d)" % (self.w.eps, self.w.seed))

    def call(self, lib, dev_mats, dev_vecs, out, plan, stream):
        w = self.w
        return lib.rmsnorm_residual_rows_ex(dev_mats[0].data_ptr(), dev_mats[1].data_ptr(),
                                            dev_vecs[0].data_ptr(), out.data_ptr(), w.M, w.N, w.ld,
                                            w.ld, w.N, w.eps, w.dtype, plan, stream)

    def plan(self, sr, dev_mats, dev_vecs, out, plan):
        w = self.w
        return sr.rmsnorm_residual_rows_plan(dev_mats[0], dev_mats[1], dev_vecs[0], out, w.M, w.N,
                                             w.ld, w.ld, w.N, w.eps, w.dtype, plan, 0)

    def oracle_rows(self, rows):
        import oracle
        w = self.w
        x, r = (np.ascontiguousarray(m[rows]).reshape(-1) for m in self.mats)
        return oracle.load().rmsnorm_residual(x, r, self.vecs[0], len(rows), w.N, w.ld, w.ld, w.N,
                                              float(np.float32(w.eps)), w.dtype)

    def outside_gate(self, g, r, rows):
        """|g - r| <= 2^-16 |r| + ulp(r): FP32 reduction and scaling, one cast."""
        tol = 2.0 ** -16 * np.abs(r) + _ulp(r, self.w.dtype)
        return int((~(np.abs(g - r) <= tol) & ~(np.isnan(g) & np.isnan(r))).sum())

    gate = "FP32 RMS error bound plus 1 ulp of the dtype"


LANES = {"backward": BackwardLane, "rmsnorm": RmsNormLane}


def pair_cpu_sample(lane):
    """Leading rows of the workload, about 8 MB of algorithmic traffic."""
    w = lane.w
    per_row = 3 * w.N * w.elem_bytes
    return np.arange(min(w.M, max(1, (8 << 20) // per_row))), per_row


def pair_cpu_baseline(lane, budget_s: float):
    """The oracle as it stands (one thread) on leading rows, repeated for about budget_s."""
    rows, per_row = pair_cpu_sample(lane)
    times = []
    t_start = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        lane.oracle_rows(rows)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start >= budget_s:
            break
    gbs = per_row * rows.size * len(times) / sum(times) / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "first %d of %d rows of %s, %d pass(es) of the FP64 C oracle's %s, 1 thread"
                      % (rows.size, lane.w.M, lane.w.name, len(times), lane.label)}


def bench_pair(args, lane):
    """One row-pair call per step (softmax_rows_backward_ex or rmsnorm_residual_rows_ex)."""
    import torch

    import memory_bound_row_rows_gb300 as sr
    from memory_bound_row_rows_gb300 import _build
    w = lane.w
    rank, local_rank, world = dist_env()
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    lib = sr.load()
    tdt = {synth.F32: torch.float32, synth.BF16: torch.bfloat16, synth.F16: torch.float16}[w.dtype]

    def host_tensor(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return t if w.dtype == synth.F32 else t.view(torch.int16).view(tdt)

    dev_mats = [host_tensor(m).to(dev) for m in lane.mats]
    dev_vecs = [host_tensor(v).to(dev) for v in lane.vecs]
    out = torch.empty((w.M, w.N), dtype=tdt, device=dev)
    flush = torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    plan = lane.plan(sr, dev_mats, dev_vecs, out, args.plan)
    if plan < 0:
        raise RuntimeError("plan %d cannot take %s %s" % (args.plan, lane.api, w.name))

    def step():
        st = lane.call(lib, dev_mats, dev_vecs, out, args.plan, sh)
        if st != 0:
            raise RuntimeError("%s failed: %s" % (lane.api, sr.softmax_rows_strerror(st)))

    def flush_l2():
        if args.lane == "cold":
            torch.sum(flush)

    ms, clocks = timed_steps(args, step, flush_l2, stream, rank, local_rank, world)
    total_s = max_over_ranks(sum(ms) / 1e3, device="cuda" if world > 1 else "cpu")

    e2e = None
    if not args.no_e2e:
        # Host buffers: the pinned inputs copied in, the call, the output copied back.
        pins = [host_tensor(m).pin_memory() for m in lane.mats + lane.vecs]
        out_pin = torch.empty((w.M, w.N), dtype=tdt).pin_memory()
        targets = dev_mats + dev_vecs

        def e2e_step():
            for d, h in zip(targets, pins):
                d.copy_(h, non_blocking=True)
            step()
            out_pin.copy_(out, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        k = max(3, min(args.steps, 20))
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(k):
            e2e_step()
        t1.record(stream)
        torch.cuda.synchronize()
        sec = t0.elapsed_time(t1) / 1e3 / k
        e2e = {"value": round(w.fused_bytes / sec / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": sum(p.numel() * p.element_size() for p in pins),
               "d2h_bytes_per_step": w.M * w.N * w.elem_bytes,
               "ms_per_step": round(sec * 1e3, 4), "steps": k,
               "path": "pinned host inputs -> device (copies), %s call, output -> pinned host, "
                       "in order on one stream" % lane.api}
    if rank != 0:
        return None
    steps = len(ms)
    value = replica_throughput(w.fused_bytes, steps, world, total_s)
    achieved = w.fused_bytes / (sum(ms) / 1e3 / steps) / 1e9
    peaks = measured_peaks()
    pname = "%s-%s" % (lane.api, sr.PLAN_NAMES[plan])
    traffic, rec = recorded_traffic("%s:%s" % (lane.api, w.name), lane.api)
    lanename = "cold-L2" if args.lane == "cold" else "warm-L2"
    line = {
        "metric": "%s %s GB/s (%s/time)" % (lanename, lane.label, lane.model),
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(total_s / steps * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": synth.DTYPE_NAMES[w.dtype], "data": lane.data,
        "config": {"workload": "%s %s" % (lane.api, w.name), "M": w.M, "N": w.N, "ld": w.ld,
                   "plan": pname, "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": ("flushed: a 512 MiB device buffer is read before every step, outside "
                          "the event pair") if args.lane == "cold" else "warm (no flush)",
                   "inputs_resident_in_hbm": True},
        "pct_of_8000_gbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_hbm": round(100 * value / world / peaks["hbm_gbs"], 2),
        "bytes_per_step": w.fused_bytes,
        **step_stats(ms),
        "gpu_launches": steps,
        "clocks": clocks,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": traffic,
                     "traffic_note": (rec or {}).get("note") if traffic else
                     "null: no ncu capture recorded for the current kernel sources"},
        "source_hash": _build.source_hash(_build.PLAN_SOURCES[lane.api]),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if world == 1:
        line["cpu_baseline"] = pair_cpu_baseline(lane, args.cpu_budget)
        rows = np.unique(np.concatenate([np.linspace(0, w.M - 1, 64).astype(np.int64),
                                         [w.M - 1]]))
        g = out[torch.from_numpy(rows).to(dev)].cpu()
        g = g.numpy() if w.dtype == synth.F32 else g.view(torch.int16).numpy().view(np.uint16)
        r = lane.oracle_rows(rows)
        dec = lambda a: synth.storage_to_float64(np.ascontiguousarray(a[:, :w.N]), w.dtype)
        line["parity"] = {"rows": int(rows.size), "of_rows": w.M,
                          "outside_tolerance": lane.outside_gate(dec(g), dec(r), rows),
                          "gate": lane.gate}
    return line


def bench_reference(args, w):
    """The CPU oracle as the reference arm: each step is one oracle pass over the workload."""
    rank, _, world = dist_env()
    if rank != 0:
        return None
    x = w.generate()
    nthreads = synth.host_threads()
    for _ in range(max(0, args.warmup)):
        oracle_pass(w, x, nthreads)
    times = []
    for _ in range(args.steps):
        dt, _y = oracle_pass(w, x, nthreads)
        times.append(dt)
    total = sum(times)
    value = w.fused_bytes * len(times) / total / 1e9
    return {
        "impl": "reference",
        "metric": "cold-L2 softmax GB/s (2*M*N*bytes/time)",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": len(times),
        "warmup": args.warmup, "ms_per_step": round(1e3 * total / len(times), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": synth.DTYPE_NAMES[w.dtype],
        "data": "synthetic: seeded SplitMix64/Box-Muller (seed %d)" % w.seed,
        "config": {"workload": w.name, "M": w.M, "N": w.N, "ld_in": w.ld_in, "ld_out": w.ld_out},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nthreads,
                         "kind": "oracle",
                         "sample": "whole %s matrix per step, FP64 C oracle, %d threads"
                                   % (w.name, nthreads)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def bench_reference_pair(args, lane):
    """The CPU oracle as the reference arm of a row-pair lane, each step a bounded sample."""
    rank, _, world = dist_env()
    if rank != 0:
        return None
    w = lane.w
    rows, per_row = pair_cpu_sample(lane)
    for _ in range(max(0, args.warmup)):
        lane.oracle_rows(rows)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        lane.oracle_rows(rows)
        times.append(time.perf_counter() - t0)
    value = per_row * rows.size * len(times) / sum(times) / 1e9
    sample = "first %d of %d rows of %s per step, FP64 C oracle's %s, 1 thread" % (
        rows.size, w.M, w.name, lane.label)
    return {
        "impl": "reference",
        "metric": "cold-L2 %s GB/s (%s/time)" % (lane.label, lane.model),
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": len(times),
        "warmup": args.warmup, "ms_per_step": round(1e3 * sum(times) / len(times), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": synth.DTYPE_NAMES[w.dtype], "data": lane.data,
        "config": {"workload": "%s %s" % (lane.api, w.name), "M": w.M, "N": w.N, "ld": w.ld},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    if args.api in LANES:
        lane_cls = LANES[args.api]
        catalog = lane_cls.catalog
        names = (list(catalog) if args.workload == "all" else
                 [args.workload or lane_cls.headline])
    else:
        catalog = dict(synth.WORKLOADS, **synth.WIDE_FEW)
        wl = args.workload or synth.HEADLINE
        names = (list(synth.WORKLOADS) if wl == "all" else
                 list(synth.WIDE_FEW) if wl == "wide" else [wl])
    for name in names:
        w = catalog[name]
        if args.rows:
            w = w.with_rows(min(args.rows, w.M))
        if args.impl == "reference" and args.api in LANES:
            line = bench_reference_pair(args, LANES[args.api](w))
        elif args.impl == "reference":
            line = bench_reference(args, w)
        elif args.api in LANES:
            line = bench_pair(args, LANES[args.api](w))
        else:
            line = bench_ours(args, w)
        if line is not None:
            print(json.dumps(line), flush=True)
    if args.impl == "ours":
        import torch
        if torch.distributed.is_initialized():
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
