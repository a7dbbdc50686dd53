#!/usr/bin/env python3
"""Throughput of the fused row softmax on one GB300 (or N, as replicas).

One step = one softmax_rows call (the whole hot path: plan, schedule, row
load, max, exp-sum, normalise-and-store) over the workload's M x N matrix,
inputs resident in HBM. The default workload is the largest: the FP16 causal
attention-score matrix, 524288 x 2048 (seed 4), 4.29 GB moved per call.

Protocol (cold lane, the default):
  1. The input is generated on the host and copied to the device. One call
     runs and its output is checked against the CPU oracle on sampled rows
     BEFORE any timing; a result outside the tolerance prints an error line
     and exits non-zero.
  2. Cold L2 by rotation: the steps cycle through R input/output sets that
     together span at least 1 GiB (>= 4x the L2); R = 1 when one set alone
     is that large. No flush runs between steps, so every step reads input
     that left the L2 long before, and the write-back of earlier steps'
     outputs falls inside the timed region (steady state).
  3. Timing: CUDA events on the launching stream around batches of
     consecutive launches (about 200 us of work per batch, at least five
     batches), so the event timer's granularity is spread over the batch.
     The step time is the median over batches of batch time / launches;
     value = algorithmic bytes / that median (2*M*N*elem_bytes per step);
     the mean step is reported beside it.
  4. The output of the last timed call is checked against the oracle again.
  5. copy_baseline: softmax_rows_copy_ceiling, a copy of exactly the bytes the
     softmax moves at the same pitches with the same 16-byte streaming accesses,
     on the same sets and batches (torch's copy_ beside it); the row-pair lanes
     (--api backward / rmsnorm) use softmax_rows_copy_ceiling2 (two inputs read,
     one written) and torch's add.
  6. e2e: the same metric through the C ABI with pinned host buffers (pinned
     from a thread on the GPU's NUMA node), copies or host-link traffic inside
     the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME|all|wide]
                  [--lane cold|warm] [--impl ours|reference] [--api ...]

--impl reference times the CPU oracle (the plain FP64 C implementation) on the
host cores, on the same workload and metric. Prints one JSON line per
workload (rank 0).
"""
from __future__ import annotations

import argparse
import json
import math
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
# The cold lane cycles through input/output sets spanning at least this many
# device bytes (>= 4x the L2 of a GB300, checked at run time against the
# device's own L2 size).
ROTATE_BYTES = 1 << 30
# Work per pair of timing events, and the fewest batches a run is cut into.
BATCH_TARGET_US = 200.0
MIN_BATCHES = 5
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
                         "with a device workspace (the split plan for wide rows); masked: "
                         "softmax_rows_masked with the workload's causal period (masked "
                         "entries are not read); backward: softmax_rows_backward_ex on the "
                         "backward shapes (%s); rmsnorm: rmsnorm_residual_rows_ex on the RMSNorm "
                         "shapes (%s); 'all' for every shape of the lane"
                         % (", ".join(synth.BACKWARD), ", ".join(synth.RMSNORM)))
    ap.add_argument("--lane", choices=("cold", "warm"), default="cold")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--plan", type=int, default=0, help="forced plan (0 = automatic)")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle time for the CPU baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-copy", action="store_true", help="skip the copy baseline")
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


def dram_rate(traffic, median_step_us: float, peak_gbs: float) -> dict:
    """DRAM GB/s implied by the recorded bytes per launch (ncu, steady state) over the
    measured median step, beside the algorithmic GB/s: {} when no traffic is recorded."""
    if not traffic or median_step_us <= 0:
        return {}
    gbs = traffic / (median_step_us / 1e6) / 1e9
    return {"dram_gbs": round(gbs, 2), "dram_frac": round(gbs / peak_gbs, 4)}


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


def cpu_baseline(w, x, budget_s: float) -> dict:
    """The oracle as it stands, on all host cores, repeated for about budget_s."""
    nthreads = synth.host_threads()
    times = []
    t_start = time.perf_counter()
    while True:
        dt, _y = oracle_pass(w, x, nthreads)
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
                       "cores": 1, "sample": "first %d rows, one pass" % rows}}


# ---- protocol (host logic, no GPU) ------------------------------------------------

def rotation_count(set_bytes: int, lane: str, rotate_bytes: int = ROTATE_BYTES) -> int:
    """Input/output sets the cold lane cycles through: the fewest whose bytes
    together reach rotate_bytes (1 when one set alone does). The warm lane
    reuses one set."""
    if lane == "warm":
        return 1
    return max(1, -(-int(rotate_bytes) // max(1, int(set_bytes))))


def batch_plan(steps: int, est_us: float, target_us: float = BATCH_TARGET_US,
               min_batches: int = MIN_BATCHES) -> int:
    """Launches per timed batch: enough for about target_us of work, but no
    more than leaves min_batches batches (when there are that many steps)."""
    b = max(1, int(math.ceil(target_us / max(float(est_us), 1e-3))))
    if steps >= min_batches:
        b = min(b, steps // min_batches)
    return max(1, min(b, max(1, steps)))


def batch_bounds(steps: int, b: int):
    """[start, end) step ranges of consecutive batches of b launches (the last may be short)."""
    return [(s, min(s + b, steps)) for s in range(0, steps, b)]


def batch_stats(batch_ms, bounds) -> dict:
    """Per-step statistics in µs from batch times: each batch contributes its
    time / launches; the median and spread are over the full batches (every
    batch when all are short), the mean over every step."""
    per = np.asarray([ms * 1e3 / (e - s) for ms, (s, e) in zip(batch_ms, bounds)],
                     dtype=np.float64)
    full_len = bounds[0][1] - bounds[0][0]
    full = np.asarray([p for p, (s, e) in zip(per, bounds) if e - s == full_len])
    if full.size == 0:
        full = per
    steps = bounds[-1][1]
    med = float(np.median(full))
    return {"median_step_us": round(med, 3),
            "mean_step_us": round(float(sum(batch_ms)) * 1e3 / steps, 3),
            "p10_p90_step_us": [round(float(np.percentile(full, 10)), 3),
                                round(float(np.percentile(full, 90)), 3)],
            "mad_step_us": round(float(np.median(np.abs(full - med))), 3),
            "min_max_step_us": [round(float(full.min()), 3), round(float(full.max()), 3)],
            "batches": len(bounds), "launches_per_batch": full_len}


def l2_protocol(set_bytes: int, lane: str) -> str:
    """The config's statement of how the L2 is kept from serving a step's input."""
    if lane == "warm":
        return "warm: one input/output set, no flush (diagnostic; L2 may serve the input)"
    r = rotation_count(set_bytes, lane)
    if r == 1:
        return ("inputs larger than L2: one input/output set of %.2f GB, no flush; the "
                "write-back of the previous step's output falls inside the timed region"
                % (set_bytes / 1e9))
    return ("rotation: %d input/output sets of %.1f MB (%.2f GB in all, >= 4x L2), no flush; "
            "each step's input was last touched %.2f GB of traffic earlier and the write-back "
            "of earlier outputs falls inside the timed region"
            % (r, set_bytes / 1e6, r * set_bytes / 1e9, (r - 1) * set_bytes / 1e9))


def workload_config(w, lane: str, world: int) -> dict:
    """The config object both arms print for a softmax workload."""
    set_bytes = (w.M * w.ld_in + w.M * w.ld_out) * w.elem_bytes
    return {"workload": w.name, "M": w.M, "N": w.N, "ld_in": w.ld_in, "ld_out": w.ld_out,
            "l2": l2_protocol(set_bytes, lane),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def parity_rows(M: int, N: int, max_elements: int = 1 << 25, seed: int = 12345) -> np.ndarray:
    """Rows the bench checks against the oracle: all of them when the matrix has at
    most max_elements entries, else a seeded sample of about max_elements / N rows
    (always with the first and the last)."""
    if M * N <= max_elements:
        return np.arange(M, dtype=np.int64)
    k = max(2, min(M, max_elements // N))
    rng = np.random.default_rng(seed)
    rows = rng.choice(M, size=k - 2, replace=False).astype(np.int64)
    return np.unique(np.concatenate([rows, [0, M - 1]]))


def oracle_rows(w, x, rows) -> np.ndarray:
    """The oracle's output for the selected rows of the input x (M x ld_in)."""
    import oracle
    xs = np.ascontiguousarray(x[rows])
    return oracle.softmax_rows(xs.reshape(-1), len(rows), w.N, w.ld_in, w.ld_out, w.dtype,
                               nthreads=synth.host_threads())


def compare_rows(w, got, ref, rows) -> dict:
    """The gate |got - ref| <= atol + rtol |ref| (NaN where the oracle is NaN)
    at the tolerances of the workload's dtype, over the given rows."""
    g = synth.storage_to_float64(np.ascontiguousarray(got[:, :w.N]), w.dtype)
    r = synth.storage_to_float64(np.ascontiguousarray(ref[:, :w.N]), w.dtype)
    atol = 1e-6 if w.dtype == synth.F32 else 4e-3
    bad = ~(np.abs(g - r) <= atol + atol * np.abs(r))
    bad &= ~(np.isnan(g) & np.isnan(r))
    diff = np.abs(g - r)
    return {"rows": int(len(rows)), "of_rows": w.M, "elements": int(g.size),
            "outside_tolerance": int(bad.sum()), "atol": atol, "rtol": atol,
            "max_abs_err": float(np.nanmax(diff)) if np.isfinite(diff).any() else 0.0}


# ---- GPU leg ----------------------------------------------------------------------

def gpu_uuid(device_index: int):
    import torch
    try:
        u = torch.cuda.get_device_properties(device_index).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


def device_l2_bytes(dev) -> int:
    import torch
    props = torch.cuda.get_device_properties(dev)
    return int(getattr(props, "L2_cache_size", 0) or 0)


def device_rows(t, rows) -> np.ndarray:
    """Selected rows of a device matrix as host storage (uint16 bits for 16-bit types)."""
    import torch
    y = t[torch.from_numpy(np.asarray(rows, dtype=np.int64)).to(t.device)].detach().cpu()
    if y.dtype in (torch.bfloat16, torch.float16):
        return y.view(torch.int16).numpy().view(np.uint16)
    return y.numpy()


def timed_batches(args, launch, n_sets, stream, rank, local_rank, world):
    """Warm-up, a burst of load, then exactly args.steps launches between CUDA
    events on `stream`, recorded at batch boundaries; step k uses set
    k mod n_sets (the counter runs on through warm-up, so rotation never
    restarts). nvidia-smi samples the clocks during the burst and the timed
    region. Returns (batch ms list, bounds, clocks, set of the last timed step)."""
    import torch
    k = 0

    def run(count):
        nonlocal k
        for _ in range(count):
            launch(k % n_sets)
            k += 1

    run(max(3, args.warmup))
    torch.cuda.synchronize()
    # Estimate a step from a run of launches in one event pair.
    n_est = max(4, min(n_sets, 64))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(n_est)
    e1.record(stream)
    torch.cuda.synchronize()
    est_us = e0.elapsed_time(e1) * 1e3 / n_est
    b = batch_plan(args.steps, est_us)
    bounds = batch_bounds(args.steps, b)
    clk = ClockSampler(gpu_uuid(local_rank) if rank == 0 else None)
    with clk:
        t_end = time.perf_counter() + args.burst
        while time.perf_counter() < t_end:
            run(max(1, min(64, int(20000 / max(est_us, 1.0)))))
            torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(bounds) + 1)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        evs[0].record(stream)
        for j, (s, e) in enumerate(bounds):
            run(e - s)
            evs[j + 1].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
    batch_ms = [evs[j].elapsed_time(evs[j + 1]) for j in range(len(bounds))]
    return batch_ms, bounds, clk.summary(), (k - 1) % n_sets


def kernel_record(sr) -> dict:
    """Registers, local (spill) bytes and launch shape of the last kernel launched."""
    try:
        info = sr.softmax_rows_last_launch()
    except Exception as exc:  # pragma: no cover - reported, not fatal
        return {"error": str(exc)}
    return {"name": info["name"], "registers": info["registers"],
            "local_bytes": info["local_bytes"], "static_smem_bytes": info["static_smem_bytes"],
            "dynamic_smem_bytes": info["dynamic_smem_bytes"], "grid": info["grid"],
            "block": info["block"], "cluster": info["cluster"]}


def parse_cpulist(text: str) -> set:
    """A Linux cpulist ("0-3,8,10-11") as a set of CPU numbers."""
    cpus = set()
    for part in text.strip().split(","):
        if not part:
            continue
        if "-" in part:
            lo, hi = part.split("-")
            cpus.update(range(int(lo), int(hi) + 1))
        else:
            cpus.add(int(part))
    return cpus


def gpu_numa_cpus(dev):
    """The CPUs (of those this process may use) on the NUMA node the GPU's PCI device
    reports in sysfs, and a note saying where they came from; (None, note) when the
    node or its CPUs cannot be found. Host buffers pinned by a thread running there are
    placed in that node's memory, next to the GPU's host link."""
    try:
        import torch
        p = torch.cuda.get_device_properties(dev)
        bus = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        with open("/sys/bus/pci/devices/%s/numa_node" % bus) as f:
            node = int(f.read())
        if node < 0:
            return None, {"gpu_pci": bus, "numa_node": node}
        with open("/sys/devices/system/node/node%d/cpulist" % node) as f:
            cpus = parse_cpulist(f.read()) & os.sched_getaffinity(0)
        return (cpus or None), {"gpu_pci": bus, "numa_node": node, "cpus": len(cpus)}
    except (OSError, ValueError, AttributeError, RuntimeError, AssertionError) as e:
        return None, {"numa": "not found (%s)" % type(e).__name__}


def run_e2e(args, w, x, dev, lib, host_tensor, tdt):
    """Same metric through the C ABI with host buffers, timed around whole calls with the
    input in pinned host memory and the result landing back in pinned host memory. Two
    public entry points: softmax_rows_host_mapped (the kernel reads and writes the mapped
    host buffers itself, zero copy) and softmax_rows_host (staged through a device
    workspace, copy-in, compute and copy-out of chunks overlapped on three streams).
    The line reports the faster, and both figures."""
    import torch
    import memory_bound_row_rows_gb300 as sr
    # Pin the host buffers from a thread on the GPU's NUMA node, so that their pages
    # sit next to its host link; the process's CPU set is restored afterwards.
    cpus, numa = gpu_numa_cpus(dev)
    saved = os.sched_getaffinity(0)
    try:
        if cpus:
            os.sched_setaffinity(0, cpus)
        x_pin = host_tensor(x).pin_memory()
        y_pin = torch.empty((w.M, w.ld_out), dtype=tdt).pin_memory()
        y_pin.zero_()
    finally:
        os.sched_setaffinity(0, saved)
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
            "staged_gbs": round(w.fused_bytes / sec_s / 1e9, 2),
            "host_buffers": numa}



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
    all ranks' bytes over the slowest rank's time (for `steps` steps; the bench
    passes one step and the slowest rank's median step time)."""
    return world * fused_bytes * steps / slowest_total_s / 1e9




class ParityFailure(RuntimeError):
    """The GPU output left the tolerance: no throughput is reported."""

    def __init__(self, line):
        super().__init__("parity gate failed")
        self.line = line


def torch_dtype(dtype):
    import torch
    return {synth.F32: torch.float32, synth.BF16: torch.bfloat16, synth.F16: torch.float16}[dtype]


def to_device(a, dtype, dev):
    """Host storage (float32, or uint16 bits) -> device tensor of the dtype."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype != synth.F32:
        t = t.view(torch.int16).view(torch_dtype(dtype))
    return t.to(dev)


def timed_copy(args, launch_copy, n_sets, stream, rank, local_rank, world, nbytes):
    """GB/s and step statistics of a copy under the same rotation and batches."""
    batch_ms, bounds, _clk, _last = timed_batches(args, launch_copy, n_sets, stream, rank,
                                                  local_rank, world)
    st = batch_stats(batch_ms, bounds)
    med_s = max_over_ranks(st["median_step_us"] / 1e6, device="cuda" if world > 1 else "cpu")
    return round(replica_throughput(nbytes, 1, world, med_s), 2), st


def copy_baseline(args, launch_rows, launch_torch, n_sets, stream, rank, local_rank, world,
                  nbytes):
    """The copy ceiling: the library's row copy (softmax_rows_copy_ceiling: the same
    bytes at the same pitches, the same 16-byte streaming accesses, no arithmetic),
    with torch's copy_ of the same elements beside it, both under the bench protocol."""
    gbs, st = timed_copy(args, launch_rows, n_sets, stream, rank, local_rank, world, nbytes)
    tgbs, tst = timed_copy(args, launch_torch, n_sets, stream, rank, local_rank, world, nbytes)
    return {"value": gbs, "unit": "GB/s", "median_step_us": st["median_step_us"],
            "mean_step_us": st["mean_step_us"],
            "kind": "softmax_rows_copy_ceiling: the same M x N elements from the input pitch to "
                    "the output pitch with the softmax's 16-byte streaming loads and stores, "
                    "same sets and batches",
            "torch_copy_gbs": tgbs, "torch_copy_median_step_us": tst["median_step_us"]}


def bench_ours(args, w):
    import torch

    import memory_bound_row_rows_gb300 as sr
    from memory_bound_row_rows_gb300 import _build
    rank, local_rank, world = dist_env()
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    lib = sr.load()
    x = w.generate()
    tdt = torch_dtype(w.dtype)

    # Input/output sets: every set's input holds the same matrix.
    set_bytes = (w.M * w.ld_in + w.M * w.ld_out) * w.elem_bytes
    n_sets = rotation_count(set_bytes, args.lane)
    l2 = device_l2_bytes(dev)
    while args.lane == "cold" and l2 and n_sets * set_bytes < 4 * l2:
        n_sets += 1
    x_sets = torch.empty((n_sets, w.M, w.ld_in), dtype=tdt, device=dev)
    x_sets[0].copy_(to_device(x, w.dtype, dev))
    for i in range(1, n_sets):
        x_sets[i].copy_(x_sets[0])
    y_sets = torch.full((n_sets, w.M, w.ld_out), float("nan"), dtype=tdt, device=dev)
    ws, ws_bytes = None, 0
    if args.api == "split":
        ws_bytes = sr.softmax_rows_split_workspace_bytes(x_sets[0], y_sets[0], w.M, w.N, w.ld_in,
                                                         w.ld_out, w.dtype)
        ws = torch.empty(max(16, ws_bytes), dtype=torch.uint8, device=dev)
        split_shape = sr.softmax_rows_split_shape(x_sets[0], y_sets[0], w.M, w.N, w.ld_in,
                                                  w.ld_out, w.dtype)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    plan_used = sr.softmax_rows_plan(x_sets[0], y_sets[0], w.M, w.N, w.ld_in, w.ld_out,
                                     w.dtype) if args.plan == 0 else args.plan
    xp = [x_sets[i].data_ptr() for i in range(n_sets)]
    yp = [y_sets[i].data_ptr() for i in range(n_sets)]

    def launch(i):
        if args.api == "split":
            st = lib.softmax_rows_split(xp[i], yp[i], w.M, w.N, w.ld_in, w.ld_out, w.dtype,
                                        ws.data_ptr(), ws_bytes, sh)
        elif args.api == "masked":
            st = lib.softmax_rows_masked(xp[i], yp[i], w.M, w.N, w.ld_in, w.ld_out, w.dtype,
                                         None, w.causal_period, args.plan, sh)
        else:
            st = lib.softmax_rows_ex(xp[i], yp[i], w.M, w.N, w.ld_in, w.ld_out, w.dtype,
                                     args.plan, sh)
        if st != 0:
            raise RuntimeError("softmax_rows failed: %s" % sr.softmax_rows_strerror(st))

    if args.api == "split":
        plan_used = "split"
    elif args.api == "masked":
        plan_used = "masked-" + sr.PLAN_NAMES.get(plan_used, str(plan_used))
    else:
        plan_used = sr.PLAN_NAMES.get(plan_used, str(plan_used))
    config = workload_config(w, args.lane, world)
    metric = (("cold-L2 softmax GB/s (2*M*N*bytes/time)" if args.lane == "cold"
               else "warm-L2 softmax GB/s (2*M*N*bytes/time)") if args.api != "masked"
              else "cold-L2 masked softmax GB/s ((valid reads + M*N writes)*bytes/time)")

    # 1. Correctness before any timing: one call, sampled rows against the oracle.
    rows = parity_rows(w.M, w.N)
    ref = oracle_rows(w, x, rows)
    launch(0)
    torch.cuda.synchronize()
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
    gate = compare_rows(w, device_rows(y_sets[0], rows), ref, rows)
    if gate["outside_tolerance"]:
        raise ParityFailure({"metric": metric, "error": "parity: output outside the tolerance "
                             "before timing", "config": config, "plan": plan_used,
                             "parity_before_timing": gate})

    # 2-3. Timed steps over the rotating sets.
    batch_ms, bounds, clocks, last = timed_batches(args, launch, n_sets, stream, rank,
                                                   local_rank, world)
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
    kernel = kernel_record(sr)
    stats = batch_stats(batch_ms, bounds)
    med_s = max_over_ranks(stats["median_step_us"] / 1e6, device="cuda" if world > 1 else "cpu")
    mean_s = max_over_ranks(stats["mean_step_us"] / 1e6, device="cuda" if world > 1 else "cpu")

    # 4. The last timed call's output.
    after = compare_rows(w, device_rows(y_sets[last], rows), ref, rows)

    nbytes = algorithmic_bytes(w, args.api)
    copy = None
    if not args.no_copy:
        eb = w.elem_bytes

        def launch_rows(i):
            st = lib.softmax_rows_copy_ceiling(xp[i], yp[i], w.M, w.N * eb, w.ld_in * eb,
                                               w.ld_out * eb, sh)
            if st != 0:
                raise RuntimeError("softmax_rows_copy_ceiling: %s" % sr.softmax_rows_strerror(st))

        def launch_torch(i):
            y_sets[i][:, :w.N].copy_(x_sets[i][:, :w.N])
        copy = copy_baseline(args, launch_rows, launch_torch, n_sets, stream, rank, local_rank,
                             world, w.fused_bytes)
    e2e = None
    if not args.no_e2e:
        del x_sets, y_sets
        torch.cuda.empty_cache()
        e2e = run_e2e(args, w, x, dev, lib, lambda a: to_device(a, w.dtype, "cpu"), tdt)
    if rank != 0:
        return None
    steps = bounds[-1][1]
    value = replica_throughput(nbytes, 1, world, med_s)  # the slowest rank's median step
    peaks = measured_peaks()
    src_hash = _build.source_hash(_build.PLAN_SOURCES.get(plan_used.replace("masked-", "")))
    traffic, rec = recorded_traffic(("split:" if args.api == "split" else "") + w.name, plan_used)
    achieved = nbytes / (stats["median_step_us"] / 1e6) / 1e9
    line = {
        "metric": metric,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": round(med_s * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": synth.DTYPE_NAMES[w.dtype],
        "data": "synthetic: seeded SplitMix64/Box-Muller (seed %d), generated on the host" % w.seed,
        "config": config,
        "plan": plan_used,
        "statistic": "ms_per_step and value use the median step (over batches of consecutive "
                     "launches); mean_step_us is the mean over all timed steps",
        "mean_step_gbs": round(replica_throughput(nbytes, 1, world, mean_s), 2),
        "pct_of_8000_gbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_hbm": round(100 * value / world / peaks["hbm_gbs"], 2),
        "rows_per_s": round(world * w.M / med_s, 1),
        "bytes_per_step": nbytes,
        "dense_equivalent_gbs": round(world * w.fused_bytes / med_s / 1e9, 2),
        **stats,
        "sets": n_sets,
        "gpu_launches": steps,
        "kernel": kernel,
        "clocks": clocks,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": traffic,
                     **dram_rate(traffic, stats["median_step_us"], peaks["hbm_gbs"]),
                     "traffic_note": (rec or {}).get("note") if traffic else
                     "null: no ncu capture recorded for the current kernel sources"},
        "source_hash": src_hash,
        "parity_before_timing": gate,
        "parity": after,
    }
    if args.api == "split":
        # One kernel per call, after a memset of the workspace's counters.
        line["split_shape"] = split_shape
        line["memsets_per_step"] = 1
    if copy is not None:
        copy["ratio"] = round(value / world / (copy["value"] / world), 4)
        line["copy_baseline"] = copy
    if e2e is not None:
        line["e2e"] = e2e
    if world == 1:
        line["cpu_baseline"] = cpu_baseline(w, x, args.cpu_budget)
    if after["outside_tolerance"]:
        line.pop("value")
        line["error"] = "parity: the last timed output is outside the tolerance"
        raise ParityFailure(line)
    return line


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




def pair_config(lane, lane_name: str, world: int) -> dict:
    """The config object both arms print for a row-pair workload."""
    w = lane.w
    set_bytes = 3 * w.M * w.ld * w.elem_bytes
    return {"workload": "%s %s" % (lane.api, w.name), "M": w.M, "N": w.N, "ld": w.ld,
            "l2": l2_protocol(set_bytes, lane_name),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def pair_parity(lane, out, rows) -> dict:
    w = lane.w
    g = device_rows(out, rows)
    r = lane.oracle_rows(rows)
    dec = lambda a: synth.storage_to_float64(np.ascontiguousarray(a[:, :w.N]), w.dtype)
    return {"rows": int(rows.size), "of_rows": w.M,
            "outside_tolerance": lane.outside_gate(dec(g), dec(r), rows), "gate": lane.gate}


def bench_pair(args, lane):
    """One row-pair call per step (softmax_rows_backward_ex or rmsnorm_residual_rows_ex),
    under the softmax lane's protocol: parity first, rotating sets, batched events."""
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
    tdt = torch_dtype(w.dtype)
    set_bytes = 3 * w.M * w.ld * w.elem_bytes
    n_sets = rotation_count(set_bytes, args.lane)
    l2 = device_l2_bytes(dev)
    while args.lane == "cold" and l2 and n_sets * set_bytes < 4 * l2:
        n_sets += 1
    sets = []
    first = [to_device(m, w.dtype, dev) for m in lane.mats]
    vecs = [to_device(v, w.dtype, dev) for v in lane.vecs]
    for i in range(n_sets):
        mats = first if i == 0 else [m.clone() for m in first]
        sets.append((mats, torch.full((w.M, w.ld), float("nan"), dtype=tdt, device=dev)))
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    plan = lane.plan(sr, sets[0][0], vecs, sets[0][1], args.plan)
    if plan < 0:
        raise RuntimeError("plan %d cannot take %s %s" % (args.plan, lane.api, w.name))

    def launch(i):
        mats, out = sets[i]
        st = lane.call(lib, mats, vecs, out, args.plan, sh)
        if st != 0:
            raise RuntimeError("%s failed: %s" % (lane.api, sr.softmax_rows_strerror(st)))

    pname = "%s-%s" % (lane.api, sr.PLAN_NAMES[plan])
    lanename = "cold-L2" if args.lane == "cold" else "warm-L2"
    metric = "%s %s GB/s (%s/time)" % (lanename, lane.label, lane.model)
    config = pair_config(lane, args.lane, world)
    rows = np.unique(np.concatenate([np.linspace(0, w.M - 1, 64).astype(np.int64), [w.M - 1]]))
    launch(0)
    torch.cuda.synchronize()
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
    gate = pair_parity(lane, sets[0][1], rows)
    if gate["outside_tolerance"]:
        raise ParityFailure({"metric": metric, "error": "parity: output outside the gate "
                             "before timing", "config": config, "plan": pname,
                             "parity_before_timing": gate})

    batch_ms, bounds, clocks, last = timed_batches(args, launch, n_sets, stream, rank,
                                                   local_rank, world)
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
    kernel = kernel_record(sr)
    stats = batch_stats(batch_ms, bounds)
    med_s = max_over_ranks(stats["median_step_us"] / 1e6, device="cuda" if world > 1 else "cpu")
    mean_s = max_over_ranks(stats["mean_step_us"] / 1e6, device="cuda" if world > 1 else "cpu")
    after = pair_parity(lane, sets[last][1], rows)

    copy = None
    if not args.no_copy:
        eb = w.elem_bytes

        def launch_rows(i):
            (a, b), out = sets[i]
            st = lib.softmax_rows_copy_ceiling2(a.data_ptr(), b.data_ptr(), out.data_ptr(), w.M,
                                                w.N * eb, w.ld * eb, w.ld * eb, w.ld * eb, sh)
            if st != 0:
                raise RuntimeError("softmax_rows_copy_ceiling2: %s" % sr.softmax_rows_strerror(st))

        def launch_torch(i):
            (a, b), out = sets[i]
            torch.add(a[:, :w.N], b[:, :w.N], out=out[:, :w.N])
        copy = copy_baseline(args, launch_rows, launch_torch, n_sets, stream, rank, local_rank,
                             world, 3 * w.M * w.N * w.elem_bytes)
        copy["kind"] = ("softmax_rows_copy_ceiling2: out = a XOR b over the same two input and "
                        "one output matrices (3*M*N*bytes; the weight vector aside), with the "
                        "same 16-byte streaming loads and stores, same sets and batches; "
                        "torch_copy_* is torch.add of the same matrices")
    e2e = None
    if not args.no_e2e:
        # Host buffers: the pinned inputs copied in, the call, the output copied back,
        # pinned from a thread on the GPU's NUMA node (as in run_e2e).
        cpus, numa = gpu_numa_cpus(dev)
        saved = os.sched_getaffinity(0)
        try:
            if cpus:
                os.sched_setaffinity(0, cpus)
            pins = [to_device(m, w.dtype, "cpu").pin_memory() for m in lane.mats + lane.vecs]
            out_pin = torch.empty((w.M, w.ld), dtype=tdt).pin_memory()
            out_pin.zero_()
        finally:
            os.sched_setaffinity(0, saved)
        mats0, out = sets[0]
        targets = mats0 + vecs

        def e2e_step():
            for d, h in zip(targets, pins):
                d.copy_(h, non_blocking=True)
            launch(0)
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
               "d2h_bytes_per_step": w.M * w.ld * w.elem_bytes,
               "ms_per_step": round(sec * 1e3, 4), "steps": k,
               "path": "pinned host inputs -> device (copies), %s call, output -> pinned host, "
                       "in order on one stream" % lane.api,
               "host_buffers": numa}
    if rank != 0:
        return None
    steps = bounds[-1][1]
    value = replica_throughput(w.fused_bytes, 1, world, med_s)  # the slowest rank's median step
    achieved = w.fused_bytes / (stats["median_step_us"] / 1e6) / 1e9
    peaks = measured_peaks()
    traffic, rec = recorded_traffic("%s:%s" % (lane.api, w.name), lane.api)
    line = {
        "metric": metric,
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(med_s * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": synth.DTYPE_NAMES[w.dtype], "data": lane.data,
        "config": config,
        "plan": pname,
        "statistic": "ms_per_step and value use the median step (over batches of consecutive "
                     "launches); mean_step_us is the mean over all timed steps",
        "mean_step_gbs": round(replica_throughput(w.fused_bytes, 1, world, mean_s), 2),
        "pct_of_8000_gbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_hbm": round(100 * value / world / peaks["hbm_gbs"], 2),
        "bytes_per_step": w.fused_bytes,
        **stats,
        "sets": n_sets,
        "gpu_launches": steps,
        "kernel": kernel,
        "clocks": clocks,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": traffic,
                     **dram_rate(traffic, stats["median_step_us"], peaks["hbm_gbs"]),
                     "traffic_note": (rec or {}).get("note") if traffic else
                     "null: no ncu capture recorded for the current kernel sources"},
        "source_hash": _build.source_hash(_build.PLAN_SOURCES[lane.api]),
        "parity_before_timing": gate,
        "parity": after,
    }
    if copy is not None:
        copy["ratio"] = round((3 * w.M * w.N * w.elem_bytes / (stats["median_step_us"] / 1e6) / 1e9)
                              / (copy["value"] / world), 4)
        line["copy_baseline"] = copy
    if e2e is not None:
        line["e2e"] = e2e
    if world == 1:
        line["cpu_baseline"] = pair_cpu_baseline(lane, args.cpu_budget)
    if after["outside_tolerance"]:
        line.pop("value")
        line["error"] = "parity: the last timed output is outside the gate"
        raise ParityFailure(line)
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
    med = float(np.median(times))
    value = w.fused_bytes / med / 1e9
    return {
        "impl": "reference",
        "metric": "cold-L2 softmax GB/s (2*M*N*bytes/time)",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": len(times),
        "warmup": args.warmup, "ms_per_step": round(1e3 * med, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": synth.DTYPE_NAMES[w.dtype],
        "data": "synthetic: seeded SplitMix64/Box-Muller (seed %d), generated on the host" % w.seed,
        "config": workload_config(w, args.lane, world),
        "statistic": "ms_per_step and value use the median step; mean_step_us is the mean",
        "mean_step_us": round(1e6 * sum(times) / len(times), 1),
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
    med = float(np.median(times))
    value = per_row * rows.size / med / 1e9
    sample = "first %d of %d rows of %s per step, FP64 C oracle's %s, 1 thread" % (
        rows.size, w.M, w.name, lane.label)
    return {
        "impl": "reference",
        "metric": "cold-L2 %s GB/s (%s/time)" % (lane.label, lane.model),
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": len(times),
        "warmup": args.warmup, "ms_per_step": round(1e3 * med, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": synth.DTYPE_NAMES[w.dtype], "data": lane.data,
        "config": pair_config(lane, args.lane, world),
        "statistic": "ms_per_step and value use the median step",
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
    failed = False
    for name in names:
        w = catalog[name]
        if args.rows:
            w = w.with_rows(min(args.rows, w.M))
        try:
            if args.impl == "reference" and args.api in LANES:
                line = bench_reference_pair(args, LANES[args.api](w))
            elif args.impl == "reference":
                line = bench_reference(args, w)
            elif args.api in LANES:
                line = bench_pair(args, LANES[args.api](w))
            else:
                line = bench_ours(args, w)
        except ParityFailure as exc:
            line, failed = exc.line, True
            if dist_env()[0] != 0:
                line = None
        if line is not None:
            print(json.dumps(line), flush=True)
    if args.impl == "ours":
        import torch
        if torch.distributed.is_initialized():
            torch.distributed.destroy_process_group()
    return 1 if failed else 0


if __name__ == "__main__":
    sys.exit(main())
