#!/usr/bin/env python
"""Benchmark of the fused RMSNorm forward + backward on GB300.

One step = one forward (rms_norm_fwd) and one backward (rms_norm_bwd, which
includes the fixed-order weight-gradient reduction) over one batch of the
workload, through the C ABI.  Default workload: a bf16 activation of 16384
rows x hidden 8192, eps 1e-5, round-once store, inputs drawn once (seeded)
and resident in HBM; ``--workload`` picks another (the round-twice store on
the same shape, the Llama-shaped 4096 x 4096, the fp16 width sweep, ...).

Timing.  The batch is copied several times in HBM (at least six L2 sizes
of data in all) and the steps cycle through the copies, the backward of a
step reading the copy whose forward ran half a cycle earlier, so every
kernel reads inputs that the other copies' traffic has evicted from L2.
The timed steps are captured, as the C-ABI calls they are, in one CUDA
graph, replayed once between CUDA events with a barrier and a device
synchronisation on both sides.  The forward and the backward are also timed
alone (graphs of back-to-back calls) for the per-kernel roofline, and as
isolated calls after an L2 flush.

Printed (rank 0, one JSON line): achieved GB/s of algorithmic bytes,
microseconds per call, the roofline of the backward and of the forward, an
end-to-end number through the public API with host buffers, the float64
oracle timed on the host as a baseline, and the SM clocks sampled while the
timed graph ran.

``--workload ln_...`` runs the LayerNorm entry points the same way (one
step = layer_norm_fwd + layer_norm_bwd).

``--impl reference`` times the oracle instead (rank 0 only, on the host
cores, on a bounded sample of the same workload).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
Under torchrun every rank runs the workload on its own GPU (weak scaling:
one batch per rank, no collective on the data path); the time is the
maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import re
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "RMSNorm fwd+bwd achieved HBM GB/s and % of GB300 peak; µs per call"
METRIC_LN = "LayerNorm fwd+bwd achieved HBM GB/s and % of GB300 peak; µs per call"
METRIC_SM = "Softmax (last dim) fwd+bwd achieved HBM GB/s and % of GB300 peak; µs per call"
METRIC_GN = "GroupNorm fwd+bwd achieved HBM GB/s and % of GB300 peak; µs per call"


def metric_for(w) -> str:
    return {"ln": METRIC_LN, "softmax": METRIC_SM, "gn": METRIC_GN}.get(w.kind, METRIC)
DEFAULT_WORKLOAD = "large_bf16_16384x8192_once"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
# Rows per weight-gradient block of the data-parallel exchange (a chunk is
# 32 blocks): the largest of these whose chunk divides a rank's rows.
DP_BLOCK_ROWS = (16, 8, 4, 2, 1)
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, world: int, device=None) -> float:
    """Maximum of ``value`` over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def shard_rows(rows: int, rank: int, world: int):
    """Contiguous slab of rows for ``rank`` (used when one batch is split)."""
    lo = rows * rank // world
    hi = rows * (rank + 1) // world
    return lo, hi


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampled every 50 ms in the background."""

    def __init__(self, gpu_id: str):
        self.t0 = time.time()
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        self.window = (0.0, 0.0)

    def mark(self, start: float, end: float):
        self.window = (start, end)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return summarize_clocks(out.splitlines(), self.window)


def summarize_clocks(lines, window):
    import datetime
    rows = []
    for ln in lines:
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 9:
            continue
        try:
            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            sm, smax = float(parts[1]), float(parts[2])
        except ValueError:
            continue
        rows.append((ts, sm, smax, parts[3], parts[5:9]))
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    inside = [r for r in rows if window[0] <= r[0] <= window[1]]
    use = inside if inside else rows
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in use for i, v in enumerate(r[4]) if v == "Active"})
    return {
        "sm_mhz": statistics.median(r[1] for r in use),
        "sm_max_mhz": max(r[2] for r in use),
        "reasons": reasons,
        "samples": len(use),
        "samples_in_timed_region": len(inside),
    }


class NvmlPoller:
    """SM clock and clock-event reasons read through NVML (the driver's
    libnvidia-ml, read-only queries) by a background thread about every
    0.2 ms, so that even a timed region of a few milliseconds holds
    samples.  ``window(t0, t1)`` summarises the samples taken between two
    time.perf_counter() readings.  Inactive (no samples) when NVML cannot be
    loaded."""

    # clock-event reason bits of nvml.h
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str):
        import ctypes
        import threading
        self.samples = []
        self._stop = threading.Event()
        self._thread = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
                return
            reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
        except (OSError, AttributeError):
            return
        self._nv, self._h, self._reasons_fn = nv, h, reasons_fn
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()

    def _run(self):
        import ctypes
        mhz, rs = ctypes.c_uint(0), ctypes.c_ulonglong(0)
        while not self._stop.is_set():
            t = time.perf_counter()
            if self._nv.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(mhz)) == 0:
                ok = self._reasons_fn(self._h, ctypes.byref(rs)) == 0
                self.samples.append((t, mhz.value, rs.value if ok else 0))
            time.sleep(0.0002)

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=2)

    def window(self, t0: float, t1: float):
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        if not inside:
            return None
        bits = 0
        for x in inside:
            bits |= x[2]
        return {"sm_mhz": statistics.median(x[1] for x in inside),
                "reasons": sorted(v for k, v in self.REASONS.items() if bits & k),
                "samples": len(inside)}


def paired_variant(name: str):
    """The other cast mode of a workload that exists in both (timed in the
    same run as the requested one), or None."""
    import workloads as W
    table = W.all_workloads()
    for a, b in (("_once", "_twice"), ("_twice", "_once")):
        if name.endswith(a) and name[:-len(a)] + b in table:
            return name[:-len(a)] + b
    return None


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def measured_peak_gbs():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


_ORACLE_INPUTS = {}


def workload_by_name(name: str):
    """RMSNorm workloads, the LayerNorm ones (names starting ``ln_``), the
    FP8-output ones (names ending ``_fp8``), the softmax ones (names
    starting ``softmax_``) and the GroupNorm ones (names starting ``gn_``)."""
    import workloads as W
    table = dict(W.all_workloads())
    table.update(W.layer_norm_workloads())
    table.update(W.fp8_workloads())
    table.update(W.softmax_workloads())
    table.update(W.group_norm_workloads())
    if name not in table:
        raise SystemExit(f"unknown workload {name!r}; known: {', '.join(sorted(table))}")
    return table[name]


def time_oracle(w, rows: int, threads: int = 1):
    """Seconds for one oracle forward + backward over ``rows`` rows of ``w``
    (inputs drawn once per row count, outside the timing), the rows split
    into ``threads`` contiguous ranges run on as many host threads; the
    per-range parameter gradients are summed in range order."""
    import workloads as W
    from oracle import fp8 as of8
    from oracle import group_norm as ogn
    from oracle import layer_norm as oln
    from oracle import rms_norm as orm
    from oracle import softmax as osm
    from oracle import threads as OT
    ws = w.with_(rows=rows)
    if (ws.name, rows) not in _ORACLE_INPUTS:
        _ORACLE_INPUTS.clear()
        inp = W.make_inputs(ws)
        _ORACLE_INPUTS[(ws.name, rows)] = tuple(
            W.as_float64(inp[k]) if k in inp else None for k in ("x", "gamma", "dy", "beta"))
    xd, gd, dyd, bd = _ORACLE_INPUTS[(ws.name, rows)]

    def run(sl):
        xs, dys = xd[sl], dyd[sl]
        if ws.kind == "softmax":
            y = osm.forward(xs, ws.dtype)
            osm.backward(dys, y, ws.dtype)
            return None
        if ws.kind == "gn":
            _, mean, rstd = ogn.forward(xs, gd, bd, ws.groups, ws.eps, ws.dtype)
            return ogn.backward(dys, xs, gd, mean, rstd, ws.groups, ws.dtype)[1]
        if ws.kind == "ln":
            _, mean, rstd = oln.forward(xs, gd, bd, ws.eps, ws.dtype)
            return oln.backward(dys, xs, gd, mean, rstd, ws.dtype)[1]
        if ws.out_fmt == "e4m3":
            _, rstd = of8.forward_fp8(xs, gd, ws.eps, ws.offset, ws.scale)
        else:
            _, rstd = orm.forward(xs, gd, ws.eps, ws.offset, ws.dtype, ws.cast_mode)
        return orm.backward(dys, xs, gd, rstd, ws.offset, ws.dtype)[1]

    t = time.perf_counter()
    parts = OT.map_rows(run, rows, threads)
    if parts[0] is not None:
        OT.sum_in_order(parts)
    return time.perf_counter() - t, ws.step_bytes()


def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_baseline(w, name: str, budget_s: float = 10.0):
    """The float64 oracle timed on the host on a bounded sample of the
    workload (its first rows, about 16 M elements, a different seeded draw
    of the same distributions): passes on one thread, then on every host
    core, each repeated until about ``budget_s`` seconds of host time (at
    least one pass).  GB/s of the sample's algorithmic bytes."""
    rows = min(w.rows, max(16, (1 << 24) // max(1, w.hidden)))
    out = {}
    for threads in sorted({1, host_threads()}):
        secs, nbytes, passes = 0.0, 0, 0
        while (secs < budget_s and passes < 50) or passes == 0:
            s_, b_ = time_oracle(w, rows, threads)
            secs += s_
            nbytes += b_
            passes += 1
        out[threads] = (nbytes / secs / 1e9, passes, secs)
    cores = max(out)
    v1, p1, s1 = out[1]
    vn, pn, sn = out[cores]
    return {"value": round(vn, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": (f"{name}: float64 forward+backward (numpy) over {rows} of {w.rows} rows "
                       f"per pass: {pn} passes on {cores} threads, the rows split in {cores} "
                       f"contiguous ranges ({sn:.1f} s); {p1} passes on 1 thread ({s1:.1f} s)"),
            "single_thread": {"value": round(v1, 4), "unit": "GB/s", "cores": 1},
            "nproc": os.cpu_count()}


def run_ours(args, rank, world, local):
    import math

    import torch

    import bwd_rms_norm_gb300 as L
    import workloads as W

    if not os.path.exists(L.LIB_PATH):
        from bwd_rms_norm_gb300 import build
        build.build()
    L.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    stream = torch.cuda.current_stream(dev)

    w = workload_by_name(args.workload)
    if args.rows:
        w = w.with_(rows=args.rows)
    ln = w.kind == "ln"
    sm = w.kind == "softmax"
    gn = w.kind == "gn"
    f8 = w.out_fmt == "e4m3"
    inp = W.make_inputs(w)
    nstat = w.rows * (w.groups if gn else 1)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or (126 << 20))

    # Several copies of the batch, cycled, so that every step finds its
    # inputs evicted from L2 by the other copies' traffic (at least six L2
    # sizes of data in the cycle).
    set_bytes = 4 * w.rows * w.hidden * w.elem_bytes + 8 * nstat
    nsets = max(2, min(8, math.ceil(6 * l2 / set_bytes)))
    sets = []
    for _ in range(nsets):
        x = inp["x"].to(dev)
        y = (torch.empty(x.shape, dtype=L.FP8_DTYPE, device=dev) if f8 else torch.empty_like(x))
        sets.append({"x": x, "dy": inp["dy"].to(dev), "y": y,
                     "dx": torch.empty_like(x),
                     "rstd": torch.empty(nstat, dtype=torch.float32, device=dev),
                     "mean": torch.empty(nstat, dtype=torch.float32, device=dev)})
    g = inp["gamma"].to(dev)
    beta = inp["beta"].to(dev) if "beta" in inp else None
    scale = torch.tensor([w.scale], dtype=torch.float32, device=dev)
    dw = torch.empty(w.param_len, dtype=torch.float32, device=dev)
    db = torch.empty(w.param_len, dtype=torch.float32, device=dev)
    if gn:
        ws_bytes = L.group_norm_bwd_workspace_size(w.rows, w.channels, w.spatial, w.groups,
                                                   g.dtype)
    else:
        ws_fn = L.layer_norm_bwd_workspace_size if ln else L.rms_norm_bwd_workspace_size
        ws_bytes = 0 if sm else ws_fn(w.rows, w.hidden, g.dtype)
    ws = torch.empty(max(16, ws_bytes), dtype=torch.uint8, device=dev)
    half = nsets // 2

    # Data parallel (more than one rank, or --dp-exchange): rank k's batch is
    # slab k of a global batch of world x rows rows, cut by the library's
    # rms_norm_rank_rows into whole chunks of 32 blocks; the backward leaves
    # its slab's weight-gradient chunk sums, the ranks all-gather them and
    # every rank adds them in chunk order -- the weight gradient of the
    # global batch, the same bits for any number of ranks.
    dp = (world > 1 or args.dp_exchange) and not (ln or sm or gn)
    dp_info = None
    if dp:
        brows = next((b for b in DP_BLOCK_ROWS if w.rows % (32 * b) == 0), None)
        if brows is None:
            raise SystemExit(f"data-parallel exchange needs rows divisible by 32 "
                             f"(a chunk of 32 one-row blocks), not {w.rows}")
        lo, hi = L.rms_norm_rank_rows(w.rows * world, brows, world, rank)
        assert (lo, hi) == (rank * w.rows, (rank + 1) * w.rows), (lo, hi)
        nch = L.rms_norm_dw_chunk_count(w.rows, brows)
        chunks = torch.empty(nch, w.hidden, dtype=torch.float32, device=dev)
        gathered = (torch.empty(world * nch, w.hidden, dtype=torch.float32, device=dev)
                    if world > 1 else chunks)
        ws = torch.empty(max(16, L.rms_norm_bwd_blocked_workspace_size(w.rows, w.hidden, brows)),
                         dtype=torch.uint8, device=dev)
        import torch.distributed as dist
        dp_info = {"block_rows": brows, "chunks_per_rank": nch, "global_rows": w.rows * world,
                   "rank_rows": [lo, hi],
                   "exchange": (f"all_gather of {nch} x {w.hidden} fp32 chunk sums per rank"
                                if world > 1 else "none (one rank)")}

    def fwd(k):
        S = sets[k]
        if sm:
            L.softmax_fwd(S["x"], y=S["y"])
        elif gn:
            L.group_norm_fwd(S["x"], g, beta, w.groups, w.eps, y=S["y"], mean=S["mean"],
                             rstd=S["rstd"])
        elif ln:
            L.layer_norm_fwd(S["x"], g, beta, w.eps, y=S["y"], mean=S["mean"], rstd=S["rstd"])
        elif f8:
            L.rms_norm_fwd_fp8(S["x"], g, scale, w.eps, w.offset, y=S["y"], rstd=S["rstd"])
        else:
            L.rms_norm_fwd(S["x"], g, w.eps, w.offset, w.cast_mode, y=S["y"], rstd=S["rstd"])

    def bwd(k):
        S = sets[k]
        if sm:
            L.softmax_bwd(S["dy"], S["y"], dx=S["dx"])
        elif gn:
            L.group_norm_bwd(S["dy"], S["x"], g, S["mean"], S["rstd"], w.groups, dx=S["dx"],
                             dgamma=dw, dbeta=db, workspace=ws)
        elif ln:
            L.layer_norm_bwd(S["dy"], S["x"], g, S["mean"], S["rstd"], dx=S["dx"], dgamma=dw,
                             dbeta=db, workspace=ws)
        elif dp:
            L.rms_norm_bwd_blocked(S["dy"], S["x"], g, S["rstd"], dp_info["block_rows"],
                                   w.offset, dx=S["dx"], chunk_sums=chunks, workspace=ws)
            if world > 1:
                dist.all_gather_into_tensor(gathered, chunks)
            L.rms_norm_dw_sum(gathered, dw=dw)
        else:
            L.rms_norm_bwd(S["dy"], S["x"], g, S["rstd"], w.offset, dx=S["dx"], dw=dw,
                           workspace=ws)

    def step(i):
        # the backward works on a copy whose forward ran `half` steps ago
        fwd(i % nsets)
        bwd((i + half) % nsets)

    if args.profile:
        # eager steps only, for a profiler: warm-up steps, then the profiled
        # ones, no graphs, no timing, nothing else launched
        for i in range(args.warmup + args.steps):
            step(i)
            if i == args.warmup - 1:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        kernels = {}
        fwd(0)
        kernels["fwd"] = L.last_kernels()
        bwd(0)
        kernels["bwd"] = L.last_kernels()
        torch.cuda.synchronize()
        if rank == 0:
            print(json.dumps({"profile": args.workload, "rows": w.rows, "hidden": w.hidden,
                              "warmup_steps": args.warmup, "steps": args.steps,
                              "sets": nsets, "kernels": kernels}), flush=True)
        return

    # eager warm-up: every kernel configuration is set up before capture
    for i in range(max(args.warmup, nsets)):
        step(i)
    torch.cuda.synchronize()
    # kernels one step launches, as the library counts them
    fwd(0)
    launches_per_step = L.last_launch_count()
    bwd(0)
    # data parallel: the last call is rms_norm_dw_sum; the blocked backward
    # before it launched two kernels
    launches_per_step += L.last_launch_count() + (2 if dp else 0)
    torch.cuda.synchronize()

    class Eager:
        """Stands in for a CUDA graph where the step holds a collective:
        replay() launches the same calls eagerly."""

        def __init__(self, fn, n):
            self.fn, self.n = fn, n

        def replay(self):
            for i in range(self.n):
                self.fn(i)

    def capture(fn, n):
        if dp and world > 1:
            return Eager(fn, n)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(n):
                fn(i)
        return graph

    g_steps = capture(step, args.steps)           # exactly the timed steps
    reps = 8 * nsets
    g_fwd = capture(lambda i: fwd(i % nsets), reps)
    g_bwd = capture(lambda i: bwd(i % nsets), reps)
    torch.cuda.synchronize()

    def timed(graph, times):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(times):
            graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    # graph warm-up, then per-kernel averages over back-to-back launches
    for _ in range(max(3, args.warmup // 4)):
        g_fwd.replay()
        g_bwd.replay()
    fwd_us = min(timed(g_fwd, 4) for _ in range(3)) * 1e3 / (4 * reps)
    bwd_us = min(timed(g_bwd, 4) for _ in range(3)) * 1e3 / (4 * reps)

    uuid = str(getattr(props, "uuid", "")) or str(local)
    gpu_id = ("GPU-" + uuid) if uuid and not uuid.isdigit() else uuid
    sampler = ClockSampler(gpu_id)
    poller = NvmlPoller(gpu_id)
    t_soak = time.time()
    while time.time() - t_soak < 0.6:      # clocks settle on the same work
        g_fwd.replay()
        g_bwd.replay()
        torch.cuda.synchronize()

    barrier(world)
    torch.cuda.synchronize()
    t_start = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    e0.record(stream)
    g_steps.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.perf_counter()
    wall = wall1 - wall0
    barrier(world)
    t_end = time.time()
    sampler.mark(t_start, t_end)
    in_region = poller.window(wall0, wall1)
    step_ms = e0.elapsed_time(e1)
    step_ms = reduce_max(step_ms, world, dev)
    # keep sampling a little after the timed region so that short regions
    # still get a sample taken under the same load
    t_tail = time.time()
    while time.time() - t_tail < 0.3:
        g_steps.replay()
        torch.cuda.synchronize()
    clocks = sampler.stop()
    poller.stop()
    if in_region is not None:
        # NVML samples taken inside the timed replay decide the clock and the
        # reasons; nvidia-smi's (around it) stay beside them
        clocks = {"sm_mhz": in_region["sm_mhz"], "sm_max_mhz": clocks.get("sm_max_mhz"),
                  "reasons": sorted(set(in_region["reasons"]) | set(clocks.get("reasons", []))),
                  "samples_in_timed_region": in_region["samples"],
                  "source": "NVML polled about every 0.2 ms inside the timed replay; "
                            "nvidia-smi every 50 ms around it",
                  "nvidia_smi": clocks}

    ms_per_step = step_ms / args.steps
    total_bytes = w.step_bytes() * args.steps * world
    value = total_bytes / (step_ms * 1e-3) / 1e9

    peak, peak_src = measured_peak_gbs()

    # The same workload with the other cast mode, on the same device buffers
    # (same seeded inputs): its own step graph and forward graph.  The cast
    # mode does not enter the backward, which is the one timed above.
    variants = []
    vname = None
    if not (args.no_variant or ln or sm or gn or f8):
        vname = paired_variant(args.workload)
    if vname is not None:
        wv = workload_by_name(vname)
        if args.rows:
            wv = wv.with_(rows=args.rows)

        def fwd_v(k):
            S = sets[k]
            L.rms_norm_fwd(S["x"], g, wv.eps, wv.offset, wv.cast_mode, y=S["y"], rstd=S["rstd"])

        def step_v(i):
            fwd_v(i % nsets)
            bwd((i + half) % nsets)

        for i in range(nsets):
            step_v(i)
        torch.cuda.synchronize()
        gv_steps = capture(step_v, args.steps)
        gv_fwd = capture(lambda i: fwd_v(i % nsets), reps)
        torch.cuda.synchronize()
        for _ in range(3):
            gv_fwd.replay()
            g_bwd.replay()
        fwd_us_v = min(timed(gv_fwd, 4) for _ in range(3)) * 1e3 / (4 * reps)
        gv_steps.replay()
        torch.cuda.synchronize()
        barrier(world)
        ms_v = reduce_max(timed(gv_steps, 1), world, dev)
        value_v = wv.step_bytes() * args.steps * world / (ms_v * 1e-3) / 1e9
        fwd_ach_v = wv.fwd_bytes() / (fwd_us_v * 1e-6) / 1e9
        variants.append({
            "workload": vname, "cast_mode": wv.cast_mode, "value": round(value_v, 1),
            "unit": "GB/s", "ms_per_step": round(ms_v / args.steps, 6),
            "pct_of_hbm_peak": round(100.0 * value_v / world / peak, 2),
            "fwd_us": round(fwd_us_v, 3), "roofline_fwd_frac": round(fwd_ach_v / peak, 4),
            "bwd_us": round(bwd_us, 3),
            "timing": ("one CUDA-graph replay of exactly `steps` steps of this cast mode, "
                       "CUDA events; the backward is the same call as the headline's"),
        })
    fwd_ach = w.fwd_bytes() / (fwd_us * 1e-6) / 1e9
    bwd_ach = w.bwd_bytes() / (bwd_us * 1e-6) / 1e9
    traffic = load_traffic(args.workload)
    if dp_info is not None:
        # the capture covers rms_norm_bwd, not the fixed-block backward
        traffic = {k: v for k, v in traffic.items() if k != "bwd"}
    iso = isolated_calls(fwd, bwd, nsets, dev, l2)

    # end to end through the public API: pinned host inputs in, results out
    e2e = run_e2e(L, w, inp, dev, args.e2e_steps, beta is not None)
    e2e["value"] = reduce_max_rate(e2e["value"], world, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(w, args.workload)

    op = "layer_norm" if ln else "softmax" if sm else "group_norm" if gn else "rms_norm"
    fwd_name = f"{op}_fwd" + ("_fp8" if f8 else "")
    line = {
        "metric": metric_for(w),
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded, see workloads/)",
        "config": {
            "workload": args.workload + (f" (rows overridden to {w.rows})" if args.rows else ""),
            "rows": w.rows, "hidden": w.hidden,
            **({"arith": "fp32 exp/sum/dot, one rounding at each store"} if sm else
               {"eps": w.eps, "stats": "fp32", "rstd": "fp32", "dw": "fp32"}),
            **({"bias": beta is not None, "mean": "fp32", "dbeta": "fp32"} if ln or gn else {}),
            **({"samples": w.rows, "channels": w.channels, "spatial": w.spatial,
                "groups": w.groups} if gn else {}),
            **({"offset": w.offset, "cast_mode": w.cast_mode} if not (ln or sm or gn) else {}),
            **({"y": "fp8 e4m3 (saturating)", "scale": w.scale} if f8 else {}),
            "global_batch_rows": w.rows * world,
            "parallelism": (f"data parallel x{world}: one slab of {w.rows} rows per rank of a "
                            f"global batch of {w.rows * world} rows; weight gradient over the "
                            f"global batch from all-gathered chunk sums" if dp else
                            f"replica x{world} (one batch per rank)"),
            **({"dp": dp_info} if dp else {}),
            "l2": (f"inputs larger than L2: {nsets} copies of the batch "
                   f"({nsets * set_bytes / 2**20:.0f} MiB) cycled; each step's backward "
                   f"reads the copy whose forward ran {half} steps earlier"),
            "timing": ("CUDA events around one CUDA-graph replay of exactly `steps` "
                       "forward+backward steps (C-ABI calls captured in order)"
                       if not (dp and world > 1) else
                       "CUDA events around exactly `steps` forward+backward steps launched "
                       "eagerly (the step holds an NCCL all_gather), max over ranks"),
            "algorithmic_bytes_per_step": w.step_bytes(),
        },
        "fwd_us": round(fwd_us, 3),
        "bwd_us": round(bwd_us, 3),
        "pct_of_hbm_peak": round(100.0 * value / world / peak, 2),
        "peak_source": f"{peak_src} HBM {peak} GB/s",
        "roofline": {
            "kernel": f"{op}_bwd (row kernel + fixed-order column sums)",
            "bound": "hbm", "achieved": round(bwd_ach, 1), "peak": peak, "unit": "GB/s",
            "frac": round(bwd_ach / peak, 4),
            "traffic": traffic.get("bwd"),
            "algorithmic_bytes": w.bwd_bytes(),
            "timing": f"{4 * reps} back-to-back backward calls in a CUDA graph, best of 3",
        },
        "roofline_fwd": {
            "kernel": fwd_name, "bound": "hbm", "achieved": round(fwd_ach, 1),
            "peak": peak, "unit": "GB/s", "frac": round(fwd_ach / peak, 4),
            "traffic": traffic.get("fwd"), "algorithmic_bytes": w.fwd_bytes(),
        },
        "isolated_call": iso,
        "e2e": e2e,
        "variants": variants,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 4),
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)


def isolated_calls(fwd, bwd, nsets, dev, l2, n=200):
    """Microseconds of single calls, each preceded by a write of twice the L2
    size and a short device-side sleep (so the host is ahead), timed with
    CUDA events around the call: the latency of a call made alone."""
    import torch
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(2 * l2 // 4, dtype=torch.int32, device=dev)
    out = {}
    for name, fn in (("fwd_us", fwd), ("bwd_us", bwd)):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for i in range(n):
            flush.fill_(i)
            torch.cuda._sleep(200_000)
            ev[i][0].record(stream)
            fn(i % nsets)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        out[name] = round(statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3, 3)
    out["timing"] = "median of 200 calls, L2 flushed (write of 2x L2) before each"
    return out


def reduce_max_rate(rate: float, world: int, dev) -> float:
    """Aggregate rate over ranks: world / (max over ranks of 1/rate)."""
    if world <= 1:
        return rate
    t = reduce_max(1.0 / rate, world, dev)
    return world / t


def run_e2e(L, w, inp, dev, steps: int, with_beta: bool = False):
    """GB/s of algorithmic bytes when every step copies the inputs from
    pinned host memory, runs forward and backward through the Python API and
    copies every result back to pinned host memory.  Steps are pipelined the
    way an input pipeline would run them: copies in, compute and copies out
    on three streams over two device buffer sets, so that one step's upload,
    another's kernels and a third's download overlap (both directions of the
    host link at once)."""
    import torch
    ln = w.kind == "ln"
    sm = w.kind == "softmax"
    gn = w.kind == "gn"
    f8 = w.out_fmt == "e4m3"
    names = ("x", "dy") if sm else ("x", "gamma", "dy") + (("beta",) if (ln or gn) and with_beta
                                                           else ())
    host_in = {k: inp[k].pin_memory() for k in names}
    nstat = w.rows * (w.groups if gn else 1)
    nstats = 0 if sm else 2 if ln or gn else 1
    ngrads = 0 if sm else 2 if (ln or gn) and with_beta else 1
    hy = (torch.empty(host_in["x"].shape, dtype=torch.uint8) if f8
          else torch.empty_like(host_in["x"])).pin_memory()
    hdx = torch.empty_like(host_in["x"]).pin_memory()
    hstats = [torch.empty(nstat, dtype=torch.float32).pin_memory() for _ in range(nstats)]
    hgrads = [torch.empty(w.param_len, dtype=torch.float32).pin_memory() for _ in range(ngrads)]
    scale = torch.tensor([w.scale], dtype=torch.float32, device=dev)
    if gn:
        ws_bytes = L.group_norm_bwd_workspace_size(w.rows, w.channels, w.spatial, w.groups,
                                                   host_in["x"].dtype)
    else:
        ws_fn = L.layer_norm_bwd_workspace_size if ln else L.rms_norm_bwd_workspace_size
        ws_bytes = 0 if sm else ws_fn(w.rows, w.hidden, host_in["x"].dtype)
    x_shape = host_in["x"].shape

    def buffers():
        d = {k: torch.empty_like(v, device=dev) for k, v in host_in.items()}
        d["y"] = torch.empty(x_shape, dtype=L.FP8_DTYPE if f8 else host_in["x"].dtype,
                             device=dev)
        d["dx"] = torch.empty(x_shape, dtype=host_in["x"].dtype, device=dev)
        d["stats"] = [torch.empty(nstat, dtype=torch.float32, device=dev) for _ in range(nstats)]
        d["grads"] = [torch.empty(w.param_len, dtype=torch.float32, device=dev)
                      for _ in range(ngrads)]
        d["ws"] = torch.empty(max(16, ws_bytes), dtype=torch.uint8, device=dev)
        return d

    sets = [buffers(), buffers()]
    s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()
    loaded = [ev(), ev()]     # inputs of the set on the device
    computed = [ev(), ev()]   # the set's kernels done (inputs free, outputs ready)
    drained = [ev(), ev()]    # the set's outputs copied out
    for e in computed + drained:
        e.record(s_run)

    def compute(d):
        x, g, dy, y, dx = d["x"], d.get("gamma"), d["dy"], d["y"], d["dx"]
        st, gr = d["stats"], d["grads"]
        if sm:
            L.softmax_fwd(x, y=y)
            L.softmax_bwd(dy, y, dx=dx)
        elif gn:
            L.group_norm_fwd(x, g, d.get("beta"), w.groups, w.eps, y=y, mean=st[0], rstd=st[1])
            L.group_norm_bwd(dy, x, g, st[0], st[1], w.groups, dx=dx, dgamma=gr[0],
                             dbeta=gr[1] if with_beta else None, with_dbeta=with_beta,
                             workspace=d["ws"])
        elif ln:
            L.layer_norm_fwd(x, g, d.get("beta"), w.eps, y=y, mean=st[0], rstd=st[1])
            L.layer_norm_bwd(dy, x, g, st[0], st[1], dx=dx, dgamma=gr[0],
                             dbeta=gr[1] if with_beta else None, with_dbeta=with_beta,
                             workspace=d["ws"])
        elif f8:
            L.rms_norm_fwd_fp8(x, g, scale, w.eps, w.offset, y=y, rstd=st[0])
            L.rms_norm_bwd(dy, x, g, st[0], w.offset, dx=dx, dw=gr[0], workspace=d["ws"])
        else:
            L.rms_norm_fwd(x, g, w.eps, w.offset, w.cast_mode, y=y, rstd=st[0])
            L.rms_norm_bwd(dy, x, g, st[0], w.offset, dx=dx, dw=gr[0], workspace=d["ws"])

    def one(i):
        k = i % 2
        d = sets[k]
        with torch.cuda.stream(s_in):        # upload once the set's last kernels are done
            s_in.wait_event(computed[k])
            for name, v in host_in.items():
                d[name].copy_(v, non_blocking=True)
            loaded[k].record(s_in)
        with torch.cuda.stream(s_run):       # compute once uploaded and the last download left
            s_run.wait_event(loaded[k])
            s_run.wait_event(drained[k])
            compute(d)
            computed[k].record(s_run)
        with torch.cuda.stream(s_out):       # download the results
            s_out.wait_event(computed[k])
            yv = d["y"].view(torch.uint8) if f8 else d["y"]
            hy.copy_(yv, non_blocking=True)
            hdx.copy_(d["dx"], non_blocking=True)
            for h, t in zip(hstats + hgrads, d["stats"] + d["grads"]):
                h.copy_(t.view(-1), non_blocking=True)
            drained[k].record(s_out)

    for i in range(10):
        one(i)
    torch.cuda.synchronize()
    t = time.perf_counter()
    for i in range(steps):
        one(i)
    torch.cuda.synchronize()
    secs = (time.perf_counter() - t) / steps
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in [hy, hdx] + hstats + hgrads)

    # the host link alone, on the same pinned buffers and streams: the bound
    # of the figure above
    def copies(up: bool, down: bool, reps: int = 5):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            d = sets[0]
            if up:
                with torch.cuda.stream(s_in):
                    for name, v in host_in.items():
                        d[name].copy_(v, non_blocking=True)
            if down:
                with torch.cuda.stream(s_out):
                    hy.copy_(d["y"].view(torch.uint8) if f8 else d["y"], non_blocking=True)
                    hdx.copy_(d["dx"], non_blocking=True)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps

    t_up, t_down, t_both = copies(True, False), copies(False, True), copies(True, True)
    big_d2h = hy.numel() * hy.element_size() + hdx.numel() * hdx.element_size()
    return {"value": round(w.step_bytes() / secs / 1e9, 2), "unit": "GB/s",
            "us_per_step": round(secs * 1e6, 2),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "timing": ("wall clock over steps after 10 warm-up steps, synchronised at both "
                       "ends; copies in, kernels and copies out on three streams over two "
                       "device buffer sets; host buffers pinned once before the warm-up"),
            "host_link_gbs": {"h2d": round(h2d / t_up / 1e9, 1),
                              "d2h": round(big_d2h / t_down / 1e9, 1),
                              "both_directions": round((h2d + big_d2h) / t_both / 1e9, 1)},
            "numa": numa_placement(dev)}


def numa_placement(dev):
    """NUMA node of the GPU (from its PCI device) and the host's node count;
    pinned host buffers are first-touched by this process on its cores."""
    import torch
    props = torch.cuda.get_device_properties(dev)
    out = {"host_nodes": len([d for d in os.listdir("/sys/devices/system/node")
                              if d.startswith("node") and d[4:].isdigit()])
           if os.path.isdir("/sys/devices/system/node") else None,
           "cpus_allowed": host_threads()}
    try:
        bus = "%04x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
        with open(f"/sys/bus/pci/devices/{bus}/numa_node") as f:
            out["gpu_node"] = int(f.read().strip())
        out["gpu_pci"] = bus
    except (AttributeError, OSError, ValueError):
        out["gpu_node"] = None
    return out


def code_of(text: str) -> str:
    """C/C++/CUDA source with its comments removed and its whitespace
    collapsed: what decides the kernels built from it."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def sources_hash(files) -> str:
    """First 16 hex digits of the SHA-256 of the named CUDA sources' code
    (file names and code_of of their contents, in the given order), to
    tell whether committed counters still describe the kernels being run;
    edits to comments or layout leave it unchanged."""
    import hashlib
    h = hashlib.sha256()
    for name in files:
        h.update(name.encode())
        with open(os.path.join(ROOT, "bwd_rms_norm_gb300", "csrc", name)) as fh:
            h.update(code_of(fh.read()).encode())
    return h.hexdigest()[:16]


def load_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary
    (profiles/traffic.json), or {} when it does not cover this workload or
    was taken on kernels other than the ones built from the current
    sources (the entry lists the source files its kernels come from)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            data = json.load(f).get(workload, {})
        if data.get("sources_sha256_16") != sources_hash(data.get("sources", [])):
            return {}
    except (OSError, ValueError):
        return {}
    return data


# ---------------------------------------------------------------------------
# reference arm: the float64 oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args, rank, world, local):
    if rank != 0:
        return
    w = workload_by_name(args.workload)
    threads = host_threads()
    # size the sample so that warmup + steps take about two minutes
    nprobe = max(threads, min(64 * threads, (1 << 22) // w.hidden))
    probe, _ = time_oracle(w, nprobe, threads)
    per_row = probe / nprobe
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(min(16, w.rows), min(w.rows, budget / per_row)))
    for _ in range(args.warmup):
        time_oracle(w, rows, threads)
    times = []
    nbytes = 0
    for _ in range(args.steps):
        s, nbytes = time_oracle(w, rows, threads)
        times.append(s)
    total = sum(times)
    value = nbytes * len(times) / total / 1e9
    sample = (f"{args.workload}: float64 oracle forward+backward over {rows} of {w.rows} rows "
              f"per step (numpy), the rows split in {threads} contiguous ranges on {threads} "
              f"host threads")
    line = {
        "impl": "reference",
        "metric": metric_for(w),
        "value": round(value, 5),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / len(times), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded, see workloads/)",
        "config": {"workload": args.workload, "rows": w.rows, "hidden": w.hidden,
                   "sample_rows": rows},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample, "nproc": os.cpu_count()},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--rows", type=int, default=0,
                    help="override the workload's row count (profiling a larger case)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dp-exchange", action="store_true",
                    help="on one rank, run the data-parallel weight-gradient path of N > 1")
    ap.add_argument("--profile", action="store_true",
                    help="run warm-up and steps eagerly and nothing else (for ncu)")
    ap.add_argument("--no-variant", action="store_true",
                    help="skip timing the other cast mode of a workload that has both")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
