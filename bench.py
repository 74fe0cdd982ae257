#!/usr/bin/env python
"""Benchmark of the fused RMSNorm forward + backward on GB300.

One step = one forward (rms_norm_fwd) and one backward (rms_norm_bwd, which
includes the fixed-order weight-gradient reduction) over one batch of the
workload, through the C ABI.  Default workload: Llama-shaped bf16
activation, 4096 rows (4 x 1024 tokens) x hidden 4096, eps 1e-5, round-once
store, inputs drawn once (seeded) and resident in HBM.

Printed (rank 0, one JSON line): achieved GB/s of algorithmic bytes over the
device time of our kernels (CUDA events on the launching stream, L2 flushed
before every timed call), microseconds per call, the roofline of the
backward call, an end-to-end number through the public API with host
buffers, the float64 oracle timed on the host as a baseline, and the SM
clocks sampled during the timed region.

``--impl reference`` times the oracle instead (rank 0 only, on the host
cores, on a bounded sample of the same workload).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
Under torchrun every rank runs the workload on its own GPU (weak scaling:
the rows of one batch per rank, no collective on the data path); the time
is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "RMSNorm fwd+bwd achieved HBM GB/s and % of GB300 peak; µs per call"
DEFAULT_WORKLOAD = "llama_bf16_4096x4096"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
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
    """nvidia-smi sampled every 100 ms in the background."""

    def __init__(self, gpu_id: str):
        self.t0 = time.time()
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", gpu_id],
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


def time_oracle(w, rows: int):
    """Seconds for one oracle forward + backward over ``rows`` rows of ``w``
    (inputs drawn once per row count, outside the timing)."""
    import workloads as W
    from oracle import rms_norm as orm
    ws = w.with_(rows=rows)
    if (ws.name, rows) not in _ORACLE_INPUTS:
        _ORACLE_INPUTS.clear()
        inp = W.make_inputs(ws)
        _ORACLE_INPUTS[(ws.name, rows)] = tuple(W.as_float64(inp[k]) for k in ("x", "gamma", "dy"))
    xd, gd, dyd = _ORACLE_INPUTS[(ws.name, rows)]
    t = time.perf_counter()
    _, rstd = orm.forward(xd, gd, ws.eps, ws.offset, ws.dtype, ws.cast_mode)
    orm.backward(dyd, xd, gd, rstd, ws.offset, ws.dtype)
    return time.perf_counter() - t, ws.step_bytes()


def run_ours(args, rank, world, local):
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

    w = W.all_workloads()[args.workload]
    inp = W.make_inputs(w)
    x, g, dy = (inp[k].to(dev) for k in ("x", "gamma", "dy"))
    y = torch.empty_like(x)
    rstd = torch.empty(w.rows, dtype=torch.float32, device=dev)
    dx = torch.empty_like(x)
    dw = torch.empty(w.hidden, dtype=torch.float32, device=dev)
    ws = torch.empty(L.rms_norm_bwd_workspace_size(w.rows, w.hidden, x.dtype), dtype=torch.uint8,
                     device=dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or (126 << 20))
    flush_elems = 2 * l2 // 4
    flush = torch.empty(flush_elems, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call_fwd():
        L.rms_norm_fwd(x, g, w.eps, w.offset, w.cast_mode, y=y, rstd=rstd)

    def call_bwd():
        L.rms_norm_bwd(dy, x, g, rstd, w.offset, dx=dx, dw=dw, workspace=ws)

    def l2_flush(i):
        flush.fill_(i)                 # writes 2x the L2 size
        torch.cuda._sleep(200_000)     # keeps the GPU busy while the host enqueues

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]

    def step(i, evs):
        l2_flush(2 * i)
        if evs: evs[0].record(stream)
        call_fwd()
        if evs: evs[1].record(stream)
        l2_flush(2 * i + 1)
        if evs: evs[2].record(stream)
        call_bwd()
        if evs: evs[3].record(stream)

    for i in range(args.warmup):
        step(i, None)
    torch.cuda.synchronize()

    uuid = str(getattr(props, "uuid", "")) or str(local)
    sampler = ClockSampler(("GPU-" + uuid) if uuid and not uuid.isdigit() else uuid)
    # let the sampler start and the clocks settle on the same work
    t_soak = time.time()
    while time.time() - t_soak < 0.5:
        for i in range(20):
            step(i, None)
        torch.cuda.synchronize()

    barrier(world)
    torch.cuda.synchronize()
    t_start = time.time()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        step(i, ev[i])
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(world)
    t_end = time.time()
    sampler.mark(t_start, t_end)
    clocks = sampler.stop()

    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[2].elapsed_time(e[3]) for e in ev]
    kern_ms = sum(fwd_ms) + sum(bwd_ms)
    kern_ms = reduce_max(kern_ms, world, dev)
    ms_per_step = kern_ms / args.steps
    total_bytes = w.step_bytes() * args.steps * world
    value = total_bytes / (kern_ms * 1e-3) / 1e9

    peak, peak_src = measured_peak_gbs()
    bwd_avg_s = statistics.mean(bwd_ms) * 1e-3
    fwd_avg_s = statistics.mean(fwd_ms) * 1e-3
    bwd_ach = w.bwd_bytes() / bwd_avg_s / 1e9
    fwd_ach = w.fwd_bytes() / fwd_avg_s / 1e9
    traffic = load_traffic(args.workload)

    # end to end through the public API: pinned host inputs in, results out
    e2e = run_e2e(L, w, inp, dev, args.e2e_steps)
    e2e["value"] = reduce_max_rate(e2e["value"], world, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # whole-workload passes of the oracle, repeated until about 10 s of
        # host time have been spent
        secs, nbytes, passes = 0.0, 0, 0
        while secs < 10.0 and passes < 50:
            s, b = time_oracle(w, w.rows)
            secs += s
            nbytes += b
            passes += 1
        cpu = {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": 1,
               "kind": "oracle",
               "sample": f"{args.workload}: {passes} float64 forward+backward passes over all "
                         f"{w.rows} rows ({secs:.1f} s, numpy, single thread)"}

    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else w.dtype,
        "data": "synthetic (seeded, see workloads/)",
        "config": {
            "workload": args.workload, "rows": w.rows, "hidden": w.hidden, "eps": w.eps,
            "offset": w.offset, "cast_mode": w.cast_mode, "stats": "fp32", "rstd": "fp32",
            "dw": "fp32", "global_batch_rows": w.rows * world,
            "parallelism": f"replica x{world} (rows per rank)",
            "l2": "flushed before every timed call (write of 2x L2)",
            "timing": "CUDA events around each C-ABI call on its stream; value = bytes / sum of event times",
            "algorithmic_bytes_per_step": w.step_bytes(),
        },
        "fwd_us": round(statistics.mean(fwd_ms) * 1e3, 3),
        "bwd_us": round(statistics.mean(bwd_ms) * 1e3, 3),
        "fwd_us_median": round(statistics.median(fwd_ms) * 1e3, 3),
        "bwd_us_median": round(statistics.median(bwd_ms) * 1e3, 3),
        "pct_of_hbm_peak": round(100.0 * value / world / peak, 2),
        "peak_source": f"{peak_src} HBM {peak} GB/s",
        "roofline": {
            "kernel": "rms_norm_bwd (row kernel + dw finalize)",
            "bound": "hbm", "achieved": round(bwd_ach, 1), "peak": peak, "unit": "GB/s",
            "frac": round(bwd_ach / peak, 4),
            "traffic": traffic.get("bwd"),
            "algorithmic_bytes": w.bwd_bytes(),
        },
        "roofline_fwd": {
            "kernel": "rms_norm_fwd", "bound": "hbm", "achieved": round(fwd_ach, 1),
            "peak": peak, "unit": "GB/s", "frac": round(fwd_ach / peak, 4),
            "traffic": traffic.get("fwd"), "algorithmic_bytes": w.fwd_bytes(),
        },
        "e2e": e2e,
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 4),
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)


def reduce_max_rate(rate: float, world: int, dev) -> float:
    """Aggregate rate over ranks: world / (max over ranks of 1/rate)."""
    if world <= 1:
        return rate
    t = reduce_max(1.0 / rate, world, dev)
    return world / t


def run_e2e(L, w, inp, dev, steps: int):
    """GB/s of algorithmic bytes when every step copies the inputs from
    pinned host memory, runs forward and backward through the Python API and
    copies every result back to pinned host memory."""
    import torch
    hx, hg, hdy = (inp[k].pin_memory() for k in ("x", "gamma", "dy"))
    hy = torch.empty_like(hx).pin_memory()
    hdx = torch.empty_like(hx).pin_memory()
    hr = torch.empty(w.rows, dtype=torch.float32).pin_memory()
    hdw = torch.empty(w.hidden, dtype=torch.float32).pin_memory()
    x = torch.empty_like(hx, device=dev)
    g = torch.empty_like(hg, device=dev)
    dy = torch.empty_like(hdy, device=dev)
    ws = torch.empty(L.rms_norm_bwd_workspace_size(w.rows, w.hidden, x.dtype), dtype=torch.uint8,
                     device=dev)

    def one():
        x.copy_(hx, non_blocking=True)
        g.copy_(hg, non_blocking=True)
        dy.copy_(hdy, non_blocking=True)
        y, rstd = L.rms_norm_fwd(x, g, w.eps, w.offset, w.cast_mode)
        dx, dw = L.rms_norm_bwd(dy, x, g, rstd, w.offset, workspace=ws)
        hy.copy_(y, non_blocking=True)
        hr.copy_(rstd, non_blocking=True)
        hdx.copy_(dx, non_blocking=True)
        hdw.copy_(dw, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    t = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    secs = (time.perf_counter() - t) / steps
    h2d = sum(t.numel() * t.element_size() for t in (hx, hg, hdy))
    d2h = sum(t.numel() * t.element_size() for t in (hy, hr, hdx, hdw))
    return {"value": round(w.step_bytes() / secs / 1e9, 2), "unit": "GB/s",
            "us_per_step": round(secs * 1e6, 2),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "timing": "wall clock over steps, synchronised at both ends"}


def load_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it covers the
    current kernels of this workload (see profiles/)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
        return data.get(workload, {})
    except (OSError, ValueError):
        return {}


# ---------------------------------------------------------------------------
# reference arm: the float64 oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args, rank, world, local):
    if rank != 0:
        return
    import workloads as W
    w = W.all_workloads()[args.workload]
    # size the sample so that warmup + steps take about two minutes
    probe, _ = time_oracle(w, 64)
    per_row = probe / 64
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(16, min(w.rows, budget / per_row)))
    for _ in range(args.warmup):
        time_oracle(w, rows)
    times = []
    nbytes = 0
    for _ in range(args.steps):
        s, nbytes = time_oracle(w, rows)
        times.append(s)
    total = sum(times)
    value = nbytes * len(times) / total / 1e9
    sample = (f"{args.workload}: float64 oracle forward+backward over {rows} of {w.rows} rows "
              f"per step (numpy, single thread)")
    line = {
        "impl": "reference",
        "metric": METRIC,
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
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": 1,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
