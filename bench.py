"""Benchmark: RMSNorm forward + backward on one GB300, through the C ABI.

One step = rms_fwd + rms_bwd (forward, backward rows, dgamma column
reduction) over the 16384 x 8192 bf16 workload, inputs resident in HBM.
Prints ONE JSON line (rank 0):

  value      whole-job algorithmic HBM GB/s of the step, summed over ranks
  roofline   the backward call (the dominant one) against the measured HBM peak
  e2e        the same metric with host buffers: pinned H2D of x, dy, gamma and
             D2H of y, rstd, dx, dgamma inside every timed step
  cpu_baseline  the fp64 oracle on a bounded row sample, on the host cores

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--shard rows|replicas]

For N > 1 launch one process per GPU with torch.distributed.run.  With
--shard rows (the default) the job is one batch of N x 16384 rows split into
contiguous blocks, one per rank: each rank normalises its own rows (the
forward and dx need no exchange) and the per-rank dgamma vectors are
all-gathered and added in rank order by the library's kernel, so every rank
ends with the whole batch's dgamma.  --shard replicas runs the same block on
every rank with no exchange.  Per-GPU work is fixed as N grows (weak
scaling); timing is max over ranks.
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

WORKLOAD = "wide_bf16_16384x8192"
METRIC = "RMSNorm fwd+bwd achieved HBM GB/s and % of GB300 peak at M×N bf16; rows/s"
L2_BYTES = 129 * 1000 * 1000
FALLBACK_HBM_GBS = 6800.0


def step_bytes(M: int, N: int, b: int):
    """Algorithmic bytes: fwd reads x, writes y and rstd; bwd reads dy, x and
    rstd, writes dx; plus gamma (read once per call) and dgamma (written once)."""
    fwd = 2 * M * N * b + 4 * M + N * b
    bwd = 3 * M * N * b + 4 * M + N * b + 4 * N
    return fwd, bwd


def ln_step_bytes(M: int, N: int, b: int, wb: int, bias: bool):
    """LayerNorm algorithmic bytes: fwd reads x, w (and b), writes y, mean and
    rstd; bwd reads dy, x, w, mean and rstd, writes dx, dw and db."""
    fwd = 2 * M * N * b + 8 * M + (2 if bias else 1) * N * wb
    bwd = 3 * M * N * b + 8 * M + N * wb + 8 * N
    return fwd, bwd


def add_step_bytes(M: int, N: int, b: int, wb: int):
    """Residual add fused into RMSNorm: fwd reads x and the residual, writes h,
    y and rstd; bwd reads dy, h, rstd and dh, writes dx and dgamma."""
    fwd = 4 * M * N * b + 4 * M + N * wb
    bwd = 4 * M * N * b + 4 * M + N * wb + 4 * N
    return fwd, bwd


def quant_fwd_bytes(M: int, N: int, b: int, wb: int):
    """Forward with an E4M3 output: reads x, writes one byte per element, the
    per-row scale and rstd."""
    return M * N * b + M * N + 8 * M + N * wb


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------- distributed
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def init_dist(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def max_over_ranks(value: float, dist, device=None) -> float:
    """Max of a float over all ranks (the whole job ends with the slowest)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.window = None
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            return
        self.first = threading.Event()
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        self.first.wait(5.0)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [c.strip() for c in line.split(",")]))
            self.first.set()

    def start(self):
        self.t0 = time.time()

    def stop(self):
        self.window = (self.t0, time.time())

    def close(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.window is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        t0, t1 = self.window
        inside = [s for t, s in self.samples if t0 - 0.1 <= t <= t1 + 0.25]
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in inside:
            try:
                sm.append(float(s[1]))
                smax = float(s[2])
            except (ValueError, IndexError):
                continue
            for name, v in zip(names, s[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------- CPU oracle
def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_worker(conn, wname, rows, workers, k):
    """One host core's share of the oracle timing: the k-th block of ``rows``
    rows of a seeded sample of the workload, run on command."""
    from oracle import rmsnorm_oracle as orc
    from synthetic import make_inputs, storage_to_float64, workload

    w = workload(wname)
    inp = make_inputs(w.with_shape(rows * workers))
    sl = slice(k * rows, (k + 1) * rows)
    x = storage_to_float64(inp["x"][sl], w.dtype)
    dy = storage_to_float64(inp["dy"][sl], w.dtype)
    g = storage_to_float64(inp["gamma"], w.wdtype)
    conn.send("ready")
    while True:
        msg = conn.recv()
        if msg is None:
            break
        what, reps = msg
        dg = None
        for _ in range(reps):
            if what in ("fwd", "step"):
                orc.rms_forward(x, g, w.eps, w.gemma)
            if what in ("bwd", "step"):
                _, dg = orc.rms_backward(x, g, dy, w.eps, w.gemma)
        conn.send(dg)
    conn.close()


class OraclePool:
    """The fp64 oracle on every host core: one spawned process per core, each
    holding its own block of rows (processes, not threads: numpy's
    elementwise work would serialise on the interpreter lock).  ``run`` sends
    one command to every worker and returns the wall time until the last
    reply, and the workers' dgamma partials summed in worker order."""

    def __init__(self, wname: str, rows_per_worker: int, workers: int):
        import multiprocessing as mp

        # one thread per worker process; spawned (not forked) workers never
        # inherit a CUDA context
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ.setdefault(var, "1")
        ctx = mp.get_context("spawn")
        self.rows, self.workers = rows_per_worker, workers
        self.conns, self.procs = [], []
        for k in range(workers):
            a, b = ctx.Pipe()
            p = ctx.Process(target=_oracle_worker, args=(b, wname, rows_per_worker, workers, k),
                            daemon=True)
            p.start()
            self.conns.append(a)
            self.procs.append(p)
        for c in self.conns:
            if c.recv() != "ready":
                raise RuntimeError("oracle worker failed to start")

    def run(self, what: str, reps: int = 1):
        t0 = time.perf_counter()
        for c in self.conns:
            c.send((what, reps))
        parts = [c.recv() for c in self.conns]
        el = time.perf_counter() - t0
        dg = None
        if parts[0] is not None:
            dg = parts[0].copy()
            for p in parts[1:]:
                dg += p
        return el, dg

    def close(self):
        for c in self.conns:
            try:
                c.send(None)
            except (BrokenPipeError, OSError):
                pass
        for p in self.procs:
            p.join(timeout=10)
            if p.is_alive():
                p.kill()


def cpu_oracle_throughput(w, seconds: float = 12.0, rows_per_worker: int = 64, runs: int = 3,
                          workers: int = 0):
    """The fp64 oracle on a bounded row sample split over every host core:
    forward and backward timed separately, each in ``runs`` runs of about
    seconds / (2 runs); medians per direction, GB/s on the same
    algorithmic-byte formula as the GPU."""
    workers = workers or host_cores()
    pool = OraclePool(w.name, rows_per_worker, workers)
    try:
        budget = seconds / (2 * runs)

        def per_call(what):
            el, _ = pool.run(what, 1)  # calibration: repetitions that fill the budget
            reps = max(1, int(budget / max(el, 1e-6)))
            times = sorted(pool.run(what, reps)[0] / reps for _ in range(runs))
            return times[len(times) // 2], reps * runs

        t_f, n_f = per_call("fwd")
        t_b, n_b = per_call("bwd")
    finally:
        pool.close()
    rows = rows_per_worker * workers
    f, b = step_bytes(rows, w.N, w.elem_bytes)
    return {
        "value": round((f + b) / (t_f + t_b) / 1e9, 3),
        "unit": "GB/s",
        "fwd_gbs": round(f / t_f / 1e9, 3),
        "bwd_gbs": round(b / t_b / 1e9, 3),
        "rows_per_s": round(rows / (t_f + t_b), 1),
        "cores": workers,
        "kind": "oracle",
        "sample": (f"fp64 numpy oracle on {rows} seeded rows of the {w.M}x{w.N} {w.dtype} "
                   f"workload, {rows_per_worker} rows on each of {workers} host cores (one "
                   f"process per core): forward ({n_f} passes) and backward ({n_b} passes) "
                   f"timed apart, median of {runs} runs each, about {seconds:.0f} s in all; "
                   "value = fwd+bwd bytes over the sum of the two medians"),
    }


# ------------------------------------------------------------------ reference
def run_reference(args):
    """The reference arm: the fp64 oracle on every host core, one bounded row
    sample of the same workload per step (each core its own rows), rank 0
    only."""
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    from synthetic import workload

    w = workload(WORKLOAD)
    workers = host_cores()
    rows_per_worker = 64
    rows = rows_per_worker * workers
    pool = OraclePool(w.name, rows_per_worker, workers)
    try:
        for _ in range(args.warmup):
            pool.run("step")
        el = sum(pool.run("step")[0] for _ in range(args.steps))
    finally:
        pool.close()
    f, b = step_bytes(rows, w.N, w.elem_bytes)
    value = (f + b) * args.steps / el / 1e9
    sample = (f"fp64 numpy oracle fwd+bwd on {rows} rows x {w.N} per step (seeded rows of the "
              f"{w.M}x{w.N} {w.dtype} workload), {rows_per_worker} rows on each of {workers} "
              "host cores, one process per core")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w),
        "rows_per_s": round(rows * args.steps / el, 2),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": workers,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_dict(w, world: int = 1, shard: str = "rows"):
    d = {
        "workload": f"RMSNorm fwd+bwd, M={w.M} rows x N={w.N} hidden, {w.dtype} I/O, "
                    f"eps={w.eps}, large-hidden synthetic rows (x ~ N(0,1) x log-uniform "
                    "row scale [0.01, 100], gamma ~ N(1, 0.2), dy ~ N(0, 1), seed 0)",
        "M": w.M, "N": w.N, "eps": w.eps, "gemma": w.gemma, "inplace_dx": w.inplace_dx,
        "l2": "inputs larger than L2: x, dy, y, dx are 256 MiB each (L2 is 129 MB)",
    }
    if world > 1:
        d["sharding"] = (
            f"rows: a batch of {world} x {w.M} rows, rank r holding rows [r*{w.M}, (r+1)*{w.M}) "
            "(drawn with seed r); dgamma all-gathered and added in rank order every step"
            if shard == "rows" else
            f"replicas: every rank runs the same {w.M}-row block, no exchange")
    return d


# ------------------------------------------------------------------------ GPU
def run_gpu(args):
    import numpy as np
    import torch

    from dataclasses import replace

    import row_wise_normalization_rms_gb300 as rms
    from row_wise_normalization_rms_gb300 import sharded
    from synthetic import make_inputs, workload

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    w = workload(WORKLOAD)
    M, N, b = w.M, w.N, w.elem_bytes
    fwd_b, bwd_b = step_bytes(M, N, b)
    rows_mode = args.shard == "rows"

    # Row shards: rank r holds rows [r M, (r+1) M) of a world x M batch, drawn
    # with seed + r (rank 0's block is the single-GPU workload itself).
    inp = make_inputs(replace(w, seed=w.seed + rank) if rows_mode and rank else w)

    def pinned(a):
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        return t.pin_memory()

    hx, hdy, hg = pinned(inp["x"]), pinned(inp["dy"]), pinned(inp["gamma"])
    x = hx.to(dev)
    dy = hdy.to(dev)
    g = hg.to(dev)
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    rstd = torch.empty(M, device=dev)
    dg = torch.empty(N, device=dev)
    ws = torch.empty(rms.rms_bwd_workspace_size(M, N), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    exchange = rows_mode and world > 1
    dg_local = torch.empty(N, device=dev) if exchange else dg

    def backward(dy, x, g, r, dx, dg, dgl, ws, s):
        """This rank's rows; with row shards over several ranks, dgamma of
        the whole batch from the rank-ordered exchange."""
        if exchange:
            sharded.rms_bwd_sharded(dy, x, g, r, dx, dg, dgl, ws, w.gemma, w.inplace_dx, stream=s)
        else:
            rms.rms_bwd(dy, x, g, r, dx, dg, ws, w.gemma, w.inplace_dx, stream=s)

    def step():
        rms.rms_fwd(x, g, y, rstd, w.eps, w.gemma, stream=stream)
        backward(dy, x, g, rstd, dx, dg, dg_local, ws, stream)

    clocks = ClockSampler(local) if rank == 0 else None
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    torch.cuda.synchronize(dev)

    # Timed region: K steps back to back, events only at its ends (events
    # between calls would serialise the kernels' programmatic overlap).
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    launches0 = rms.rms_launch_count()
    if clocks:
        clocks.start()
    e_start.record(stream)
    for _ in range(args.steps):
        step()
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.stop()
    launches = rms.rms_launch_count() - launches0
    total_ms = e_start.elapsed_time(e_end)
    barrier(dist, dev)
    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_step = total_ms / args.steps
    value = (fwd_b + bwd_b) * world / (ms_step * 1e-3) / 1e9

    # Per-call durations: the same calls, K of one kind back to back, on the
    # same stream; average = elapsed / K.
    def per_call(fn, k):
        for _ in range(3):
            fn()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(k):
            fn()
        z.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(z) / k

    k_call = max(10, args.steps // 2)
    fwd_avg = per_call(lambda: rms.rms_fwd(x, g, y, rstd, w.eps, w.gemma, stream=stream), k_call)
    bwd_avg = per_call(lambda: backward(dy, x, g, rstd, dx, dg, dg_local, ws, stream), k_call)

    # End to end: every step copies its inputs (x, dy, gamma) from pinned host
    # memory and its results (y, rstd, dx, dgamma) back, through the same C
    # ABI calls.  Steps are double-buffered the way a streaming caller would
    # run them: the H2D copies of step i+1 and the D2H copies of step i-1
    # (each direction split over two copy streams) overlap the kernels of
    # step i; events order each buffer set's reuse.
    e2e_steps = max(4, min(args.steps, 20))
    hy = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
    hdx = torch.empty_like(hy).pin_memory()
    hr = torch.empty(M).pin_memory()
    hdg = torch.empty(N).pin_memory()
    bufs = [dict(x=x, dy=dy, g=g, y=y, dx=dx, r=rstd, dg=dg, dgl=dg_local, ws=ws)]
    dg2 = torch.empty_like(dg)
    bufs.append(dict(x=torch.empty_like(x), dy=torch.empty_like(dy), g=torch.empty_like(g),
                     y=torch.empty_like(y), dx=torch.empty_like(dx), r=torch.empty_like(rstd),
                     dg=dg2, dgl=torch.empty_like(dg) if exchange else dg2,
                     ws=torch.empty_like(ws)))
    s_comp = torch.cuda.Stream(dev)
    s_in = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    s_out = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    ev = lambda: torch.cuda.Event()
    in_done = [ev(), ev()]     # inputs of the set copied in
    comp_done = [ev(), ev()]   # kernels of the set finished (inputs free, outputs ready)
    out_done = [ev(), ev()]    # outputs of the set copied out (outputs free)
    for e in comp_done + out_done:
        e.record(s_comp)

    def e2e_step(i):
        B = bufs[i % 2]
        j = i % 2
        # inputs in: after the kernels that last read this set
        for k, (dst, src) in enumerate(((B["x"], hx), (B["dy"], hdy))):
            s_in[k].wait_event(comp_done[j])
            with torch.cuda.stream(s_in[k]):
                dst.copy_(src, non_blocking=True)
                if k == 0:
                    B["g"].copy_(hg, non_blocking=True)
        in_done[j].record(s_in[0])
        s_comp.wait_event(in_done[j])
        s_comp.wait_stream(s_in[1])
        s_comp.wait_event(out_done[j])  # this set's previous outputs are out
        rms.rms_fwd(B["x"], B["g"], B["y"], B["r"], w.eps, w.gemma, stream=s_comp)
        with torch.cuda.stream(s_comp):  # the exchange's collective runs on s_comp too
            backward(B["dy"], B["x"], B["g"], B["r"], B["dx"], B["dg"], B["dgl"], B["ws"], s_comp)
        comp_done[j].record(s_comp)
        for k, (dst, src) in enumerate(((hy, B["y"]), (hdx, B["dx"]))):
            s_out[k].wait_event(comp_done[j])
            with torch.cuda.stream(s_out[k]):
                dst.copy_(src, non_blocking=True)
                if k == 0:
                    hr.copy_(B["r"], non_blocking=True)
                    hdg.copy_(B["dg"], non_blocking=True)
        s_out[0].wait_stream(s_out[1])
        out_done[j].record(s_out[0])

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in[0])
    for s_ in (s_in[1], s_comp, s_out[0], s_out[1]):
        s_.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    for s_ in (s_in[0], s_in[1], s_comp, s_out[1]):
        s_out[0].wait_stream(s_)
    e1.record(s_out[0])
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev) / e2e_steps
    h2d = (hx.numel() + hdy.numel() + hg.numel()) * 2
    d2h = (hy.numel() + hdx.numel()) * 2 + (hr.numel() + hdg.numel()) * 4

    if clocks:
        clocks.close()
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peak, peak_kind = measured_peaks()
    bwd_gbs = bwd_b / (bwd_avg * 1e-3) / 1e9
    fwd_gbs = fwd_b / (fwd_avg * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": config_dict(w, world, args.shard),
        "rows_per_s": round(M * world / (ms_step * 1e-3), 1),
        "pct_of_hbm_peak": round(100.0 * value / (peak * world), 2),
        "per_call": {
            "fwd_us": round(fwd_avg * 1e3, 2), "fwd_gbs": round(fwd_gbs, 1),
            "fwd_frac": round(fwd_gbs / peak, 4),
            "bwd_us": round(bwd_avg * 1e3, 2), "bwd_gbs": round(bwd_gbs, 1),
            "bwd_frac": round(bwd_gbs / peak, 4),
            "note": ("average over back-to-back calls of one kind (CUDA events around the "
                     "loop); bwd = backward rows kernel + dgamma column reduction"),
        },
        "roofline": {
            "bound": "hbm",
            "achieved": round(bwd_gbs, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(bwd_gbs / peak, 4),
            "traffic": captured_traffic("bwd"),
            "kernel": "rms_bwd (rms_bwd_staged_kernel + rms_colreduce4_kernel)",
            "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind}, burst copy)",
        },
        "roofline_fwd": {
            "bound": "hbm", "achieved": round(fwd_gbs, 1), "peak": peak, "unit": "GB/s",
            "frac": round(fwd_gbs / peak, 4), "traffic": captured_traffic("fwd"),
            "kernel": "rms_fwd (rms_fwd_registers_kernel)",
        },
        "e2e": {
            "value": round((fwd_b + bwd_b) * world / (e2e_ms * 1e-3) / 1e9, 2),
            "unit": "GB/s",
            "ms_per_step": round(e2e_ms, 4),
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "pipeline": ("pinned host buffers; two device buffer sets; H2D of step i+1 and D2H "
                         "of step i-1 on two copy streams per direction overlap the kernels of "
                         "step i; every step's copies inside the timed region"),
        },
        "gpu_launches": launches,
        "clocks": clocks.summary() if clocks else None,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_throughput(w)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


# DRAM bytes per call from one ncu capture of these kernels at this workload
# (dram__bytes_read.sum + dram__bytes_write.sum of one timed step, summed
# over the call's launches, as the committed launch-list summary records).
# They are reported only while the kernel sources hash to the value they were
# captured with; after any change to their code the traffic reads null.  The
# hash skips comments and whitespace, which do not reach the compiled code.
TRAFFIC_CAPTURE = {
    "src_sha256_16": "bf488343656e754c",
    "bwd": 537020416 + 233731584 + 9970176 + 0,  # staged rows kernel + column reduction
    "fwd": 268470528 + 215786240,                # register-mapping forward
}


# The sources the measured kernels (register forward, staged backward, column
# reduction) and their dispatch are built from.
MEASURED_KERNEL_SOURCES = ["api.cu", "common.cuh", "fwd_registers.cu", "internal.h", "scalar.cu",
                           "staged.cu", "tma.cuh"]


def code_tokens(text: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs collapsed to one
    space (string and character literals kept as written)."""
    import re

    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return re.sub(r"\s+", " ", "".join(out)).strip()


def kernel_source_hash() -> str:
    import hashlib

    csrc = os.path.join(ROOT, "row_wise_normalization_rms_gb300", "csrc")
    h = hashlib.sha256()
    for name in MEASURED_KERNEL_SOURCES:
        h.update(name.encode())
        with open(os.path.join(csrc, name), encoding="utf-8") as fh:
            h.update(code_tokens(fh.read()).encode())
    return h.hexdigest()[:16]


def captured_traffic(which: str):
    if kernel_source_hash() != TRAFFIC_CAPTURE["src_sha256_16"]:
        return None
    return TRAFFIC_CAPTURE[which]


SPEC_KEYS = {"M": int, "N": int, "dtype": str, "eps": float, "gemma": int, "inplace": int,
             "seed": int, "op": str, "weight": str}


def workload_from_spec(spec: str, name: str = ""):
    """A workload from ``key=value`` pairs (M, N required; dtype bf16|f16|f32,
    eps, gemma 0|1, inplace 0|1, seed, op rms|ln|rms_add|rms_quant, weight
    f32 for a float32 weight); input laws are those of the row-width sweep."""
    from synthetic import Workload

    kv = {}
    for part in filter(None, (p.strip() for p in spec.split(","))):
        key, sep, val = part.partition("=")
        if not sep or key not in SPEC_KEYS:
            raise ValueError(f"bad workload field {part!r}; fields: {', '.join(SPEC_KEYS)}")
        kv[key] = SPEC_KEYS[key](val)
    if "M" not in kv or "N" not in kv:
        raise ValueError("a workload spec needs M and N")
    if kv["M"] < 0 or kv["N"] < 1:
        raise ValueError("M >= 0 and N >= 1")
    if kv.get("dtype", "bf16") not in ("bf16", "f16", "f32"):
        raise ValueError("dtype is bf16, f16 or f32")
    if kv.get("op", "rms") not in ("rms", "ln", "rms_add", "rms_quant"):
        raise ValueError("op is rms, ln, rms_add or rms_quant")
    if kv.get("gemma", 0) not in (0, 1) or kv.get("inplace", 0) not in (0, 1):
        raise ValueError("gemma and inplace are 0 or 1")
    op = kv.get("op", "rms")
    return Workload(
        name=name or "custom_" + "_".join(f"{k}{v}" for k, v in kv.items()),
        M=kv["M"], N=kv["N"], dtype=kv.get("dtype", "bf16"), eps=kv.get("eps", 1e-6),
        gemma=kv.get("gemma", 0), inplace_dx=kv.get("inplace", 0), seed=kv.get("seed", 0),
        weight_dtype=kv.get("weight", ""), op=op,
        beta=("uniform", 0.0, 1.0) if op == "ln" else None,
        residual=("normal", 0.0, 1.0) if op == "rms_add" else None,
        note="custom shape from the command line")


def run_sweep(args):
    """Per-call forward and backward timing of every workload (not the
    contract line): one JSON line per workload and mapping.  Calls of one
    kind run back to back over k rotating buffer sets, k chosen so the sets
    together exceed three times the L2 (at most 64 sets); CUDA events around
    each loop, average per call.  With --graph the same calls are also
    captured in a CUDA graph and replayed, which leaves out the host's
    per-call enqueue cost (what bounds the smallest shapes).  (In-place
    workloads overwrite dy with dx in every backward call; the timing does
    not depend on the values.)"""
    import numpy as np
    import torch

    import row_wise_normalization_rms_gb300 as rms
    from synthetic import WORKLOADS, make_inputs

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    peak, peak_kind = measured_peaks()
    names = args.workloads.split(",") if args.workloads else list(WORKLOADS)
    custom = {}
    if args.workload_spec:
        cw = workload_from_spec(args.workload_spec)
        custom[cw.name] = cw
        names = [cw.name] if not args.workloads else names + [cw.name]
    paths = args.paths.split(",")
    for name in names:
        w = custom.get(name) or WORKLOADS[name]
        M, N, b = w.M, w.N, w.elem_bytes
        inp = make_inputs(w)

        def dev_t(a, dtype=w.dtype):
            if dtype == "bf16":
                return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
            return torch.from_numpy(a).to(dev)

        set_bytes = 4 * M * N * b
        k = int(min(64, max(1, -(-3 * L2_BYTES // set_bytes))))
        x0, dy0, g = dev_t(inp["x"]), dev_t(inp["dy"]), dev_t(inp["gamma"], w.wdtype)
        ln = w.op == "ln"
        fused = w.op == "rms_add"
        quant = w.op == "rms_quant"
        beta = dev_t(inp["beta"], w.wdtype) if ln and inp["beta"] is not None else None
        if fused:  # residual, h and dh add three matrices per set
            set_bytes = 7 * M * N * b
            k = int(min(64, max(1, -(-3 * L2_BYTES // set_bytes))))
        sets = []
        for i in range(k):
            sets.append((x0 if i == 0 else x0.clone(), dy0 if i == 0 else dy0.clone(),
                         torch.empty_like(x0), torch.empty_like(x0),
                         torch.empty(M, device=dev), torch.empty(M, device=dev)))
        if fused:
            r0, dh0 = dev_t(inp["residual"]), dev_t(inp["dh"])
            extra = [(r0 if i == 0 else r0.clone(), torch.empty_like(x0),
                      dh0 if i == 0 else dh0.clone()) for i in range(k)]
        dg = torch.empty(N, device=dev)
        db = torch.empty(N, device=dev)
        ws_need = rms.ln_bwd_workspace_size(M, N) if ln else rms.rms_bwd_workspace_size(M, N)
        ws = torch.empty(max(256, ws_need), dtype=torch.uint8, device=dev)
        wb = 4 if w.wdtype == "f32" else b
        if ln:
            fwd_b, bwd_b = ln_step_bytes(M, N, b, wb, beta is not None)
        elif fused:
            fwd_b, bwd_b = add_step_bytes(M, N, b, wb)
        elif quant:
            fwd_b, bwd_b = quant_fwd_bytes(M, N, b, wb), 0
            qsets = [(torch.empty(M, N, dtype=torch.uint8, device=dev),
                      torch.empty(M, device=dev)) for _ in range(k)]
        else:
            fwd_b, bwd_b = step_bytes(M, N, b)
        calls = max(args.steps, 2 * k)
        first = True
        for path in paths:
            if ln:
                fpath, bpath = {"vector": ("registers", "staged")}.get(path, (path, path))

                def fwd_call(i):
                    x, dy, y, dx, r, mu = sets[i % k]
                    rms.ln_fwd(x, g, beta, y, mu, r, w.eps, path=fpath)

                def bwd_call(i):
                    x, dy, y, dx, r, mu = sets[i % k]
                    rms.ln_bwd(dy, x, g, mu, r, None if w.inplace_dx else dx, dg, db, ws,
                               w.inplace_dx, path=bpath)
            elif quant:
                def fwd_call(i):
                    x, dy, y, dx, r, _ = sets[i % k]
                    qq, ss = qsets[i % k]
                    rms.rms_fwd_quant(x, g, qq, ss, r, w.eps, w.gemma, path=path)

                bwd_call = None
            elif fused:
                def fwd_call(i):
                    x, dy, y, dx, r, _ = sets[i % k]
                    rr, hh, dh = extra[i % k]
                    rms.rms_fwd_add(x, rr, g, y, hh, r, w.eps, w.gemma, path=path)

                def bwd_call(i):
                    x, dy, y, dx, r, _ = sets[i % k]
                    rr, hh, dh = extra[i % k]
                    rms.rms_bwd_add(dy, hh, g, r, dh, dx, dg, ws, w.gemma, 0, path=path)
            else:
                def fwd_call(i):
                    x, dy, y, dx, r, _ = sets[i % k]
                    rms.rms_fwd(x, g, y, r, w.eps, w.gemma, path=path)

                def bwd_call(i):
                    x, dy, y, dx, r, _ = sets[i % k]
                    rms.rms_bwd(dy, x, g, r, None if w.inplace_dx else dx, dg, ws, w.gemma,
                                w.inplace_dx, path=path)

            def timed(fn, n):
                for i in range(max(3, args.warmup)):
                    fn(i)
                a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                for i in range(n):
                    fn(i)
                z.record()
                torch.cuda.synchronize()
                return a.elapsed_time(z) / n

            def graphed(fn, n, reps=3):
                """The same n calls captured once in a CUDA graph and replayed:
                per-call device time without the host's enqueue cost."""
                side = torch.cuda.Stream()
                side.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(side):
                    for i in range(3):
                        fn(i)
                torch.cuda.current_stream().wait_stream(side)
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr):
                    for i in range(n):
                        fn(i)
                gr.replay()
                torch.cuda.synchronize()
                a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                for _ in range(reps):
                    gr.replay()
                z.record()
                torch.cuda.synchronize()
                return a.elapsed_time(z) / (reps * n)

            fg_ms = bg_ms = None
            try:
                for i in range(k):
                    fwd_call(i)  # every set gets its rstd before the backward loop
                if first:  # the first mapping timed also pays for touching fresh buffers
                    timed(fwd_call, calls)
                    if bwd_call:
                        timed(bwd_call, calls)
                    first = False
                f_ms = timed(fwd_call, calls)
                b_ms = timed(bwd_call, calls) if bwd_call else None
                if args.graph:
                    n_graph = min(calls, max(2 * k, 64))
                    fg_ms = graphed(fwd_call, n_graph)
                    bg_ms = graphed(bwd_call, n_graph) if bwd_call else None
            except rms.RmsError as e:
                print(json.dumps({"workload": name, "path": path, "error": str(e)}), flush=True)
                continue
            fg = fwd_b / (f_ms * 1e-3) / 1e9
            bg = bwd_b / (b_ms * 1e-3) / 1e9 if b_ms else None
            print(json.dumps({
                "workload": name, "op": w.op, "M": M, "N": N, "dtype": w.dtype,
                "weight_dtype": w.wdtype,
                "gemma": w.gemma,
                "inplace_dx": w.inplace_dx, "path": path, "calls": calls, "buffer_sets": k,
                "l2": ("rotating sets exceed 3x L2" if k * set_bytes >= 3 * L2_BYTES
                       else "sets fit in L2: launch-bound shape"),
                "fwd_bytes": fwd_b, "bwd_bytes": bwd_b or None,
                "fwd_rows_per_s": round(M / (f_ms * 1e-3), 1),
                "bwd_rows_per_s": round(M / (b_ms * 1e-3), 1) if b_ms else None,
                "fwd_us": round(f_ms * 1e3, 2), "fwd_gbs": round(fg, 1),
                "fwd_frac": round(fg / peak, 4),
                "bwd_us": round(b_ms * 1e3, 2) if b_ms else None,
                "bwd_gbs": round(bg, 1) if bg else None,
                "bwd_frac": round(bg / peak, 4) if bg else None,
                "graph_fwd_us": round(fg_ms * 1e3, 2) if fg_ms else None,
                "graph_fwd_frac": (round(fwd_b / (fg_ms * 1e-3) / 1e9 / peak, 4) if fg_ms
                                   else None),
                "graph_bwd_us": round(bg_ms * 1e3, 2) if bg_ms else None,
                "graph_bwd_frac": (round(bwd_b / (bg_ms * 1e-3) / 1e9 / peak, 4) if bg_ms
                                   else None),
                "peak_gbs": peak, "peak_source": peak_kind}), flush=True)
        del sets, x0, dy0
        torch.cuda.empty_cache()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shard", default="rows", choices=["rows", "replicas"],
                    help="N > 1: split one batch into row blocks (dgamma exchanged), or run "
                         "replicas")
    ap.add_argument("--sweep", action="store_true",
                    help="per-call timing of every workload instead of the benchmark line")
    ap.add_argument("--workloads", default="", help="comma-separated workload names (--sweep)")
    ap.add_argument("--paths", default="auto", help="comma-separated row mappings (--sweep)")
    ap.add_argument("--workload-spec", default="",
                    help="--sweep: one more workload from key=value pairs, e.g. "
                         "M=4096,N=2048,dtype=f16,eps=1e-5,gemma=0,inplace=0,seed=0,op=rms")
    ap.add_argument("--graph", action="store_true",
                    help="--sweep: also time the calls replayed from a CUDA graph")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.workload_spec:
        if not args.sweep:
            ap.error("--workload-spec goes with --sweep")
        try:
            workload_from_spec(args.workload_spec)
        except ValueError as e:
            ap.error(f"--workload-spec: {e}")
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        if args.steps == 4000:
            args.steps = 50
        return run_sweep(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
