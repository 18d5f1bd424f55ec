#!/usr/bin/env python
"""RMSNorm / LayerNorm forward+backward throughput on GB300.

One step = norm_fwd + norm_bwd (three kernel launches: the fused forward,
the fused backward row pass, the fixed-order dgamma/dbeta partial reduce)
over one batch of seeded synthetic bf16 input resident in HBM.  The metric
is achieved HBM bandwidth: the minimal (algorithmic) bytes of the step
divided by its device time.  Minimal bytes per pass, with k = 1 (RMSNorm)
or 2 (LayerNorm) and P the number of partial rows the backward writes:
    forward  4MN + 2kN + 4kM    (read x, gamma[, beta]; write y, rstd[, mean])
    backward 6MN + 2N + 4kM + 4kPN
             (read x, dy, gamma, rstd[, mean]; write dx and the partials)

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
       python bench.py --impl reference ...   (the fp64 CPU oracle, timed)
Under torchrun each rank runs an independent replica of the workload on its
own GPU (rows are independent; no data-path collective) and rank 0 prints
one JSON line.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "RMSNorm/LayerNorm fwd+bwd achieved HBM GB/s and % of GB300 peak per (M,N)"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def algo_bytes(M, N, mode, P, residual=False, fp8=None):
    """Minimal bytes of the forward and backward pass.  The fused residual
    variant adds r read and h written (4MN) to the forward and dh read (2MN)
    to the backward, which reads h where the plain one reads x.  E4M3 output
    (fp8 = 0 per-row scale, 1 MX blocks) writes MN code bytes instead of the
    2MN of bf16 y, plus 4M scale bytes or MN/32 exponent bytes."""
    k = 2 if mode == 1 else 1
    y_bytes = 2 * M * N
    if fp8 is not None:
        y_bytes = M * N + (4 * M if fp8 == 0 else M * N // 32)
    fwd = 2 * M * N + y_bytes + 2 * k * N + 4 * k * M + (4 * M * N if residual else 0)
    bwd = 6 * M * N + 2 * N + 4 * k * M + 4 * k * P * N + (2 * M * N if residual else 0)
    return fwd, bwd


def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The sources each recorded kernel is built from (its translation unit and
# the headers it includes); a traffic record is valid while they are
# unchanged.  Host sources choose and launch kernels but compile to no device
# code: the plan a record was taken with is kept beside its counters instead.
_SHARED = ("common.cuh", "ptx.cuh", "rowops.cuh")
KERNEL_SOURCES = {
    "norm_fwd_kernel": ("fwd.cu", "fwd_kernel.cuh", "tiles.cuh") + _SHARED,
    "norm_bwd_kernel": ("bwd.cu", "tiles.cuh") + _SHARED,
    "norm_gemm_kernel": ("gemm.cu", "tcgen05.cuh") + _SHARED,
}


def source_hash(kernel="norm_bwd_kernel"):
    """Hash of the sources that define `kernel`'s device code."""
    csrc = os.path.join(ROOT, "memory_bound_normalization_rmsnorm_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def _plan_key(p):
    """The fields of a norm_plan dict that decide which kernel a launch runs
    and how it walks the rows."""
    keys = ("cluster", "threads_per_row", "chunks_per_thread", "groups", "rows_per_group",
            "stages", "grid", "exact", "long_rows", "param_smem_bytes")
    return {k: p[k] for k in keys}


def ncu_traffic(workload, kernel, plan=None):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current device code and the same launch plan (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
        rec = data[workload][kernel]
        if rec.get("source_hash") != source_hash(kernel):
            return None
        if plan is not None and rec.get("plan") is not None and rec["plan"] != plan:
            return None
        return rec["bytes_per_launch"]
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "timestamp")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_index)],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            self.rows = []
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        self.rows = rows
        return self.summary(rows)

    @staticmethod
    def _epoch(stamp):
        import datetime

        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp, fmt).timestamp()
            except ValueError:
                pass
        return None

    def window(self, t0, t1):
        """Summary of the samples taken between wall-clock times t0 and t1
        (time.time()); None when no sample fell inside."""
        sel = [r for r in getattr(self, "rows", [])
               if len(r) >= 10 and (e := self._epoch(r[9])) is not None and t0 <= e <= t1]
        return self.summary(sel) if sel else None

    @staticmethod
    def summary(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        # "under load": samples above the median power of the run
        loaded = [s for s, p in zip(sm, pw) if p >= statistics.median(pw)] if pw else sm
        return {"sm_mhz": statistics.median(loaded or sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


def dist_setup(backend="nccl"):
    """One process per GPU under torchrun: (world, rank, local_rank).  Only
    the timing uses the process group (a barrier and a max over ranks): the
    replicas exchange no data."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        if not dist.is_initialized():
            dist.init_process_group(backend)
    return world, rank, local


def aggregate_throughput(step_bytes, steps, ms_per_rank_max, world):
    """Whole-job GB/s: every rank processed `steps` steps of `step_bytes`;
    the job took the slowest rank's time."""
    return world * step_bytes * steps / (ms_per_rank_max * 1e-3) / 1e9


def max_over_ranks(v, world, device):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def gpu_index(local):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",")]
        if local < len(ids) and ids[local].isdigit():
            return int(ids[local])
    return local


# --------------------------------------------------------------- CPU oracle
def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_inputs(w, rows, seed=0):
    """bf16 bits of `rows` rows of the workload's distribution (CPU draw)."""
    from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

    case = wl.like(w, rows, w.N)
    x, g, b, dy = wl.make_inputs(case, "cpu", seed=seed)
    bb = None if b is None else wl.bf16_bits(b)
    return wl.bf16_bits(x), wl.bf16_bits(g), bb, wl.bf16_bits(dy)


def oracle_pass(w, xb, gb_, bb, dyb):
    """The oracle's forward, dx and column sums over the given rows."""
    import oracle

    eps = float(w.eps)
    oracle.fwd_bf16(xb, gb_, bb, eps, w.mode)
    oracle.bwd_dx_bf16(dyb, xb, gb_, eps, w.mode)
    oracle.param_grads_bf16(dyb, xb, gb_, eps, w.mode)


def oracle_sample(w, rows, seed=0):
    """Oracle fwd + dx + column sums on `rows` rows of the workload
    distribution, one thread; returns (seconds, bytes by the same minimal-byte
    formula)."""
    xb, gb_, bb, dyb = oracle_inputs(w, rows, seed)
    t0 = time.perf_counter()
    oracle_pass(w, xb, gb_, bb, dyb)
    dt = time.perf_counter() - t0
    f, bw = algo_bytes(rows, w.N, w.mode, 1)
    return dt, f + bw


def oracle_threads(w, rows, threads, seconds, seed=0):
    """The oracle on every host core: `rows` rows drawn once, cut into one
    block of consecutive rows per thread, each thread running the oracle's
    forward, dx and column sums over its block (the C calls release the
    interpreter lock, so the blocks run in parallel), repeated until about
    `seconds` have passed.  Returns (seconds, bytes, passes)."""
    import concurrent.futures as cf

    import numpy as np

    xb, gb_, bb, dyb = oracle_inputs(w, rows, seed)
    cuts = np.linspace(0, rows, threads + 1).astype(int)
    blocks = [(np.ascontiguousarray(xb[a:b]), np.ascontiguousarray(dyb[a:b]))
              for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
    f, bw = algo_bytes(rows, w.N, w.mode, 1)
    total, passes = 0.0, 0
    with cf.ThreadPoolExecutor(len(blocks)) as ex:
        while total < seconds or passes == 0:
            t0 = time.perf_counter()
            list(ex.map(lambda blk: oracle_pass(w, blk[0], gb_, bb, blk[1]), blocks))
            total += time.perf_counter() - t0
            passes += 1
    return total, passes * (f + bw), passes


def cpu_baseline(w, seconds=12.0, threaded_seconds=8.0):
    """The fp64 oracle as it stands, timed on this host: on every core
    (threads over row blocks; the line's value) and on one thread."""
    import oracle

    oracle.default()
    rows = max(1, min(w.M, (1 << 20) // w.N))
    dt, _ = oracle_sample(w, rows)
    reps_rows = max(1, int(rows * seconds / max(dt, 1e-3)))
    reps_rows = min(reps_rows, w.M)
    total_t, total_b, done = 0.0, 0, 0
    while done < reps_rows:
        r = min(rows, reps_rows - done)
        dt, nb = oracle_sample(w, r, seed=done + 1)
        total_t += dt
        total_b += nb
        done += r
    single = {"value": total_b / total_t / 1e9, "unit": "GB/s", "cores": 1,
              "sample": f"{done} of {w.M} rows x N={w.N} ({w.mode_name}), fwd + dx + column "
                        f"sums, fp64, single thread, {total_t:.1f} s"}
    n = host_cores()
    # rows for the threaded sample: the whole workload, or what ~2 s of the
    # all-core pass covers if that is less (and at least one row per thread)
    per_row = total_t / max(done, 1)
    trows = int(min(w.M, max(n, 2.0 * n / max(per_row, 1e-9))))
    tt, tb, passes = oracle_threads(w, trows, n, threaded_seconds, seed=7)
    return {"value": tb / tt / 1e9, "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"{trows} of {w.M} rows x N={w.N} ({w.mode_name}) x {passes} passes, "
                      f"fwd + dx + column sums, fp64, {n} threads over row blocks, {tt:.1f} s",
            "single_thread": single}


def gemm_cpu_baseline(w0, Nout, seconds=3.0):
    """The fp64 oracle's norm(x) W^T on a bounded sample of rows of the same
    workload (single thread), as TF/s of the same 2 K Nout flops per row."""
    import oracle
    from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

    oracle.default()
    x, g, b, _ = wl.make_inputs(wl.like(w0, 64, w0.N), "cpu", with_dy=False)
    wt = wl.make_gemm_weight(w0, Nout, "cpu")
    xb, gb_, wb = wl.bf16_bits(x), wl.bf16_bits(g), wl.bf16_bits(wt)
    bb = None if b is None or w0.mode == 0 else wl.bf16_bits(b)
    rows, total_t, done = 1, 0.0, 0
    while total_t < seconds and done < 64:
        sel = list(range(done, min(64, done + rows)))
        t0 = time.perf_counter()
        oracle.norm_gemm_bf16(xb, gb_, bb, wb, float(w0.eps), w0.mode, rows=sel)
        total_t += time.perf_counter() - t0
        done += len(sel)
        rows *= 2
    flops = 2.0 * done * w0.N * Nout
    return {"value": flops / total_t / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} rows x K={w0.N} x Nout={Nout} ({w0.mode_name}), fp64 norm then "
                      f"dot products, single thread, {total_t:.1f} s"}


def run_reference(args):
    """The reference arm: the fp64 oracle, as it stands, on every host core
    (threads over row blocks); each step one pass over a bounded sample of
    the workload's rows, sized so the whole run takes about two minutes."""
    world, rank, local = dist_setup()
    from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

    w = wl.WORKLOADS[args.workload]
    if rank != 0:
        barrier(world)
        return
    import oracle

    oracle.default()
    n = host_cores()
    dt, _ = oracle_sample(w, 8)
    per_row = dt / 8 / n  # all cores
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(n, min(w.M, budget / max(per_row, 1e-9))))
    for i in range(args.warmup):
        oracle_threads(w, rows, n, 0.0, seed=1000 + i)
    tt, tb = 0.0, 0
    for i in range(args.steps):
        dt, nb, _ = oracle_threads(w, rows, n, 0.0, seed=i)
        tt += dt
        tb += nb
    value = tb / tt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "mode": w.mode_name, "M": w.M, "N": w.N, "eps": w.eps},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": n, "kind": "oracle",
                         "sample": f"{rows} of {w.M} rows per step, fwd + dx + column sums, "
                                   f"fp64, {n} threads over row blocks"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    barrier(world)


# ------------------------------------------------------------------ GPU arm
class DirectStep:
    """One fwd+bwd step through the C ABI with pre-marshalled arguments (no
    per-call Python tensor checks inside the timed loop).  With `r` and `dh`
    given it runs the fused residual add variant (norm_add_fwd/norm_add_bwd)."""

    def __init__(self, gb, w, x, g, b, dy, stream, r=None, dh=None, fp8=None, fwd_only=False):
        import torch

        M, N = w.M, w.N
        dev = x.device
        self.y = torch.empty_like(x)
        self.dx = torch.empty_like(x)
        self.rstd = torch.empty(M, dtype=torch.float32, device=dev)
        self.mean = torch.empty(M, dtype=torch.float32, device=dev) if w.mode == 1 else None
        self.dg = torch.empty(N, dtype=torch.float32, device=dev)
        self.db = torch.empty(N, dtype=torch.float32, device=dev) if w.mode == 1 else None
        fused = r is not None
        ws_query = gb.norm_add_bwd_workspace_bytes if fused else gb.norm_bwd_workspace_bytes
        nbytes = 16 if fwd_only else ws_query(M, N, w.mode)
        self.ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
        L = gb.lib()
        vp = ctypes.c_void_p

        def p(t):
            return None if t is None else vp(t.data_ptr())

        s = vp(stream.cuda_stream)
        eps = ctypes.c_float(w.eps)
        ws = [p(self.ws), ctypes.c_size_t(self.ws.numel()), s]
        if fused:
            self.h = torch.empty_like(x)
        if fp8 is not None:
            self.q = torch.empty(M, N, dtype=torch.uint8, device=dev)
            self.scale = (torch.empty(M, dtype=torch.float32, device=dev) if fp8 == 0 else
                          torch.empty(M, N // 32, dtype=torch.uint8, device=dev))
            fwd_fp8 = (L.norm_fwd_fp8, [p(x), p(r), p(g), p(b), M, N, eps, w.mode, int(fp8),
                                        p(self.h) if fused else None, p(self.q),
                                        p(self.scale), p(self.rstd), p(self.mean), s])
        if fused:
            self.fwd_args = (L.norm_add_fwd, [p(x), p(r), p(g), p(b), M, N, eps, w.mode,
                                              p(self.h), p(self.y), p(self.rstd),
                                              p(self.mean), s])
            self.bwd_args = (L.norm_add_bwd, [p(dy), p(dh), p(self.h), p(g), p(self.rstd),
                                              p(self.mean), M, N, w.mode, p(self.dx),
                                              p(self.dg), p(self.db)] + ws)
        else:
            self.fwd_args = (L.norm_fwd, [p(x), p(g), p(b), M, N, eps, w.mode, p(self.y),
                                          p(self.rstd), p(self.mean), s])
            self.bwd_args = (L.norm_bwd, [p(dy), p(x), p(g), p(self.rstd), p(self.mean), M,
                                          N, w.mode, p(self.dx), p(self.dg), p(self.db)] + ws)
        if fp8 is not None:
            self.fwd_args = fwd_fp8

    def fwd(self):
        f, a = self.fwd_args
        st = f(*a)
        if st:
            raise RuntimeError(f"norm_fwd status {st}")

    def bwd(self):
        f, a = self.bwd_args
        st = f(*a)
        if st:
            raise RuntimeError(f"norm_bwd status {st}")


def timed_loop(fn, iters, stream):
    """Milliseconds per call of `iters` back-to-back calls of fn, CUDA events
    on `stream` around the whole loop (nothing between the calls)."""
    import torch

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(iters):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def auto_iters(fn, stream, seconds, lo=10, hi=2000):
    """Calls of fn that take about `seconds` (after three warm-up calls)."""
    for _ in range(3):
        fn()
    ms = timed_loop(fn, 5, stream)
    return int(max(lo, min(hi, seconds * 1e3 / max(ms, 1e-4))))


def plan_str(p):
    """Compact text of a norm_plan dict."""
    if p is None:
        return None
    s = (f"C{p['cluster']} tpr{p['threads_per_row']} K{p['chunks_per_thread']} "
         f"G{p['groups']} rpg{p['rows_per_group']} S{p['stages']} grid{p['grid']}")
    if p.get("long_rows"):
        s += " long"
    if p.get("param_smem_bytes"):
        s += " gsm"
    if p.get("split_segments"):
        s += f" split{p['split_segments']}"
    if p.get("streamed"):
        s += " stream"
    return s


def cold_ms(fn, flush, stream, reps):
    """Median time of one call with L2 flushed before it: a buffer larger
    than L2 is written, then CUDA events bracket the call alone."""
    import torch

    times = []
    for i in range(reps):
        flush.fill_(i & 0xff)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times)


def measure_workload(gb, w, peak, seconds=0.15, warmup=3, steps=0, fused=False, fp8=None,
                     fwd_only=False, sampler=None, flush=None, cold_reps=15):
    """Forward, backward and whole-step (forward then backward) throughput of
    one workload: CUDA events around back-to-back calls of each on the
    current stream, inputs resident in HBM (larger than L2 except for the
    1 MB case).  `steps` > 0 fixes the call count, else about `seconds` of
    calls per measurement.  With `flush` (a buffer larger than L2) also the
    median of `cold_reps` calls each run after L2 was flushed."""
    import torch

    from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

    if fused:
        x, r, g, b, dy, dh = wl.make_residual_inputs(w, "cuda")
    else:
        (x, g, b, dy), r, dh = wl.make_inputs(w, "cuda"), None, None
    stream = torch.cuda.current_stream()
    step = DirectStep(gb, w, x, g, b, dy, stream, r=r, dh=dh, fp8=fp8, fwd_only=fwd_only)
    pf = gb.norm_plan(w.M, w.N, w.mode, False, residual=fused, fp8=fp8 is not None)
    pb = None if fwd_only else gb.norm_plan(w.M, w.N, w.mode, True, residual=fused)

    def both():
        step.fwd()
        step.bwd()

    passes = [("fwd", step.fwd)] if fwd_only else [("fwd", step.fwd), ("bwd", step.bwd),
                                                    ("step", both)]
    res, cold = {}, {}
    t0 = time.time()
    for name, fn in passes:
        for _ in range(warmup):
            fn()
        n = steps if steps > 0 else auto_iters(fn, stream, seconds)
        res[name] = timed_loop(fn, n, stream)
        res[name + "_iters"] = n
    t1 = time.time()
    if flush is not None:
        for name, fn in passes:
            cold[name] = cold_ms(fn, flush, stream, cold_reps)
    if gb.norm_get_device_error() != 0:
        raise RuntimeError(f"device error word set on {w.name}")
    P = 0 if pb is None else pb["partials"]
    if pb is not None and pb.get("split_segments"):
        P = P * pb["cols_per_cta"] / w.N  # slots are one segment wide
    fb, bb = algo_bytes(w.M, w.N, w.mode, P, residual=fused, fp8=fp8)
    out = {"workload": w.name, "mode": w.mode_name, "M": w.M, "N": w.N,
           "fwd_us": 1e3 * res["fwd"], "fwd_GBs": fb / res["fwd"] / 1e6,
           "fwd_frac": fb / res["fwd"] / 1e6 / peak, "plan_fwd": plan_str(pf)}
    if pb is not None:
        out.update({"bwd_us": 1e3 * res["bwd"], "bwd_GBs": bb / res["bwd"] / 1e6,
                    "bwd_frac": bb / res["bwd"] / 1e6 / peak,
                    "step_us": 1e3 * res["step"], "step_GBs": (fb + bb) / res["step"] / 1e6,
                    "step_frac": (fb + bb) / res["step"] / 1e6 / peak,
                    "plan_bwd": plan_str(pb), "partials": pb["partials"]})
    out["iters"] = {k[:-6]: v for k, v in res.items() if k.endswith("_iters")}
    if cold:
        nb = {"fwd": fb, "bwd": bb, "step": fb + bb}
        out["cold"] = {f"{k}_frac": nb[k] / ms / 1e6 / peak for k, ms in cold.items()}
        out["cold"]["reps"] = cold_reps
    if sampler is not None:
        out["window"] = (t0, t1)
    del step, x, g, b, dy, r, dh
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import memory_bound_normalization_rmsnorm_gb300 as gb
    from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

    w = wl.WORKLOADS[args.workload]
    if args.rows:
        w = wl.like(w, args.rows, w.N)
    x, g, b, dy = wl.make_inputs(w, dev, seed=w.seed + rank)
    stream = torch.cuda.current_stream(dev)
    step = DirectStep(gb, w, x, g, b, dy, stream)
    plan_f = gb.norm_plan(w.M, w.N, w.mode, False)
    plan_b = gb.norm_plan(w.M, w.N, w.mode, True)
    P = plan_b["partials"]
    fwd_b, bwd_b = algo_bytes(w.M, w.N, w.mode, P)
    peak, peak_kind = peak_hbm()

    sampler = ClockSampler(gpu_index(local))
    sampler.start()
    busy0 = time.time()
    for _ in range(args.warmup):
        step.fwd()
        step.bwd()
    torch.cuda.synchronize()
    if gb.norm_get_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    # The timed region: K steps back to back, CUDA events only at its two
    # ends, so each kernel's launch overlaps the previous one's tail as it
    # does in a training loop.
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        step.fwd()
        step.bwd()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    if gb.norm_get_device_error() != 0:
        raise RuntimeError("device error word set during the timed region")
    total_ms = t0.elapsed_time(t1)
    total_ms_max = max_over_ranks(total_ms, world, dev)
    step_bytes = fwd_b + bwd_b
    value = aggregate_throughput(step_bytes, args.steps, total_ms_max, world)

    # Per-pass durations for the roofline, AFTER the timed region: the
    # forward and the backward call each timed over back-to-back calls of
    # that pass alone (an event between two kernels would hold the second
    # one's launch until the first ends).
    nk = max(20, min(200, args.steps))
    fwd_ms = timed_loop(step.fwd, nk, stream)
    bwd_ms = timed_loop(step.bwd, nk, stream)

    # Cold figure: a 512 MB buffer written before every step evicts the
    # inputs and outputs from L2 (129 MB); events around each step alone.
    cold = None
    if not args.no_cold:
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        times = []
        for i in range(max(5, min(20, args.steps))):
            flush.fill_(i & 0xff)
            a_ = torch.cuda.Event(enable_timing=True)
            b_ = torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            step.fwd()
            step.bwd()
            b_.record(stream)
            torch.cuda.synchronize()
            times.append(a_.elapsed_time(b_))
        del flush
        cms = statistics.median(times)
        cold = {"ms_per_step": cms, "GB/s": step_bytes / cms / 1e6,
                "frac": step_bytes / cms / 1e6 / peak, "reps": len(times),
                "how": "512 MB buffer written before each step; events around that step"}
    busy1 = time.time()
    if gb.norm_get_device_error() != 0:
        raise RuntimeError("device error word set after the per-kernel passes")

    # end to end through the public Python API from pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(gb, w, x, g, b, dy, dev, args.e2e_steps, step_bytes, world, local,
                      fwd_ms + bwd_ms)
    del step, x, g, b, dy
    torch.cuda.empty_cache()

    # Every benchmark workload, one after the other, same process (rank 0 of
    # a single-GPU run only).
    sweep = None
    if world == 1 and not args.no_sweep:
        sweep = []
        flush = None if args.no_cold else torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        for name in wl.ALL:
            e = measure_workload(gb, wl.ALL[name], peak, sampler=sampler, flush=flush)
            if name in wl.WIDE:
                e["beyond_configs"] = "rows wider than one cluster holds in shared memory (streamed or two-pass)"
            sweep.append(e)
    clocks_all = sampler.stop()
    clocks = sampler.window(busy0, busy1) or clocks_all
    if sweep is not None:
        for e in sweep:
            c = sampler.window(*e.pop("window"))
            e["sm_mhz"] = None if c is None else c["sm_mhz"]

    bwd_gbs = bwd_b / (bwd_ms * 1e-3) / 1e9
    fwd_gbs = fwd_b / (fwd_ms * 1e-3) / 1e9
    traffic = ncu_traffic(w.name, "norm_bwd_kernel", plan=_plan_key(plan_b))
    roofline = {"bound": "hbm", "achieved": bwd_gbs, "peak": peak, "unit": "GB/s",
                "frac": bwd_gbs / peak, "traffic": traffic,
                "kernel": "norm_bwd (fused row kernel + fixed-order partial reduce)",
                "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "bytes_per_launch": bwd_b, "launch_ms": bwd_ms,
                "timing": f"{nk} back-to-back norm_bwd calls after the timed region"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "mode": w.mode_name, "M": w.M, "N": w.N,
                       "eps": w.eps, "io_dtype": "bf16", "accumulate": "fp32",
                       "parallelism": f"replicas x{world} (rows independent)",
                       "l2": "inputs larger than L2 (each of x, dy, y, dx is "
                             f"{w.M * w.N * 2 / 1e6:.0f} MB > 129 MB); no flush in the timed "
                             "region (a flushed figure is under 'cold')",
                       "kernel_timing": f"timed region: {args.steps} back-to-back steps, "
                                        "events at its ends only; per-pass times from "
                                        f"{nk} back-to-back calls of each pass afterwards",
                       "plan_fwd": plan_f, "plan_bwd": plan_b},
            "pct_of_nominal_8TBs": 100.0 * value / world / NOMINAL_HBM_GBS,
            "pct_of_measured_peak": 100.0 * value / world / peak,
            "fwd": {"ms": fwd_ms, "GB/s": fwd_gbs, "frac": fwd_gbs / peak, "bytes": fwd_b},
            "bwd": {"ms": bwd_ms, "GB/s": bwd_gbs, "frac": bwd_gbs / peak, "bytes": bwd_b,
                    "partials": P},
            "cold": cold,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": 3 * args.steps,
            "clocks": clocks,
            "sweep": sweep,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def gpu_host_locality(local):
    """The GPU's PCI address and, from sysfs, the NUMA node and CPU list the
    kernel reports as local to it (None where unknown)."""
    import torch

    info = {"pci": None, "numa_node": None, "local_cpus": None}
    try:
        pr = torch.cuda.get_device_properties(local)
        info["pci"] = f"{pr.pci_domain_id:04x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
    except Exception:
        try:
            out = subprocess.run(["nvidia-smi", "--query-gpu=pci.bus_id", "--format=csv,noheader",
                                  "-i", str(gpu_index(local))], capture_output=True, text=True,
                                 timeout=20).stdout.strip()
            dom, rest = out.split(":", 1)
            info["pci"] = f"{int(dom, 16):04x}:{rest.lower()}"
        except Exception:
            return info
    base = f"/sys/bus/pci/devices/{info['pci']}"
    try:
        with open(base + "/numa_node") as f:
            info["numa_node"] = int(f.read().strip())
    except Exception:
        pass
    try:
        with open(base + "/local_cpulist") as f:
            cpus = set()
            for part in f.read().strip().split(","):
                if "-" in part:
                    a, b = part.split("-")
                    cpus.update(range(int(a), int(b) + 1))
                elif part:
                    cpus.add(int(part))
            info["local_cpus"] = sorted(cpus)
    except Exception:
        pass
    return info


def pages_by_node(addr):
    """NUMA node -> pages of the mapping that holds host address `addr`,
    from /proc/self/numa_maps (None where the kernel does not say)."""
    try:
        start = None
        with open("/proc/self/maps") as f:
            for line in f:
                a, b = line.split()[0].split("-")
                if int(a, 16) <= addr < int(b, 16):
                    start = a
                    break
        if start is None:
            return None
        with open("/proc/self/numa_maps") as f:
            for line in f:
                if line.split()[0].lstrip("0") == start.lstrip("0"):
                    nodes = {}
                    for tok in line.split()[1:]:
                        if tok.startswith("N") and "=" in tok:
                            k, v = tok[1:].split("=")
                            if k.isdigit():
                                nodes[int(k)] = int(v)
                    return nodes or None
    except Exception:
        return None
    return None


def run_e2e(gb, w, x, g, b, dy, dev, steps, step_bytes, world, local, kernel_ms):
    """Per step one norm_fwd_bwd_host call: host (pinned) x, dy, gamma(,
    beta) in; y, rstd(, mean), dx, dgamma(, dbeta) back in pinned host
    buffers.  The library streams the rows through device buffers in chunks
    with both copy directions and the kernels overlapped; timed with CUDA
    events on the calling stream around the whole step.  The pinned buffers
    are allocated from a thread bound to the CPUs local to the GPU (when
    sysfs names them), so their pages sit on the GPU's side of the host;
    the line records where they landed and what single copies of the same
    buffers achieve, and from those the copy-bound time of a step."""
    import torch

    loc = gpu_host_locality(local)
    old_aff = None
    bound = False
    if loc["local_cpus"]:
        try:
            old_aff = os.sched_getaffinity(0)
            use = set(loc["local_cpus"]) & set(old_aff)
            if use:
                os.sched_setaffinity(0, use)
                bound = True
        except Exception:
            old_aff = None
    try:
        hx = x.cpu().pin_memory()
        hdy = dy.cpu().pin_memory()
        hg = g.cpu().pin_memory()
        hb = None if b is None else b.cpu().pin_memory()
        M, N = w.M, w.N
        ln = w.mode == 1
        out = (torch.empty(M, N, dtype=torch.bfloat16, pin_memory=True),
               torch.empty(M, dtype=torch.float32, pin_memory=True),
               torch.empty(M, dtype=torch.float32, pin_memory=True) if ln else None,
               torch.empty(M, N, dtype=torch.bfloat16, pin_memory=True),
               torch.empty(N, dtype=torch.float32, pin_memory=True),
               torch.empty(N, dtype=torch.float32, pin_memory=True) if ln else None)
        ws = torch.empty(gb.norm_host_workspace_bytes(M, N, w.mode), dtype=torch.uint8,
                         device=dev)
        h2d = sum(t.numel() * t.element_size() for t in (hx, hdy, hg, hb) if t is not None)
        d2h = sum(t.numel() * t.element_size() for t in out if t is not None)

        def one():
            gb.norm_fwd_bwd_host(hx, hdy, hg, hb, w.eps, w.mode, out=out, workspace=ws)

        one()
        torch.cuda.synchronize()
        # three trials of `steps` calls each, the median reported: the host
        # links are shared with other jobs on the machine, and one trial has
        # been seen at half the rate of the trials around it
        trials = []
        for _ in range(3):
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record()
            for _ in range(steps):
                one()
            s1.record()
            torch.cuda.synchronize()
            trials.append(s0.elapsed_time(s1))
        ms = max_over_ranks(statistics.median(trials), world, dev)

        # single copies of the same pinned buffers: x in, dx out, and both at
        # once on two streams
        dbuf = torch.empty_like(x)
        dbuf2 = torch.empty_like(x)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def copy_ms(fns, reps=3):
            best = None
            for _ in range(reps):
                torch.cuda.synchronize()
                t = time.perf_counter()
                for st, fn in fns:
                    with torch.cuda.stream(st):
                        fn()
                torch.cuda.synchronize()
                dt = (time.perf_counter() - t) * 1e3
                best = dt if best is None else min(best, dt)
            return best

        nbytes = hx.numel() * 2
        h2d_ms = copy_ms([(s_in, lambda: dbuf.copy_(hx, non_blocking=True))])
        d2h_ms = copy_ms([(s_out, lambda: out[3].copy_(dbuf2, non_blocking=True))])
        both_ms = copy_ms([(s_in, lambda: dbuf.copy_(hx, non_blocking=True)),
                           (s_out, lambda: out[3].copy_(dbuf2, non_blocking=True))])
        h2d_gbs = nbytes / h2d_ms / 1e6
        d2h_gbs = nbytes / d2h_ms / 1e6
        both_gbs = 2 * nbytes / both_ms / 1e6
        # copy-bound model of one step: the bytes of both directions at the
        # rate the two directions reach together, or the kernels, whichever
        # is longer
        model_ms = max((h2d + d2h) / both_gbs / 1e6, kernel_ms)
        placement = {"x_pages_by_node": pages_by_node(hx.data_ptr()),
                     "dx_pages_by_node": pages_by_node(out[3].data_ptr())}
        del dbuf, dbuf2
    finally:
        if old_aff is not None:
            try:
                os.sched_setaffinity(0, old_aff)
            except Exception:
                pass
    return {"value": world * step_bytes * steps / (ms * 1e-3) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms / steps,
            "steps": steps, "trials_ms_per_step": [t / steps for t in trials],
            "api": "norm_fwd_bwd_host (host tensors, chunked, copies overlapped)",
            "h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs, "both_directions_gbs": both_gbs,
            "copy_bound_model_ms": model_ms,
            "vs_model": model_ms / (ms / steps),
            "gpu_locality": {"pci": loc["pci"], "numa_node": loc["numa_node"],
                             "local_cpus": (f"{loc['local_cpus'][0]}-{loc['local_cpus'][-1]}"
                                            if loc["local_cpus"] else None),
                             "pinned_from_local_cpus": bound},
            "placement": placement}


def run_sweep(args):
    """One JSON line per workload: fwd and bwd timed separately and the whole
    step (CUDA events around back-to-back calls of each on the default
    stream, inputs resident in HBM and larger than L2 except for the small
    case)."""
    import torch

    import memory_bound_normalization_rmsnorm_gb300 as gb
    from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

    torch.cuda.set_device(0)
    peak, peak_kind = peak_hbm()
    names = (list(wl.WORKLOADS) if args.sweep == "all" else
             list(wl.WIDE) if args.sweep == "wide" else args.sweep.split(","))
    fp8 = {"": None, "row": 0, "mx": 1}[args.fp8]
    for name in names:
        w = wl.ALL[name]
        if args.rows or args.cols:
            w = wl.like(w, args.rows or w.M, args.cols or w.N)
        line = measure_workload(gb, w, peak, warmup=args.warmup, steps=args.steps,
                                fused=args.fused_residual, fp8=fp8, fwd_only=args.fwd_only)
        line.update({"fused_residual": args.fused_residual, "fp8": args.fp8 or None,
                     "peak": peak, "peak_kind": peak_kind})
        print(json.dumps(line), flush=True)


def run_ablate(args):
    """The two knobs the first page tunes for the backward pass, on one
    workload's backward call: the number of partial rows (split size; the
    persistent grid is capped with GBNORM_PLAN grid=P) and the number of
    pipeline stages (GBNORM_PLAN S=n).  One JSON line per setting."""
    import torch

    import memory_bound_normalization_rmsnorm_gb300 as gb
    from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

    torch.cuda.set_device(0)
    peak, _ = peak_hbm()
    w = wl.WORKLOADS[args.workload]
    x, g, b, dy = wl.make_inputs(w, "cuda")
    stream = torch.cuda.current_stream()
    # partial rows: the persistent grid capped below one CTA per SM, the
    # default, and two smaller CTAs (one row group) per SM; stages: tiles of
    # one row per group (half the default tile) so that up to 6 fit
    settings = [("grid", f"grid={p}") for p in (19, 38, 76, 114)]
    settings += [("grid", ""), ("grid", "G=1,rpg=1,S=3,ctas=2")]
    settings += [("stages", f"rpg=1,S={k}") for k in range(2, 8)]
    for kind, ov in settings:
        if ov:
            os.environ["GBNORM_PLAN"] = ov
        try:
            step = DirectStep(gb, w, x, g, b, dy, stream)
            pb = gb.norm_plan(w.M, w.N, w.mode, True)
            step.fwd()
            for _ in range(args.warmup):
                step.bwd()
            ms = timed_loop(step.bwd, max(20, args.steps), stream)
        except Exception as e:  # a setting the planner cannot schedule
            print(json.dumps({"workload": w.name, "knob": kind, "override": ov,
                              "error": str(e)}), flush=True)
            continue
        finally:
            os.environ.pop("GBNORM_PLAN", None)
        if gb.norm_get_device_error() != 0:
            raise RuntimeError(f"device error word set under {ov}")
        _, bb = algo_bytes(w.M, w.N, w.mode, pb["partials"])
        print(json.dumps({"workload": w.name, "knob": kind, "override": ov,
                          "partials": pb["partials"], "rows_per_partial": w.M / pb["partials"],
                          "stages": pb["stages"], "plan": plan_str(pb), "bwd_us": 1e3 * ms,
                          "bwd_GBs": bb / ms / 1e6, "bwd_frac": bb / ms / 1e6 / peak}),
              flush=True)
        del step
        torch.cuda.empty_cache()


def peak_bf16():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


NORM_GEMM_CASES = [(mode, 32768, k, k) for mode in (0, 1) for k in (2048, 3072, 4096, 5120, 8192)]


def run_norm_gemm(args):
    """One JSON line per (mode, M, K, Nout): the fused normalisation-GEMM
    (norm_gemm_fwd, weights prepared once) against the unfused sequence
    norm_fwd + cuBLAS bf16 GEMM (torch.matmul) on the same inputs, each timed
    with CUDA events around back-to-back calls on the current stream.  The
    roofline is the tensor-core one: 2 M K Nout flops per call against the
    measured cuBLAS bf16 burst peak."""
    import torch

    import memory_bound_normalization_rmsnorm_gb300 as gb
    from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

    torch.cuda.set_device(0)
    peak, peak_kind = peak_bf16()
    cases = NORM_GEMM_CASES
    if args.norm_gemm != "all":
        k = int(args.norm_gemm)
        cases = [c for c in cases if c[2] == k]

    def timed(fn):
        # About 0.3 s of calls (at most --steps), so that the clock samples
        # fall inside the timed region.
        t0 = time.perf_counter()
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        per = (time.perf_counter() - t0) / args.warmup
        iters = max(1, min(args.steps, int(0.3 / max(per, 1e-6))))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / iters, iters

    for mode, M, K, Nout in cases:
        w0 = wl.Workload(f"norm_gemm_{'rms' if mode == 0 else 'layer'}_{M}x{K}x{Nout}", mode, M,
                         K, 1e-5, "normal_offset", "one_plus_0.1n")
        x, g, b, _ = wl.make_inputs(w0, "cuda", with_dy=False)
        b = b if mode == 1 else None
        w = wl.make_gemm_weight(w0, Nout, "cuda")
        wg, u, v = gb.norm_gemm_prepare(w, g, b, mode)
        out, rstd, mean = gb.norm_gemm_fwd(x, wg, u, v, 1e-5, mode)
        y, r2, m2 = gb.norm_fwd(x, g, b, 1e-5, mode)
        prod = torch.empty(M, Nout, dtype=torch.bfloat16, device="cuda")
        wt = w.t()
        clk = ClockSampler(0)
        clk.start()
        t_fused, iters = timed(lambda: gb.norm_gemm_fwd(x, wg, u, v, 1e-5, mode, out=out,
                                                        rstd=rstd, mean=mean))
        clocks = clk.stop()
        t_norm, _ = timed(lambda: gb.norm_fwd(x, g, b, 1e-5, mode, y=y, rstd=r2, mean=m2))
        t_gemm, _ = timed(lambda: torch.matmul(y, wt, out=prod))

        def unfused():
            gb.norm_fwd(x, g, b, 1e-5, mode, y=y, rstd=r2, mean=m2)
            torch.matmul(y, wt, out=prod)

        t_unfused, _ = timed(unfused)
        if gb.norm_get_device_error() != 0:
            raise RuntimeError(f"device error word set on {w0.name}")
        flops = 2.0 * M * K * Nout
        achieved = flops / (t_fused * 1e-3) / 1e12
        line = {"workload": w0.name, "mode": w0.mode_name, "M": M, "K": K, "Nout": Nout,
                "dtype": "bf16 in, fp32 accumulate, bf16 out", "iters": iters,
                "fused_us": 1e3 * t_fused, "fused_tflops": achieved,
                "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                             "unit": "TFLOP/s", "frac": achieved / peak,
                             "peak_kind": f"cuBLAS bf16 burst, {peak_kind}",
                             "traffic": ncu_traffic(w0.name, "norm_gemm_kernel")},
                "unfused_us": 1e3 * t_unfused, "norm_fwd_us": 1e3 * t_norm,
                "cublas_us": 1e3 * t_gemm, "cublas_tflops": flops / (t_gemm * 1e-3) / 1e12,
                "speedup_vs_unfused": t_unfused / t_fused,
                "norm_time_hidden_frac": (t_unfused - t_fused) / t_norm,
                "clocks": clocks}
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = gemm_cpu_baseline(w0, Nout)
        print(json.dumps(line), flush=True)
        del x, g, b, w, wg, u, v, out, rstd, mean, y, r2, m2, prod
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="layer_32768x4096")
    ap.add_argument("--rows", type=int, default=0,
                    help="override M (smaller cases for profiling captures only; also "
                         "with --sweep)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cold", action="store_true",
                    help="skip the L2-flushed per-step figure")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the per-workload sweep in the benchmark line")
    ap.add_argument("--ablate", action="store_true",
                    help="partial-row count and stage count of the backward pass on "
                         "--workload, one JSON line per setting (not the benchmark line)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cols", type=int, default=0,
                    help="with --sweep: row length of the workload (same distributions)")
    ap.add_argument("--sweep", default="",
                    help="'all', 'wide' or comma-separated workload names: per-workload "
                         "fwd/bwd timings, one JSON line each (not the benchmark line)")
    ap.add_argument("--fused-residual", action="store_true",
                    help="with --sweep: time norm_add_fwd/norm_add_bwd (h = x + r fused in)")
    ap.add_argument("--fwd-only", action="store_true",
                    help="with --sweep: time the forward pass only")
    ap.add_argument("--fp8", choices=["", "row", "mx"], default="",
                    help="with --sweep: the forward writes E4M3 (norm_fwd_fp8) with per-row "
                         "or MX block scaling")
    ap.add_argument("--norm-gemm", default="",
                    help="'all' or one K: the normalisation fused into the tcgen05 GEMM "
                         "against norm_fwd + cuBLAS, one JSON line per case")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.ablate:
        run_ablate(args)
    elif args.norm_gemm:
        run_norm_gemm(args)
    elif args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
