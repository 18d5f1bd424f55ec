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


# Host-only sources: they choose and launch kernels but compile to no device
# code; the plan they chose is recorded beside the counters instead.
HOST_ONLY_SOURCES = ("api.cu", "host.cu")
# The normalisation-GEMM's own sources (its kernels are in gemm.cu alone),
# and the shared headers that gemm.cu also includes.
NORM_GEMM_SOURCES = ("gemm.cu", "tcgen05.cuh")
NORM_GEMM_HEADERS = ("common.cuh", "ptx.cuh", "rowops.cuh")


def source_hash(kind="norm"):
    """Hash of the sources that define the device code of the normalisation
    kernels (kind "norm") or of the normalisation-GEMM kernel ("gemm")."""
    csrc = os.path.join(ROOT, "memory_bound_normalization_rmsnorm_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        if kind == "norm" and (name in HOST_ONLY_SOURCES or name in NORM_GEMM_SOURCES):
            continue
        if kind == "gemm" and name not in NORM_GEMM_SOURCES + NORM_GEMM_HEADERS:
            continue
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def _plan_key(p):
    """The fields of a norm_plan dict that decide which kernel a launch runs
    and how it walks the rows."""
    keys = ("cluster", "threads_per_row", "chunks_per_thread", "groups", "rows_per_group",
            "stages", "grid", "exact", "long_rows", "param_smem_bytes")
    return {k: p[k] for k in keys}


def ncu_traffic(workload, kernel, plan=None, kind="norm"):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current device code and the same launch plan (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
        rec = data[workload][kernel]
        if rec.get("source_hash") != source_hash(kind):
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
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

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
def oracle_sample(w, rows, seed=0):
    """Oracle fwd + dx + column sums on the first `rows` rows of the workload
    distribution; returns (seconds, bytes by the same minimal-byte formula)."""
    import oracle
    from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

    case = wl.like(w, rows, w.N)
    x, g, b, dy = wl.make_inputs(case, "cpu", seed=seed)
    xb, gb_, dyb = wl.bf16_bits(x), wl.bf16_bits(g), wl.bf16_bits(dy)
    bb = None if b is None else wl.bf16_bits(b)
    eps = float(w.eps)
    t0 = time.perf_counter()
    oracle.fwd_bf16(xb, gb_, bb, eps, w.mode)
    oracle.bwd_dx_bf16(dyb, xb, gb_, eps, w.mode)
    oracle.param_grads_bf16(dyb, xb, gb_, eps, w.mode)
    dt = time.perf_counter() - t0
    f, bw = algo_bytes(rows, w.N, w.mode, 1)
    return dt, f + bw


def cpu_baseline(w, seconds=12.0):
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
    return {"value": total_b / total_t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} of {w.M} rows x N={w.N} ({w.mode_name}), fwd + dx + column "
                      f"sums, fp64, single thread, {total_t:.1f} s"}


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
    world, rank, local = dist_setup()
    from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

    w = wl.WORKLOADS[args.workload]
    if rank != 0:
        barrier(world)
        return
    import oracle

    oracle.default()
    # size one step so that warmup + steps take about two minutes in all
    dt, _ = oracle_sample(w, 8)
    per_row = dt / 8
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(w.M, budget / max(per_row, 1e-9))))
    for i in range(args.warmup):
        oracle_sample(w, rows, seed=1000 + i)
    tt, tb = 0.0, 0
    for i in range(args.steps):
        dt, nb = oracle_sample(w, rows, seed=i)
        tt += dt
        tb += nb
    value = tb / tt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "mode": w.mode_name, "M": w.M, "N": w.N, "eps": w.eps},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{rows} of {w.M} rows per step, fwd + dx + column sums, "
                                   f"fp64, single thread"},
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

    sampler = ClockSampler(gpu_index(local))
    sampler.start()
    for _ in range(args.warmup):
        step.fwd()
        step.bwd()
    torch.cuda.synchronize()
    if gb.norm_get_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    # Per-kernel durations (for the roofline) come from CUDA events around the
    # forward and the backward call of the first `nev` timed steps.  An event
    # recorded between two kernels makes the second wait for the first to
    # finish (no programmatic overlap of its launch with the first's tail),
    # which on every step would slow the step by ~5 %; the remaining steps
    # run back to back, as a training loop runs them.
    nev = min(args.steps, 50)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nev)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        if i < nev:
            ev[i][0].record(stream)
            step.fwd()
            ev[i][1].record(stream)
            step.bwd()
            ev[i][2].record(stream)
        else:
            step.fwd()
            step.bwd()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    if gb.norm_get_device_error() != 0:
        raise RuntimeError("device error word set during the timed region")

    total_ms = t0.elapsed_time(t1)
    total_ms_max = max_over_ranks(total_ms, world, dev)
    fwd_ms = statistics.fmean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.fmean(e[1].elapsed_time(e[2]) for e in ev)
    step_bytes = fwd_b + bwd_b
    value = aggregate_throughput(step_bytes, args.steps, total_ms_max, world)

    # end to end through the public Python API from pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(gb, w, x, g, b, dy, dev, args.e2e_steps, fwd_b + bwd_b, world)

    peak, peak_kind = peak_hbm()
    bwd_gbs = bwd_b / (bwd_ms * 1e-3) / 1e9
    fwd_gbs = fwd_b / (fwd_ms * 1e-3) / 1e9
    traffic = ncu_traffic(w.name, "norm_bwd_kernel", plan=_plan_key(plan_b))
    roofline = {"bound": "hbm", "achieved": bwd_gbs, "peak": peak, "unit": "GB/s",
                "frac": bwd_gbs / peak, "traffic": traffic,
                "kernel": "norm_bwd (fused row kernel + fixed-order partial reduce)",
                "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "bytes_per_launch": bwd_b, "launch_ms": bwd_ms}
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
                             f"{w.M * w.N * 2 / 1e6:.0f} MB > 129 MB); no flush",
                       "kernel_timing": f"CUDA events around the forward and the backward "
                                        f"call of the first {nev} of the {args.steps} timed steps",
                       "plan_fwd": plan_f, "plan_bwd": plan_b},
            "pct_of_nominal_8TBs": 100.0 * value / world / NOMINAL_HBM_GBS,
            "pct_of_measured_peak": 100.0 * value / world / peak,
            "fwd": {"ms": fwd_ms, "GB/s": fwd_gbs, "frac": fwd_gbs / peak, "bytes": fwd_b},
            "bwd": {"ms": bwd_ms, "GB/s": bwd_gbs, "frac": bwd_gbs / peak, "bytes": bwd_b,
                    "partials": P},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": 3 * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def run_e2e(gb, w, x, g, b, dy, dev, steps, step_bytes, world):
    """Per step one norm_fwd_bwd_host call: host (pinned) x, dy, gamma(,
    beta) in; y, rstd(, mean), dx, dgamma(, dbeta) back in pinned host
    buffers.  The library streams the rows through device buffers in chunks
    with both copy directions and the kernels overlapped; timed with CUDA
    events on the calling stream around the whole step."""
    import torch

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
    ws = torch.empty(gb.norm_host_workspace_bytes(M, N, w.mode), dtype=torch.uint8, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in (hx, hdy, hg, hb) if t is not None)
    d2h = sum(t.numel() * t.element_size() for t in out if t is not None)

    def one():
        gb.norm_fwd_bwd_host(hx, hdy, hg, hb, w.eps, w.mode, out=out, workspace=ws)

    one()
    torch.cuda.synchronize()
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(steps):
        one()
    s1.record()
    torch.cuda.synchronize()
    ms = s0.elapsed_time(s1)
    ms = max_over_ranks(ms, world, dev)
    return {"value": world * step_bytes * steps / (ms * 1e-3) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms / steps,
            "steps": steps, "api": "norm_fwd_bwd_host (host tensors, chunked, copies overlapped)"}


def run_sweep(args):
    """One JSON line per workload: fwd and bwd timed separately (CUDA events
    around `iters` back-to-back calls of each pass on the default stream,
    inputs resident in HBM and larger than L2 except for the small case)."""
    import torch

    import memory_bound_normalization_rmsnorm_gb300 as gb
    from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

    torch.cuda.set_device(0)
    peak, peak_kind = peak_hbm()
    names = list(wl.WORKLOADS) if args.sweep == "all" else args.sweep.split(",")
    for name in names:
        w = wl.WORKLOADS[name]
        fused = args.fused_residual
        fp8 = {"": None, "row": 0, "mx": 1}[args.fp8]
        if fused:
            x, r, g, b, dy, dh = wl.make_residual_inputs(w, "cuda")
        else:
            (x, g, b, dy), r, dh = wl.make_inputs(w, "cuda"), None, None
        step = DirectStep(gb, w, x, g, b, dy, torch.cuda.current_stream(), r=r, dh=dh, fp8=fp8,
                          fwd_only=args.fwd_only)
        pf = gb.norm_plan(w.M, w.N, w.mode, False, residual=fused, fp8=fp8 is not None)
        pb = None if args.fwd_only else gb.norm_plan(w.M, w.N, w.mode, True, residual=fused)
        res = {}
        passes = (("fwd", step.fwd),) if args.fwd_only else (("fwd", step.fwd), ("bwd", step.bwd))
        for name_, fn in passes:
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.steps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            res[name_] = e0.elapsed_time(e1) / args.steps
        if gb.norm_get_device_error() != 0:
            raise RuntimeError(f"device error word set on {name}")
        fb, bb = algo_bytes(w.M, w.N, w.mode, 0 if pb is None else pb["partials"],
                            residual=fused, fp8=fp8)
        keep = ("cluster", "threads_per_row", "chunks_per_thread", "groups", "rows_per_group",
                "stages", "grid", "exact")
        line = {"workload": w.name, "mode": w.mode_name, "M": w.M, "N": w.N,
                "fused_residual": fused, "fp8": args.fp8 or None, "fwd_us": 1e3 * res["fwd"],
                "fwd_GBs": fb / res["fwd"] / 1e6, "peak": peak, "peak_kind": peak_kind,
                "iters": args.steps, "plan_fwd": {k: pf[k] for k in keep}}
        if pb is not None:
            line.update({"bwd_us": 1e3 * res["bwd"], "bwd_GBs": bb / res["bwd"] / 1e6,
                         "step_GBs": (fb + bb) / (res["fwd"] + res["bwd"]) / 1e6,
                         "step_frac": (fb + bb) / (res["fwd"] + res["bwd"]) / 1e6 / peak,
                         "plan_bwd": {k: pb[k] for k in keep}})
        print(json.dumps(line), flush=True)
        del step, x, g, b, dy, r, dh
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
                             "traffic": ncu_traffic(w0.name, "norm_gemm_kernel", kind="gemm")},
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
                    help="override M (smaller cases for profiling captures only)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sweep", default="",
                    help="'all' or comma-separated workload names: per-workload fwd/bwd "
                         "timings, one JSON line each (not the benchmark line)")
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
    if args.norm_gemm:
        run_norm_gemm(args)
    elif args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
