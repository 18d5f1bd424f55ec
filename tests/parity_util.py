"""Runs the CUDA path through the binding and compares it with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import memory_bound_normalization_rmsnorm_gb300 as gb
from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

import oracle
import tolerances


def run_gpu(x, gamma, beta, dy, eps, mode):
    y, rstd, mean = gb.norm_fwd(x, gamma, beta, eps, mode)
    dx, dg, db = gb.norm_bwd(dy, x, gamma, rstd, mean, mode)
    torch.cuda.synchronize()
    return y, rstd, mean, dx, dg, db


def f64(t):
    return t.detach().float().cpu().double().numpy()


def compare(mode, eps, x, gamma, beta, dy, outs, rows=None, label=""):
    """Check all six outputs against the oracle.  `rows` selects the rows
    whose y/dx/rstd/mean are checked (None: all); dgamma/dbeta always use
    every row.  Returns a dict of floor-only pass counts."""
    y, rstd, mean, dx, dg, db = outs
    eps64 = float(np.float32(eps))  # the value the kernels receive
    xb, gb_, db_ = wl.bf16_bits(x), wl.bf16_bits(gamma), wl.bf16_bits(dy)
    bb = None if beta is None else wl.bf16_bits(beta)
    sel = None if rows is None else np.asarray(rows, np.int64)
    y_ref, r_ref, m_ref = oracle.fwd_bf16(xb, gb_, bb, eps64, mode, rows=sel)
    dx_ref = oracle.bwd_dx_bf16(db_, xb, gb_, eps64, mode, rows=sel)
    dg_ref, dbt_ref, dg_abs, dbt_abs = oracle.param_grads_bf16(db_, xb, gb_, eps64, mode)
    if sel is None:
        y_g, dx_g, r_g = f64(y), f64(dx), f64(rstd)
        m_g = None if mean is None else f64(mean)
        xs = oracle.bf16_bits_to_f64(xb)
    else:
        idx = torch.as_tensor(sel, device=y.device)
        y_g, dx_g, r_g = f64(y[idx]), f64(dx[idx]), f64(rstd[idx])
        m_g = None if mean is None else f64(mean[idx])
        xs = oracle.bf16_bits_to_f64(xb[sel])
    counts = {}
    counts["y"] = tolerances.check_t1(y_g, y_ref, f"{label} y")
    counts["dx"] = tolerances.check_t1(dx_g, dx_ref, f"{label} dx")
    tolerances.check_t2(r_g, r_ref, None, f"{label} rstd")
    if mode == wl.LAYER:
        tolerances.check_t2(m_g, m_ref, np.abs(xs).mean(axis=1), f"{label} mean")
        tolerances.check_t2(f64(db), dbt_ref, dbt_abs, f"{label} dbeta")
    else:
        assert mean is None and db is None
    tolerances.check_t2(f64(dg), dg_ref, dg_abs, f"{label} dgamma")
    return counts


def sample_rows(M, n=256, seed=1):
    rng = np.random.default_rng(seed)
    head = np.arange(min(8, M))
    tail = np.arange(max(0, M - 8), M)
    mid = rng.choice(M, size=min(n, M), replace=False)
    return np.unique(np.concatenate([head, mid, tail]))
