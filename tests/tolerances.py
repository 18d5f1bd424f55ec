"""Comparison rules between the CUDA path and the fp64 oracle.

T1 (bf16 outputs y, dx), element-wise:
    |gpu - ref| <= max(2 * ulp_bf16(ref), 1e-2 * |ref|, 2**-16 * max_row|ref|)
  ulp_bf16(r) = 2**(floor(log2|r|) - 7) on the fp64 reference.  The first
  two terms are the stated bound; the third, row-scaled floor covers
  elements whose reference is ~1e-5 of the row's scale, where fp32
  cancellation (in y = xhat*gamma + beta, and in dx) leaves an absolute
  error of ~1e-7 of the row scale that no relative bound can absorb.  The
  number of elements passing only through the floor is returned and must
  stay below 1e-5 of all elements.
T2 (fp32 outputs rstd, mean, dgamma, dbeta):
    |gpu - ref| <= 1e-3 * |ref| + 1e-6 * S
  S = the oracle's sum of |summands| of that reduction (|x|/N summed for the
  mean, |dy * xhat| over rows for dgamma, |dy| over rows for dbeta; 0 for
  rstd, which has no cancellation).
"""
from __future__ import annotations

import numpy as np


def ulp_bf16(ref):
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 7), 0.0)


def check_t1(gpu, ref, name="", floor_frac=1e-5):
    """gpu, ref: float64 arrays [R, N].  Returns the count of floor-only
    passes; raises AssertionError on any violation."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    err = np.abs(gpu - ref)
    strict = np.maximum(2.0 * ulp_bf16(ref), 1e-2 * np.abs(ref))
    rowmax = np.abs(ref).max(axis=1, keepdims=True)
    bound = np.maximum(strict, 2.0 ** -16 * rowmax)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        msg = "; ".join(f"[{i},{j}] gpu={gpu[i, j]!r} ref={ref[i, j]!r} bound={bound[i, j]:.3g}"
                        for i, j in idx)
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} elements out of "
                             f"tolerance: {msg}")
    floor_only = int(((err > strict) & ~bad).sum())
    limit = max(2, int(floor_frac * err.size))
    assert floor_only <= limit, f"{name}: {floor_only} elements pass only by the floor"
    return floor_only


def check_t2(gpu, ref, scale=None, name=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    s = 0.0 if scale is None else np.asarray(scale, np.float64)
    bound = 1e-3 * np.abs(ref) + 1e-6 * s
    err = np.abs(gpu - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad.reshape(-1))[:5, 0]
        g, r, b = gpu.reshape(-1), ref.reshape(-1), np.broadcast_to(bound, ref.shape).reshape(-1)
        msg = "; ".join(f"[{i}] gpu={g[i]!r} ref={r[i]!r} bound={b[i]:.3g}" for i in idx)
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} out of tolerance: {msg}")


def check_t4(gpu, ref, x, gamma, beta, w, rstd, mean, name=""):
    """T4, the normalisation-GEMM out = norm(x) W^T (bf16 out [R, Nout]).

    The kernel computes rstd * (x W'^T - mean * u) + v with W' = bf16(W *
    gamma), fp32 accumulation, and rounds the result to bf16.  With
    tau_j = xhat_j * gamma_j * W_kj (the exact terms) and u_b = 2^-8 (bf16
    unit roundoff), each element obeys the worst-case bound
        |gpu - ref| <= (u_b + 2^-20) |ref| + u_b * sum_j |tau_j|
                       + K 2^-23 * (rstd (sum_j |x_j gamma_j W_kj|
                                          + |mean| sum_j |gamma_j W_kj|)
                                    + sum_j |beta_j W_kj| + |ref - v_k|)
    (output rounding; W' rounding, at most u_b per term; fp32 sums of K
    terms, in the contraction, in u, v and the row statistics).  The bound is
    loose for random signs, so the RMS error over all elements is also held
    to 1.5x its expected size, sqrt(u_b^2 / 3 * mean(sum_j tau_j^2 + ref^2))
    (independent rounding errors, each at most u_b relative).

    x: float64 [R, K] (the bf16 rows), gamma/beta float64 [K] (beta may be
    None), w float64 [Nout, K]; rstd/mean: the oracle's fp64 statistics [R].
    """
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    K = x.shape[1]
    ub = 2.0 ** -8
    mu = np.zeros(x.shape[0]) if mean is None else np.asarray(mean, np.float64)
    r = np.asarray(rstd, np.float64)
    xhat = (x - mu[:, None]) * r[:, None]
    gw = np.abs(w * gamma[None, :])                      # |gamma_j W_kj|
    A = np.abs(xhat) @ gw.T
    Q = (xhat ** 2) @ (gw ** 2).T
    B = r[:, None] * (np.abs(x) @ gw.T + np.abs(mu)[:, None] * gw.sum(axis=1)[None, :])
    v = np.zeros(w.shape[0]) if beta is None else w @ beta
    V = np.zeros(w.shape[0]) if beta is None else np.abs(w) @ np.abs(beta)
    bound = ((ub + 2.0 ** -20) * np.abs(ref) + ub * A
             + K * 2.0 ** -23 * (B + V[None, :] + np.abs(ref - v[None, :])))
    err = np.abs(gpu - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        msg = "; ".join(f"[{i},{j}] gpu={gpu[i, j]!r} ref={ref[i, j]!r} bound={bound[i, j]:.3g}"
                        for i, j in idx)
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} elements out of "
                             f"tolerance: {msg}")
    rms = float(np.sqrt(np.mean(err ** 2)))
    expect = float(np.sqrt(ub ** 2 / 3.0 * np.mean(Q + ref ** 2)))
    assert rms <= 1.5 * expect, f"{name}: RMS error {rms:.3g} above 1.5 x expected {expect:.3g}"
    return rms / expect
