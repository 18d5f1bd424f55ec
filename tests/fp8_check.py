"""Comparison of E4M3 output (codes and scales) with the oracle.

The kernels form y in fp32, so a code is decided from a value that may
differ from the oracle's exact y.  Bound used for that difference, per
element (fp32 arithmetic leaves about 2^-22 of the row scale for LayerNorm,
where x - mean and the + beta cancel, and about 2^-22 of |y| for RMSNorm,
a product of three roundings and rstd; the bound keeps an 8x margin):
    LayerNorm  |y_gpu - y| <= 2^-19 * max|y_row|
    RMSNorm    |y_gpu - y| <= 2^-19 * |y| + 2^-24 * max|y_row|
Every code whose value lies between the E4M3 roundings of the exact scaled
value pushed down and up by that bound (scaled) is correct; where both
roundings agree the code is unique and must match exactly.  Scales:
  per row  amax within the bound of the row's largest element, then one
           rounding of amax / 448 (and of 448 / amax for the codes);
  MX       an exponent floor(log2 a) - 8 (clamped at -127) of some a within
           the bound of the exact block amax.
+0 and -0 codes count as equal (the sign of a zero y is rounding noise).
"""
from __future__ import annotations

import numpy as np

import oracle

REL = 2.0 ** -19
FLOOR_RMS = 2.0 ** -24


def y_bound(y, mode):
    rowmax = np.abs(y).max(axis=1, keepdims=True)
    if mode == 1:
        return np.broadcast_to(REL * rowmax, y.shape)
    return REL * np.abs(y) + FLOOR_RMS * rowmax


def _e8m0_exponent(a):
    a = np.asarray(a, np.float64)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0))) - 8
    return np.where(a > 0, np.maximum(e, -127), -127).astype(np.int64)


def check_fp8(q, scale, ref, scaling, mode, label=""):
    """q: uint8 [R, N] from the GPU; scale: fp32 [R] (row) or uint8 [R, N/32]
    (MX); ref: oracle.fwd_fp8_bf16 output for the same rows; mode 0 RMSNorm,
    1 LayerNorm.  Returns the fraction of codes that were not unique."""
    y = ref["y"]
    R, N = y.shape
    q = np.asarray(q, np.uint8)
    assert q.shape == (R, N)
    dyv = y_bound(y, mode)
    if scaling == oracle.FP8_ROW:
        amax = ref["amax"]
        live = amax > 0
        am1 = np.where(live, amax, 1.0)
        rel = dyv.max(axis=1) / am1 + 2.0 ** -23           # amax_gpu's relative error
        s = np.asarray(scale, np.float64)
        want = np.where(live, amax / 448.0, 1.0)
        bad = ~(np.abs(s - want) <= np.where(live, rel * want, 0.0))
        assert not bad.any(), f"{label}: row scale off in {int(bad.sum())} rows"
        v = np.where(live[:, None], (y / am1[:, None]) * 448.0, y)
        delta = np.where(live[:, None],
                         448.0 * dyv / am1[:, None] + np.abs(v) * (rel[:, None] + 2.0 ** -23),
                         dyv)
    else:
        nb = N // 32
        e = np.asarray(scale, np.int64) - 127
        assert e.shape == (R, nb)
        amax = ref["amax"]
        db = dyv.reshape(R, nb, 32).max(axis=2)
        e_lo = _e8m0_exponent(np.maximum(amax - db, 0.0))
        e_hi = _e8m0_exponent(amax + db)
        bad = (e < e_lo) | (e > e_hi)
        assert not bad.any(), f"{label}: MX exponent off in {int(bad.sum())} blocks"
        X = np.repeat(np.exp2(e.astype(np.float64)), 32, axis=1)
        v = y / X
        delta = dyv / X
    lo = oracle.e4m3_encode(v - delta)
    hi = oracle.e4m3_encode(v + delta)
    d_lo, d_hi = oracle.e4m3_decode(lo), oracle.e4m3_decode(hi)
    d = oracle.e4m3_decode(q)
    assert not np.isnan(d).any(), f"{label}: NaN code"
    ok = (d >= d_lo) & (d <= d_hi)
    if not ok.all():
        i, j = np.argwhere(~ok)[0]
        raise AssertionError(f"{label}: {int((~ok).sum())} codes out of range; first [{i},{j}] "
                             f"code {q[i, j]:#04x} ({d[i, j]!r}) allowed [{d_lo[i, j]!r}, "
                             f"{d_hi[i, j]!r}] around {v[i, j]!r}")
    unique = d_lo == d_hi
    same = (q == lo) | (((q & 0x7F) == 0) & ((lo & 0x7F) == 0))
    assert same[unique].all(), f"{label}: unique codes differ"
    return 1.0 - float(unique.mean())
