"""Fused residual add + norm (norm_add_fwd / norm_add_bwd) against the
oracle: h = bf16(x + r) bit for bit; y, rstd, mean, dx = norm dx + dh, dgamma
and dbeta within the parity tolerances."""
import numpy as np
import pytest
import torch

import memory_bound_normalization_rmsnorm_gb300 as gb
from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

import oracle
import parity_util as pu
import tolerances

pytestmark = pytest.mark.gpu


def _run(x, r, g, b, dy, dh, eps, mode):
    h, y, rstd, mean = gb.norm_add_fwd(x, r, g, b, eps, mode)
    dx, dg, db = gb.norm_add_bwd(dy, dh, h, g, rstd, mean, mode)
    torch.cuda.synchronize()
    return h, y, rstd, mean, dx, dg, db


def _compare(mode, eps, x, r, g, b, dy, dh, outs, rows=None, label=""):
    h, y, rstd, mean, dx, dg, db = outs
    eps64 = float(np.float32(eps))
    xb, rb, gbits = wl.bf16_bits(x), wl.bf16_bits(r), wl.bf16_bits(g)
    bb = None if b is None else wl.bf16_bits(b)
    dyb, dhb = wl.bf16_bits(dy), wl.bf16_bits(dh)
    h_ref = oracle.residual_add_bf16(xb, rb)
    assert np.array_equal(wl.bf16_bits(h), h_ref), f"{label}: h differs from bf16(x + r)"
    sel = None if rows is None else np.asarray(rows, np.int64)
    y_ref, r_ref, m_ref = oracle.fwd_bf16(h_ref, gbits, bb, eps64, mode, rows=sel)
    dx_ref = oracle.add_bwd_dx_bf16(dyb, h_ref, dhb, gbits, eps64, mode, rows=sel)
    dg_ref, db_ref, dg_abs, db_abs = oracle.param_grads_bf16(dyb, h_ref, gbits, eps64, mode)
    idx = slice(None) if sel is None else torch.as_tensor(sel, device=y.device)
    tolerances.check_t1(pu.f64(y[idx]), y_ref, f"{label} y")
    tolerances.check_t1(pu.f64(dx[idx]), dx_ref, f"{label} dx")
    tolerances.check_t2(pu.f64(rstd[idx]), r_ref, None, f"{label} rstd")
    tolerances.check_t2(pu.f64(dg), dg_ref, dg_abs, f"{label} dgamma")
    if mode == wl.LAYER:
        hs = oracle.bf16_bits_to_f64(h_ref if sel is None else h_ref[sel])
        tolerances.check_t2(pu.f64(mean[idx]), m_ref, np.abs(hs).mean(axis=1), f"{label} mean")
        tolerances.check_t2(pu.f64(db), db_ref, db_abs, f"{label} dbeta")


SHAPES = [(1, 8), (3, 24), (257, 256), (1031, 776), (4099, 1024), (2053, 2048),
          (1201, 3072), (2001, 4096), (617, 5120), (509, 8192)]


@pytest.mark.parametrize("mode", [0, 1], ids=["rms", "layer"])
@pytest.mark.parametrize("M,N", SHAPES)
def test_fused_residual_parity(mode, M, N):
    base = wl.WORKLOADS["layer_32768x4096" if mode else "rms_262144x1024_outliers"]
    case = wl.like(base, M, N)
    ins = [None if t is None else t.cuda()
           for t in wl.make_residual_inputs(case, "cpu", seed=M * 7 + N)]
    x, r, g, b, dy, dh = ins
    outs = _run(x, r, g, b, dy, dh, case.eps, mode)
    _compare(mode, case.eps, x, r, g, b, dy, dh, outs, label=f"{mode}:{M}x{N}")


@pytest.mark.parametrize("name", ["layer_32768x4096", "rms_32768x8192_resid",
                                  "layer_32768x2048_resid", "rms_4096x65536"])
def test_fused_residual_full_size(name):
    w = wl.WORKLOADS[name]
    x, r, g, b, dy, dh = wl.make_residual_inputs(w, "cuda")
    outs = _run(x, r, g, b, dy, dh, w.eps, w.mode)
    rows = pu.sample_rows(w.M, 128, seed=5)
    _compare(w.mode, w.eps, x, r, g, b, dy, dh, outs, rows=rows, label=name)
    assert gb.norm_get_device_error() == 0


def test_fused_residual_deterministic_and_matches_unfused():
    """Bitwise reproducible.  The fused kernels run the same row arithmetic
    as the plain ones on h (same threads per row and chunks per thread at
    this shape), so y, rstd, mean, dgamma and dbeta equal norm_fwd /
    norm_bwd on h bit for bit; dx differs only by the one rounding the
    unfused dx + dh would add."""
    M, N = 3001, 4096
    case = wl.like(wl.WORKLOADS["layer_32768x4096"], M, N)
    x, r, g, b, dy, dh = [t.cuda() for t in wl.make_residual_inputs(case, "cpu")]
    a = _run(x, r, g, b, dy, dh, case.eps, 1)
    c = _run(x, r, g, b, dy, dh, case.eps, 1)
    for u, v in zip(a, c):
        assert torch.equal(u, v)
    for bwd in (False, True):
        p = gb.norm_plan(M, N, 1, bwd)
        q = gb.norm_plan(M, N, 1, bwd, residual=True)
        keys = ("threads_per_row", "chunks_per_thread", "cluster", "partials")
        assert all(p[k] == q[k] for k in keys), (p, q)
    h = a[0]
    y2, rs2, m2 = gb.norm_fwd(h, g, b, case.eps, 1)
    dx2, dg2, db2 = gb.norm_bwd(dy, h, g, rs2, m2, 1)
    torch.cuda.synchronize()
    assert torch.equal(y2, a[1]) and torch.equal(rs2, a[2]) and torch.equal(m2, a[3])
    assert torch.equal(dg2, a[5]) and torch.equal(db2, a[6])
    # fused = RN(d + dh), unfused = RN(RN(d) + dh) with RN to bf16 (unit
    # roundoff u = 2^-8): |RN(d) - d| <= u|d| plus one rounding of each sum.
    fused, unfused = a[4].float(), (dx2.float() + dh.float()).to(torch.bfloat16).float()
    u = 2.0 ** -8
    bound = u * dx2.float().abs() + u * (fused.abs() + unfused.abs()) + 1e-30
    assert ((fused - unfused).abs() <= bound).all()


@pytest.mark.parametrize("mode,M,N", [(1, 67, 16384), (0, 45, 16384), (1, 33, 24576),
                                      (0, 21, 32768), (1, 19, 65536), (0, 9, 131072),
                                      (0, 5, 262144)])
@pytest.mark.parametrize("stream", ["", "stream=0"], ids=["default", "resident"])
def test_fused_residual_long_rows(mode, M, N, stream, monkeypatch):
    """Rows wider than one CTA's registers: the long-row kernels (shared-
    memory-resident slices, clusters beyond 16384 / 32768 columns) with the
    residual tensor in the same stage, and the backward that streams its
    slices where that is the default (rows of 32768 x 2^k columns); with
    stream=0 the resident long-row backward at those widths too."""
    if stream:
        monkeypatch.setenv("GBNORM_PLAN", stream)
    base = wl.WORKLOADS["layer_32768x4096" if mode else "rms_4096x16384"]
    case = wl.like(base, M, N)
    for bwd in (False, True):
        p = gb.norm_plan(M, N, mode, bwd, residual=True)
        assert (p["long_rows"] == 1 or p["streamed"] == 1
                or p["chunks_per_thread"] * p["threads_per_row"] * 8 >= N)
        if stream:
            assert p["streamed"] == 0
    ins = [None if t is None else t.cuda()
           for t in wl.make_residual_inputs(case, "cpu", seed=M + N)]
    x, r, g, b, dy, dh = ins
    outs = _run(x, r, g, b, dy, dh, case.eps, mode)
    _compare(mode, case.eps, x, r, g, b, dy, dh, outs, label=f"long {mode}:{M}x{N}")
    assert gb.norm_get_device_error() == 0


@pytest.mark.parametrize("mode,M,N", [(1, 45, 32768), (0, 81, 65536), (1, 7, 131072),
                                      (0, 40, 131072), (0, 12, 262144), (1, 5, 262144)])
def test_fused_residual_streamed_backward(mode, M, N, monkeypatch):
    """The streamed long-row backward with the residual gradient (stream=1:
    h and dy read twice, the second time from L2, dh once with the dx
    pass's pieces)."""
    monkeypatch.setenv("GBNORM_PLAN", "stream=1")
    assert gb.norm_plan(M, N, mode, True, residual=True)["streamed"] == 1
    base = wl.WORKLOADS["layer_32768x4096" if mode else "rms_4096x16384"]
    case = wl.like(base, M, N)
    x, r, g, b, dy, dh = [None if t is None else t.cuda()
                          for t in wl.make_residual_inputs(case, "cpu", seed=M + N + 1)]
    outs = _run(x, r, g, b, dy, dh, case.eps, mode)
    _compare(mode, case.eps, x, r, g, b, dy, dh, outs, label=f"stream resid {mode}:{M}x{N}")
    assert gb.norm_get_device_error() == 0
