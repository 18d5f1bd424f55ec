"""E4M3 output of the forward pass (norm_fwd_fp8) against the oracle:
codes, per-row scales and MX block exponents (tests/fp8_check.py gives the
rule), rstd and mean; plain and fused-residual; full-size sampled rows."""
import numpy as np
import pytest
import torch

import memory_bound_normalization_rmsnorm_gb300 as gb
from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

import fp8_check
import oracle
import parity_util as pu
import tolerances

pytestmark = pytest.mark.gpu

SCALINGS = [(gb.FP8_ROW, oracle.FP8_ROW), (gb.FP8_MX, oracle.FP8_MX)]


def _compare(case, x, r, g, b, outs, scaling, rows=None, label=""):
    q, scale, rstd, mean, h = outs
    eps64 = float(np.float32(case.eps))
    bb = None if b is None else wl.bf16_bits(b)
    rb = None if r is None else wl.bf16_bits(r)
    sel = None if rows is None else np.asarray(rows, np.int64)
    ref = oracle.fwd_fp8_bf16(wl.bf16_bits(x), rb, wl.bf16_bits(g), bb, eps64, case.mode,
                              scaling, rows=sel)
    idx = slice(None) if sel is None else torch.as_tensor(sel, device=q.device)
    qs = q[idx].cpu().numpy()
    ss = scale[idx].cpu().numpy()
    amb = fp8_check.check_fp8(qs, ss, ref, scaling, case.mode, label)
    assert amb < 0.01, f"{label}: {amb:.3%} of codes are not unique"
    src = wl.bf16_bits(x) if r is None else oracle.residual_add_bf16(wl.bf16_bits(x), rb)
    if h is not None:
        assert np.array_equal(wl.bf16_bits(h), src), f"{label}: h"
    _, r_ref, m_ref = oracle.fwd_bf16(src, wl.bf16_bits(g), bb, eps64, case.mode, rows=sel)
    tolerances.check_t2(pu.f64(rstd[idx]), r_ref, None, f"{label} rstd")
    if case.mode == wl.LAYER:
        xs = oracle.bf16_bits_to_f64(src if sel is None else src[sel])
        tolerances.check_t2(pu.f64(mean[idx]), m_ref, np.abs(xs).mean(axis=1), f"{label} mean")
    return amb


SHAPES = [(1, 32), (3, 64), (257, 256), (1031, 800), (4099, 1024), (2053, 2048),
          (1201, 3072), (2001, 4096), (617, 5120), (509, 8192), (33, 16384)]


@pytest.mark.parametrize("residual", [False, True], ids=["plain", "resid"])
@pytest.mark.parametrize("sc", SCALINGS, ids=["row", "mx"])
@pytest.mark.parametrize("mode", [0, 1], ids=["rms", "layer"])
@pytest.mark.parametrize("M,N", SHAPES)
def test_fp8_parity(M, N, mode, sc, residual):
    gsc, osc = sc
    if mode == 1 and N > 8192 and residual:
        pytest.skip("covered by the plain LayerNorm case at this width")
    base = wl.WORKLOADS["layer_32768x4096" if mode else "rms_262144x1024_outliers"]
    case = wl.like(base, M, N)
    x, r, g, b, _, _ = [None if t is None else t.cuda()
                        for t in wl.make_residual_inputs(case, "cpu", seed=M * 5 + N)]
    if not residual:
        r = None
    outs = gb.norm_fwd_fp8(x, g, b, case.eps, mode, gsc, r=r)
    torch.cuda.synchronize()
    _compare(case, x, r, g, b, outs, osc, label=f"{mode}:{M}x{N}:{gsc}:{residual}")


@pytest.mark.parametrize("sc", SCALINGS, ids=["row", "mx"])
@pytest.mark.parametrize("name", ["layer_32768x4096", "rms_262144x1024_outliers",
                                  "rms_32768x8192_resid", "layer_32768x5120_resid"])
def test_fp8_full_size(name, sc):
    gsc, osc = sc
    w = wl.WORKLOADS[name]
    x, g, b, _ = wl.make_inputs(w, "cuda", with_dy=False)
    outs = gb.norm_fwd_fp8(x, g, b, w.eps, w.mode, gsc)
    torch.cuda.synchronize()
    rows = pu.sample_rows(w.M, 96, seed=7)
    _compare(w, x, None, g, b, outs, osc, rows=rows, label=name)
    assert gb.norm_get_device_error() == 0


def test_fp8_stats_match_bf16_forward_and_deterministic(monkeypatch):
    """rstd / mean of the E4M3 forward equal norm_fwd's bit for bit when both
    run the same plan (the E4M3 forward stages gamma/beta in shared memory at
    this shape; the plan override makes norm_fwd do the same); two runs give
    identical codes and scales."""
    case = wl.like(wl.WORKLOADS["layer_32768x4096"], 3001, 4096)
    x, g, b, _ = [None if t is None else t.cuda() for t in wl.make_inputs(case, "cpu")]
    p8 = gb.norm_plan(3001, 4096, 1, False, fp8=True)
    assert p8["param_smem_bytes"] > 0
    monkeypatch.setenv("GBNORM_PLAN", "gsm=1")
    pb = gb.norm_plan(3001, 4096, 1, False)
    keys = ("threads_per_row", "chunks_per_thread", "groups", "rows_per_group")
    assert all(pb[k] == p8[k] for k in keys), (pb, p8)
    y, rs, mu = gb.norm_fwd(x, g, b, case.eps, 1)
    monkeypatch.delenv("GBNORM_PLAN")
    for gsc in (gb.FP8_ROW, gb.FP8_MX):
        a = gb.norm_fwd_fp8(x, g, b, case.eps, 1, gsc)
        c = gb.norm_fwd_fp8(x, g, b, case.eps, 1, gsc)
        torch.cuda.synchronize()
        assert torch.equal(a[0], c[0]) and torch.equal(a[1], c[1])
        assert torch.equal(a[2], rs) and torch.equal(a[3], mu)


def test_fp8_zero_rows_and_tiny_blocks():
    """A zero row (RMSNorm of zeros) has scale 1 / exponent byte 0 and zero
    codes; a block of tiny values takes the clamped exponent."""
    M, N = 4, 128
    x = torch.randn(M, N, device="cuda").to(torch.bfloat16)
    x[1] = 0
    g = torch.ones(N, device="cuda", dtype=torch.bfloat16)
    g[96:] = 2.0 ** -130
    q, s, _, _, _ = gb.norm_fwd_fp8(x, g, None, 1e-6, 0, gb.FP8_ROW)
    torch.cuda.synchronize()
    assert s[1].item() == 1.0 and int((q[1] & 0x7F).max()) == 0
    q, e, _, _, _ = gb.norm_fwd_fp8(x, g, None, 1e-6, 0, gb.FP8_MX)
    torch.cuda.synchronize()
    assert int(e[1].max()) == 0 and int((q[1] & 0x7F).max()) == 0
    assert int(e[0, 3]) == 0  # block of values ~2^-130: exponent clamped at -127
    ref = oracle.fwd_fp8_bf16(wl.bf16_bits(x), None, wl.bf16_bits(g), None,
                              float(np.float32(1e-6)), 0, oracle.FP8_MX)
    fp8_check.check_fp8(q.cpu().numpy(), e.cpu().numpy(), ref, oracle.FP8_MX, 0, "tiny")


@pytest.mark.parametrize("residual", [False, True], ids=["plain", "resid"])
@pytest.mark.parametrize("mode,M,N", [(0, 37, 32768), (0, 21, 40000), (1, 29, 18432),
                                      (1, 17, 24576), (0, 9, 65536), (0, 5, 131072),
                                      (1, 7, 65536), (1, 3, 131072), (1, 11, 40000),
                                      (0, 301, 65536)])
def test_fp8_long_rows(mode, M, N, residual):
    """Rows wider than one CTA's registers (long-row kernels, clusters):
    both scalings; with a cluster, per-row scaling sends the CTAs' slice
    maxima of a row in the next row's DSMEM exchange (and one last exchange
    after the last row), so every cluster case here has rows whose codes
    are written one exchange later, and the 301-row case gives each cluster
    several."""
    base = wl.WORKLOADS["layer_32768x4096" if mode else "rms_4096x16384"]
    case = wl.like(base, M, N)
    x, r, g, b, _, _ = [None if t is None else t.cuda()
                        for t in wl.make_residual_inputs(case, "cpu", seed=M * 3 + N)]
    if not residual:
        r = None
    plan = gb.norm_plan(M, N, mode, False, residual=residual, fp8=True)
    assert plan["long_rows"] == 1
    for gsc, osc in SCALINGS:
        outs = gb.norm_fwd_fp8(x, g, b, case.eps, mode, gsc, r=r)
        torch.cuda.synchronize()
        _compare(case, x, r, g, b, outs, osc, label=f"long {mode}:{M}x{N}:{gsc}:{residual}")
    assert gb.norm_get_device_error() == 0
