"""The two-pass path for rows wider than one thread-block cluster holds
(N > NORM_MAX_N_ONEPASS), against the fp64 oracle through the C ABI.

Small cases force the path with the plan override split=1 and 1024-column
segments, so that many segments, a ragged last segment (down to one 16-byte
chunk) and units that straddle segments are checked on every row.  Wide
rows (262152 to 1048576 columns) take it by themselves; at a few rows every
row is checked, at thousands of rows a sample of rows and every column sum.
"""
import ctypes

import numpy as np
import pytest
import torch

import memory_bound_normalization_rmsnorm_gb300 as gb
from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

import parity_util as pu

pytestmark = pytest.mark.gpu


def _base(mode, wide=False):
    if mode == wl.LAYER:
        return wl.WORKLOADS["layer_32768x4096"]
    return wl.WORKLOADS["rms_4096x131072" if wide else "rms_262144x1024_outliers"]


FORCED = [(37, 1024), (130, 3000), (70, 4104), (9, 8200), (1, 8), (3, 1016), (600, 2048),
          (257, 5120)]


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER], ids=["rms", "layer"])
@pytest.mark.parametrize("M,N", FORCED)
def test_forced_two_pass_small(mode, M, N, monkeypatch):
    monkeypatch.setenv("GBNORM_PLAN", "split=1,W=1024")
    case = wl.like(_base(mode), M, N)
    x, g, b, dy = [None if t is None else t.cuda()
                   for t in wl.make_inputs(case, "cpu", seed=M + N)]
    assert gb.norm_plan(M, N, mode, True)["split_segments"] == -(-N // 1024)
    outs = pu.run_gpu(x, g, b, dy, case.eps, mode)
    assert gb.norm_get_device_error() == 0
    pu.compare(mode, case.eps, x, g, b, dy, outs, label=f"split {mode}:{M}x{N}")


WIDE = [(3, 262152), (6, 524288), (5, 1048576), (2, 300008), (4, 262144 + 4096 * 3 + 8),
        (2, 1 << 24)]  # the widest row the library takes (NORM_MAX_N): 4096 segments


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER], ids=["rms", "layer"])
@pytest.mark.parametrize("M,N", WIDE)
def test_wide_rows_every_row(mode, M, N, monkeypatch):
    # stream=0: the two-pass path also at the widths the streaming kernels
    # take by default (test_stream.py covers those)
    monkeypatch.setenv("GBNORM_PLAN", "stream=0")
    case = wl.like(_base(mode, wide=True), M, N)
    x, g, b, dy = [None if t is None else t.cuda()
                   for t in wl.make_inputs(case, "cpu", seed=N % 1000 + M)]
    assert gb.norm_plan(M, N, mode, False)["split_segments"] == -(-N // 4096)
    outs = pu.run_gpu(x, g, b, dy, case.eps, mode)
    assert gb.norm_get_device_error() == 0
    pu.compare(mode, case.eps, x, g, b, dy, outs, label=f"wide {mode}:{M}x{N}")


@pytest.mark.slow
@pytest.mark.parametrize("mode,M,N", [(wl.RMS, 4096, 524288), (wl.LAYER, 2048, 524288),
                                      (wl.RMS, 1024, 1048576)])
def test_wide_rows_many(mode, M, N):
    """Thousands of wide rows (the very-long-row workload family extended
    past the cluster limit), with the default plans (streamed where they
    stream, else two-pass): sampled rows against the oracle, dgamma /
    dbeta over every row, and every row's LayerNorm identity sum(dx) = 0."""
    case = wl.like(_base(mode, wide=True), M, N)
    x, g, b, dy = wl.make_inputs(case, "cuda")
    outs = pu.run_gpu(x, g, b, dy, case.eps, mode)
    assert gb.norm_get_device_error() == 0
    rows = pu.sample_rows(M, 24, seed=N + M)
    pu.compare(mode, case.eps, x, g, b, dy, outs, rows=rows, label=f"many {mode}:{M}x{N}")
    y, rstd, mean, dx, dg, db = outs
    assert torch.isfinite(rstd).all() and (rstd > 0).all()
    assert torch.isfinite(y.float()).all() and torch.isfinite(dx.float()).all()
    if mode == wl.LAYER:
        dxf = dx.float()
        rowsum = dxf.sum(dim=1, dtype=torch.float64)
        bound = 2.0 ** -7 * dxf.abs().sum(dim=1, dtype=torch.float64) + 1e-30
        assert (rowsum.abs() <= bound).all()


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER], ids=["rms", "layer"])
def test_two_pass_bitwise_reproducible(mode, monkeypatch):
    monkeypatch.setenv("GBNORM_PLAN", "stream=0")
    M, N = 300, 524288
    case = wl.like(_base(mode, wide=True), M, N)
    x, g, b, dy = wl.make_inputs(case, "cuda")
    first = pu.run_gpu(x, g, b, dy, case.eps, mode)
    for _ in range(3):
        again = pu.run_gpu(x, g, b, dy, case.eps, mode)
        for a, c in zip(first, again):
            if a is not None:
                assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                                   c.view(torch.int16) if c.dtype == torch.bfloat16 else c)
    assert gb.norm_get_device_error() == 0


def test_two_pass_workspace_contents_ignored():
    """The backward's workspace may hold anything on entry (NaN here): the
    dx pass writes every slot the reduction reads."""
    M, N, mode = 7, 300008, wl.LAYER
    case = wl.like(_base(mode), M, N)
    x, g, b, dy = wl.make_inputs(case, "cuda")
    y, rstd, mean = gb.norm_fwd(x, g, b, case.eps, mode)
    ref = gb.norm_bwd(dy, x, g, rstd, mean, mode)
    nbytes = gb.norm_bwd_workspace_bytes(M, N, mode)
    ws = torch.full((nbytes // 4 + 4,), float("nan"), device="cuda")
    dx, dg, db = gb.norm_bwd(dy, x, g, rstd, mean, mode, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(dx.view(torch.int16), ref[0].view(torch.int16))
    assert torch.equal(dg, ref[1]) and torch.equal(db, ref[2])


def test_two_pass_through_host_pipeline():
    """norm_fwd_bwd_host on wide rows: y, rstd, mean and dx equal the device
    path's bit for bit; dgamma / dbeta (summed per chunk, then over chunks)
    within the T2 tolerance."""
    import tolerances

    M, N, mode = 40, 524288, wl.LAYER
    case = wl.like(_base(mode), M, N)
    x, g, b, dy = wl.make_inputs(case, "cuda")
    dev = pu.run_gpu(x, g, b, dy, case.eps, mode)
    hx, hdy = x.cpu().pin_memory(), dy.cpu().pin_memory()
    host = gb.norm_fwd_bwd_host(hx, hdy, g.cpu(), b.cpu(), case.eps, mode)
    torch.cuda.synchronize()
    hy, hr, hm, hdx, hdg, hdb = host
    assert torch.equal(hy.view(torch.int16), dev[0].cpu().view(torch.int16))
    assert torch.equal(hr, dev[1].cpu()) and torch.equal(hm, dev[2].cpu())
    assert torch.equal(hdx.view(torch.int16), dev[3].cpu().view(torch.int16))
    s = dy.float().abs().sum(0).double().cpu().numpy()
    tolerances.check_t2(pu.f64(hdb), pu.f64(dev[5]), s, "host dbeta")


def test_fused_variants_keep_their_limit():
    """The fused residual and E4M3 entry points stop at NORM_MAX_N_FUSED."""
    M, N = 2, 262152
    x = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(N, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gb.NormError) as e:
        gb.norm_add_fwd(x, x, g, None, 1e-6, wl.RMS)
    assert e.value.status == 2
    with pytest.raises(gb.NormError) as e:
        gb.norm_fwd_fp8(x, g, None, 1e-6, wl.RMS, gb.FP8_ROW)
    assert e.value.status == 2
