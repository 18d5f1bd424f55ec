"""The streaming long-row backward (row slices of 32768 columns read twice,
the second time from L2, column sums in tensor memory) against the fp64
oracle through the C ABI.

The path is forced with the plan override stream=1 at every width it takes
(N = C x 32768, C = 1 .. 16): a single CTA per row, clusters of 2 to 16, few
rows (clusters with one row and with none beyond the first) and more rows
than clusters (each cluster streams several rows, the software pipeline of
pass 1 of row j with pass 2 of row j - 1 runs through).  Where it is the
default backward, the resident long-row kernel it replaces stays covered
here with stream=0.
"""
import numpy as np
import pytest
import torch

import memory_bound_normalization_rmsnorm_gb300 as gb
from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

import parity_util as pu

pytestmark = pytest.mark.gpu


def _base(mode):
    return wl.WORKLOADS["layer_32768x4096" if mode == wl.LAYER else "rms_4096x131072"]


CASES = [(1, 32768), (5, 32768), (300, 32768), (3, 65536), (81, 65536), (2, 131072),
         (45, 131072), (7, 262144), (40, 262144), (3, 524288), (12, 524288)]


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER], ids=["rms", "layer"])
@pytest.mark.parametrize("M,N", CASES)
@pytest.mark.parametrize("piece", ["", "other"], ids=["default-piece", "other-piece"])
def test_stream_every_row(mode, M, N, piece, monkeypatch):
    # the piece width the mode does not take by default: 8192 columns for
    # RMSNorm, 16384 for LayerNorm (two register batches of accumulators)
    if piece:
        piece = ",W=8192" if mode == wl.RMS else ",W=16384"
    monkeypatch.setenv("GBNORM_PLAN", "stream=1" + piece)
    plan = gb.norm_plan(M, N, mode, True)
    assert plan["streamed"] == 1 and plan["cluster"] == N // 32768
    case = wl.like(_base(mode), M, N)
    x, g, b, dy = [None if t is None else t.cuda()
                   for t in wl.make_inputs(case, "cpu", seed=N % 977 + M)]
    outs = pu.run_gpu(x, g, b, dy, case.eps, mode)
    assert gb.norm_get_device_error() == 0
    pu.compare(mode, case.eps, x, g, b, dy, outs, label=f"stream {mode}:{M}x{N}")


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER], ids=["rms", "layer"])
def test_stream_many_rows_sampled(mode, monkeypatch):
    """The full-size very-long-row workload (4096 x 131072): sampled rows
    against the oracle, dgamma / dbeta over every row, LayerNorm's
    sum(dx) = 0 per row."""
    monkeypatch.setenv("GBNORM_PLAN", "stream=1")
    M, N = 4096, 131072
    case = wl.like(_base(mode), M, N)
    x, g, b, dy = wl.make_inputs(case, "cuda")
    outs = pu.run_gpu(x, g, b, dy, case.eps, mode)
    assert gb.norm_get_device_error() == 0
    rows = pu.sample_rows(M, 24, seed=N + M)
    pu.compare(mode, case.eps, x, g, b, dy, outs, rows=rows, label=f"stream many {mode}")
    dx = outs[3].float()
    assert torch.isfinite(dx).all()
    if mode == wl.LAYER:
        rowsum = dx.sum(dim=1, dtype=torch.float64)
        bound = 2.0 ** -7 * dx.abs().sum(dim=1, dtype=torch.float64) + 1e-30
        assert (rowsum.abs() <= bound).all()


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER], ids=["rms", "layer"])
@pytest.mark.parametrize("N", [32768, 131072])
def test_stream_bitwise_reproducible(mode, N, monkeypatch):
    monkeypatch.setenv("GBNORM_PLAN", "stream=1")
    M = 200
    case = wl.like(_base(mode), M, N)
    x, g, b, dy = wl.make_inputs(case, "cuda")
    y, rstd, mean = gb.norm_fwd(x, g, b, case.eps, mode)
    first = gb.norm_bwd(dy, x, g, rstd, mean, mode)
    for _ in range(3):
        again = gb.norm_bwd(dy, x, g, rstd, mean, mode)
        assert torch.equal(first[0].view(torch.int16), again[0].view(torch.int16))
        assert torch.equal(first[1], again[1])
        if mode == wl.LAYER:
            assert torch.equal(first[2], again[2])
    assert gb.norm_get_device_error() == 0


def test_stream_workspace_contents_ignored(monkeypatch):
    """Every partial row the reduction reads is written by the kernel."""
    monkeypatch.setenv("GBNORM_PLAN", "stream=1")
    M, N, mode = 9, 65536, wl.LAYER
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


def test_stream_not_taken_where_it_does_not_apply(monkeypatch):
    """Rows that are not a multiple of 32768 columns (or wider than 16
    slices) keep the other backward plans under the override."""
    monkeypatch.setenv("GBNORM_PLAN", "stream=1")
    for N in (16384, 98304 + 8, 1048576):
        assert gb.norm_plan(64, N, wl.RMS, True)["streamed"] == 0
    p = gb.norm_plan(64, 98304, wl.RMS, True)  # three slices: a cluster of 3
    assert p["streamed"] == 1 and p["cluster"] == 3


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER], ids=["rms", "layer"])
@pytest.mark.parametrize("M,N", [(45, 131072), (7, 262144), (300, 32768)])
def test_resident_long_rows_where_streaming_is_default(mode, M, N, monkeypatch):
    """stream=0: the resident long-row backward (slice held in shared
    memory, clusters of up to 16) at widths that stream by default."""
    monkeypatch.setenv("GBNORM_PLAN", "stream=0")
    plan = gb.norm_plan(M, N, mode, True)
    assert plan["streamed"] == 0 and plan["long_rows"] == 1
    case = wl.like(_base(mode), M, N)
    x, g, b, dy = [None if t is None else t.cuda()
                   for t in wl.make_inputs(case, "cpu", seed=N % 991 + M)]
    outs = pu.run_gpu(x, g, b, dy, case.eps, mode)
    assert gb.norm_get_device_error() == 0
    pu.compare(mode, case.eps, x, g, b, dy, outs, label=f"resident {mode}:{M}x{N}")


@pytest.mark.parametrize("mode,M,N,ov", [(wl.RMS, 5, 65536, "stream=1,K=16"),
                                         (wl.RMS, 40, 262144, "stream=1,K=16"),
                                         (wl.RMS, 7, 131072, "stream=1,K=8"),
                                         (wl.RMS, 3, 1048576, ""), (wl.RMS, 9, 524288, ""),
                                         (wl.LAYER, 6, 524288, "stream=1")])
def test_stream_forward_wide_and_wide_slices(mode, M, N, ov, monkeypatch):
    """The streaming forward where it is the default (RMSNorm rows of 524288
    and 1048576 columns, 65536-column slices) and forced (65536- and
    32768-column slices at narrower rows, LayerNorm): every row against the
    oracle."""
    if ov:
        monkeypatch.setenv("GBNORM_PLAN", ov)
    p = gb.norm_plan(M, N, mode, False)
    assert p["streamed"] == 1
    if "K=16" in ov or not ov:
        assert p["cols_per_cta"] == 65536
    case = wl.like(_base(mode), M, N)
    x, g, b, dy = [None if t is None else t.cuda()
                   for t in wl.make_inputs(case, "cpu", seed=N % 983 + M)]
    outs = pu.run_gpu(x, g, b, dy, case.eps, mode)
    assert gb.norm_get_device_error() == 0
    pu.compare(mode, case.eps, x, g, b, dy, outs, label=f"stream fwd {mode}:{M}x{N}")


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER], ids=["rms", "layer"])
def test_stream_forward_bitwise_reproducible(mode, monkeypatch):
    monkeypatch.setenv("GBNORM_PLAN", "stream=1")
    M, N = 100, 524288
    case = wl.like(_base(mode), M, N)
    x, g, b, dy = wl.make_inputs(case, "cuda")
    assert gb.norm_plan(M, N, mode, False)["streamed"] == 1
    first = gb.norm_fwd(x, g, b, case.eps, mode)
    for _ in range(3):
        again = gb.norm_fwd(x, g, b, case.eps, mode)
        assert torch.equal(first[0].view(torch.int16), again[0].view(torch.int16))
        assert torch.equal(first[1], again[1])
        if mode == wl.LAYER:
            assert torch.equal(first[2], again[2])
    assert gb.norm_get_device_error() == 0
