"""Normalisation fused into the tcgen05 GEMM (norm_gemm_prepare /
norm_gemm_fwd) against the oracle's fp64 norm(x) W^T: out within T4, rstd
and mean within T2, the prepared weights exact, results reproducible."""
import numpy as np
import pytest
import torch

import memory_bound_normalization_rmsnorm_gb300 as gb
from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

import oracle
import parity_util as pu
import tolerances

pytestmark = pytest.mark.gpu

EPS = 1e-5


def _inputs(mode, M, K, Nout, seed=0, dist="normal", row_offset=0.0):
    w0 = wl.Workload(f"gemm_{M}x{K}x{Nout}", mode, M, K, EPS, dist, "one_plus_0.1n", seed=seed)
    x, gamma, beta, _ = wl.make_inputs(w0, "cuda", with_dy=False)
    if row_offset:
        x = (x.float() + row_offset).to(torch.bfloat16)
    w = wl.make_gemm_weight(w0, Nout, "cuda")
    return x, gamma, (beta if mode == wl.LAYER else None), w


def _run(x, gamma, beta, w, mode):
    wg, u, v = gb.norm_gemm_prepare(w, gamma, beta, mode)
    out, rstd, mean = gb.norm_gemm_fwd(x, wg, u, v, EPS, mode)
    torch.cuda.synchronize()
    st = gb.norm_get_device_error()
    assert st == 0, f"device error word {st}"
    return wg, u, v, out, rstd, mean


def _compare(x, gamma, beta, w, outs, mode, rows=None, label=""):
    _, _, _, out, rstd, mean = outs
    xb, gbits, wb = wl.bf16_bits(x), wl.bf16_bits(gamma), wl.bf16_bits(w)
    bb = None if beta is None else wl.bf16_bits(beta)
    sel = None if rows is None else np.asarray(rows, np.int64)
    eps64 = float(np.float32(EPS))
    ref, r_ref, m_ref = oracle.norm_gemm_bf16(xb, gbits, bb, wb, eps64, mode, rows=sel)
    f = oracle.bf16_bits_to_f64
    idx = slice(None) if sel is None else torch.as_tensor(sel, device=out.device)
    xs = f(xb if sel is None else xb[sel])
    ratio = tolerances.check_t4(pu.f64(out[idx]), ref, xs, f(gbits),
                                None if bb is None else f(bb), f(wb), r_ref,
                                m_ref if mode == wl.LAYER else None, f"{label} out")
    tolerances.check_t2(pu.f64(rstd[idx]), r_ref, None, f"{label} rstd")
    if mode == wl.LAYER:
        tolerances.check_t2(pu.f64(mean[idx]), m_ref, np.abs(xs).mean(axis=1), f"{label} mean")
    else:
        assert mean is None
    return ratio


SMALL = [(1, 64, 32), (7, 128, 96), (128, 256, 256), (129, 512, 288), (255, 256, 128),
         (256, 128, 512), (300, 1024, 544), (1000, 2048, 1024), (257, 4096, 512)]


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER])
@pytest.mark.parametrize("M,K,Nout", SMALL)
def test_parity_small(mode, M, K, Nout):
    """Shapes spanning one to several 128 x 256 tiles in each direction, K
    from one 64-wide block up, with ragged M and Nout tails."""
    x, gamma, beta, w = _inputs(mode, M, K, Nout, seed=M + K)
    outs = _run(x, gamma, beta, w, mode)
    _compare(x, gamma, beta, w, outs, mode, label=f"{M}x{K}x{Nout}")


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER])
@pytest.mark.parametrize("form", ["1", "2"])
@pytest.mark.parametrize("M,K,Nout", [(1, 64, 32), (129, 512, 288), (300, 1024, 544),
                                      (1000, 2048, 1024), (200, 256, 96)])
def test_cluster_kernels(mode, form, M, K, Nout, monkeypatch):
    """Both kernel forms on ragged shapes: the single-CTA kernel
    (GBNORM_GEMM_CTAS=1, 128 x 256 tiles) and the 2-CTA cluster kernel (the
    default, also selected with GBNORM_GEMM_CTAS=2: cta_group::2 MMAs over
    256-row tiles), including a last 256-row block whose second CTA owns no
    row."""
    monkeypatch.setenv("GBNORM_GEMM_CTAS", form)
    x, gamma, beta, w = _inputs(mode, M, K, Nout, seed=M + 3 * K)
    outs = _run(x, gamma, beta, w, mode)
    _compare(x, gamma, beta, w, outs, mode, label=f"form {form} {M}x{K}x{Nout}")


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER])
@pytest.mark.parametrize("form", ["1", "2"])
def test_cluster_kernels_full_size(mode, form, monkeypatch):
    """Both kernel forms at 32768 x 4096 x 4096: sampled rows against the
    oracle (rows of either CTA of a cluster) and every row's rstd against
    float64 statistics."""
    monkeypatch.setenv("GBNORM_GEMM_CTAS", form)
    M, K = 32768, 4096
    x, gamma, beta, w = _inputs(mode, M, K, K, seed=12)
    outs = _run(x, gamma, beta, w, mode)
    rows = pu.sample_rows(M, n=64, seed=3)
    _compare(x, gamma, beta, w, outs, mode, rows=rows, label="pair full size")
    xd = x.double()
    if mode == wl.LAYER:
        var = ((xd - xd.mean(dim=1, keepdim=True)) ** 2).mean(dim=1)
    else:
        var = (xd ** 2).mean(dim=1)
    r64 = 1.0 / torch.sqrt(var + float(np.float32(EPS)))
    assert (outs[4].double() / r64 - 1).abs().max().item() < 1e-5


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER])
@pytest.mark.parametrize("K", [5120, 8192])
def test_default_kernel_wide(mode, K):
    """The default kernel at the widest benchmark shapes, 32768 x K x K (CTA
    pairs, statistics units of 5 and 8 column tiles, 2048-row tile groups):
    sampled rows against the oracle, every row's rstd against float64
    statistics."""
    M = 32768
    x, gamma, beta, w = _inputs(mode, M, K, K, seed=K + mode)
    outs = _run(x, gamma, beta, w, mode)
    rows = pu.sample_rows(M, n=32, seed=K)
    _compare(x, gamma, beta, w, outs, mode, rows=rows, label=f"default {K}")
    xd = x.double()
    if mode == wl.LAYER:
        var = ((xd - xd.mean(dim=1, keepdim=True)) ** 2).mean(dim=1)
    else:
        var = (xd ** 2).mean(dim=1)
    r64 = 1.0 / torch.sqrt(var + float(np.float32(EPS)))
    assert (outs[4].double() / r64 - 1).abs().max().item() < 1e-5


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER])
@pytest.mark.parametrize("group", ["2", "4"])
@pytest.mark.parametrize("pair", ["1", "2"])
def test_statistics_shared_by_column_tiles(mode, group, pair, monkeypatch):
    """A CTA (pair) taking 2 or 4 consecutive column tiles of a row block
    computes the row statistics once and reuses them (forced with
    GBNORM_GEMM_GROUP; LayerNorm chooses it by itself at full size)."""
    monkeypatch.setenv("GBNORM_GEMM_GROUP", group)
    monkeypatch.setenv("GBNORM_GEMM_CTAS", pair)
    x, gamma, beta, w = _inputs(mode, 700, 1024, 1024, seed=5, row_offset=1.0)
    outs = _run(x, gamma, beta, w, mode)
    _compare(x, gamma, beta, w, outs, mode, label=f"group {group} ctas {pair}")


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER])
@pytest.mark.parametrize("group,Nout", [("5", 2560), ("8", 2048)])
@pytest.mark.parametrize("pair", ["1", "2"])
def test_statistics_shared_by_wide_units(mode, group, Nout, pair, monkeypatch):
    """Units of 5 and 8 column tiles (the planner's choice at 5120 and 8192
    output columns), forced on smaller shapes whose tile counts they divide."""
    monkeypatch.setenv("GBNORM_GEMM_GROUP", group)
    monkeypatch.setenv("GBNORM_GEMM_CTAS", pair)
    x, gamma, beta, w = _inputs(mode, 900, 512, Nout, seed=7, row_offset=0.5)
    outs = _run(x, gamma, beta, w, mode)
    _compare(x, gamma, beta, w, outs, mode, label=f"group {group} Nout {Nout} ctas {pair}")


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER])
def test_large_row_offset(mode):
    """Rows offset by 3 (mean far from 0): the mean correction after the
    contraction, and the one-pass block statistics, hold up."""
    x, gamma, beta, w = _inputs(mode, 384, 2048, 512, seed=3, row_offset=3.0)
    outs = _run(x, gamma, beta, w, mode)
    _compare(x, gamma, beta, w, outs, mode, label="offset 3")


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER])
def test_prepared_weights(mode):
    """W' = bf16(W * gamma) bit for bit (torch's own float32 product and
    bf16 rounding), u = row sums of W' and v = W beta to fp32 accuracy."""
    x, gamma, beta, w = _inputs(mode, 4, 1024, 320, seed=9)
    wg, u, v = gb.norm_gemm_prepare(w, gamma, beta, mode)
    torch.cuda.synchronize()
    want = (w.float() * gamma.float()[None, :]).to(torch.bfloat16)
    assert torch.equal(wg.view(torch.int16), want.view(torch.int16))
    if mode == wl.LAYER:
        wg64 = wg.double().cpu()
        u_ref = wg64.sum(dim=1)
        v_ref = w.double().cpu() @ beta.double().cpu()
        tolerances.check_t2(pu.f64(u), u_ref.numpy(), wg64.abs().sum(dim=1).numpy(), "u")
        s = (w.double().abs() @ beta.double().abs()).cpu().numpy()
        tolerances.check_t2(pu.f64(v), v_ref.numpy(), s, "v")
    else:
        assert u is None and v is None


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER])
@pytest.mark.parametrize("K", [2048, 3072, 4096, 5120, 8192])
def test_full_size_sampled(mode, K):
    """The transformer-block shapes (M = 2 x 16384 tokens, Nout = K) with
    the residual-stream-like input, checked on sampled rows (the first and
    last rows of the first and last tiles included)."""
    M = 32768
    dist = "normal" if K == 4096 else "normal_offset"
    x, gamma, beta, w = _inputs(mode, M, K, K, seed=0, dist=dist)
    outs = _run(x, gamma, beta, w, mode)
    rows = pu.sample_rows(M, n=48 if K > 4096 else 96, seed=K)
    _compare(x, gamma, beta, w, outs, mode, rows=rows, label=f"{M}x{K}x{K}")


def test_ragged_full_width():
    """M not a multiple of the 128-row tile at K = Nout = 4096."""
    M = 32768 - 45
    x, gamma, beta, w = _inputs(wl.LAYER, M, 4096, 4096, seed=4)
    outs = _run(x, gamma, beta, w, wl.LAYER)
    rows = np.unique(np.concatenate([pu.sample_rows(M, n=48, seed=2), np.arange(M - 83, M)]))
    _compare(x, gamma, beta, w, outs, wl.LAYER, rows=rows, label="ragged M")


def test_reproducible():
    x, gamma, beta, w = _inputs(wl.LAYER, 1000, 4096, 1536, seed=6)
    a = _run(x, gamma, beta, w, wl.LAYER)
    b = _run(x, gamma, beta, w, wl.LAYER)
    for s, t in zip(a, b):
        assert torch.equal(s.view(torch.int16) if s.dtype == torch.bfloat16 else s,
                           t.view(torch.int16) if t.dtype == torch.bfloat16 else t)


@pytest.mark.parametrize("mode", [wl.RMS, wl.LAYER])
def test_every_row_statistics_repeatable(mode):
    """Every row's rstd (and mean) at 32768 x 4096 x 4096 against float64
    statistics recomputed by torch from the same bf16 x, over three runs
    that must agree bit for bit: a stale x chunk read from the shared-memory
    ring in any row of any tile shows up here."""
    M, K = 32768, 4096
    x, gamma, beta, w = _inputs(mode, M, K, K, seed=11)
    xd = x.double()
    if mode == wl.LAYER:
        mu = xd.mean(dim=1)
        var = ((xd - mu[:, None]) ** 2).mean(dim=1)
    else:
        mu = None
        var = (xd ** 2).mean(dim=1)
    r64 = 1.0 / torch.sqrt(var + float(np.float32(EPS)))
    first = None
    for _ in range(3):
        outs = _run(x, gamma, beta, w, mode)
        rstd, mean = outs[4], outs[5]
        assert (rstd.double() / r64 - 1).abs().max().item() < 1e-5
        if mode == wl.LAYER:
            s = xd.abs().mean(dim=1)
            assert ((mean.double() - mu).abs() <= 1e-3 * mu.abs() + 1e-6 * s).all()
        if first is None:
            first = [t.clone() for t in outs[3:] if t is not None]
        else:
            for a, b in zip(first, [t for t in outs[3:] if t is not None]):
                assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                                   b.view(torch.int16) if b.dtype == torch.bfloat16 else b)


def test_memory_not_on_this_device_is_refused():
    """x, W' and out are moved by tiled tensor copies, which need memory this
    GPU reaches directly: pinned host memory and pageable host memory given
    as any of them are refused with NORM_ERR_MEMORY before anything is
    launched, and the device path still works afterwards."""
    import ctypes

    M, K, Nout = 256, 512, 288
    x, gamma, beta, w = _inputs(wl.LAYER, M, K, Nout, seed=21)
    wg, u, v, out, rstd, mean = _run(x, gamma, beta, w, wl.LAYER)
    pinned = torch.empty(M * max(K, Nout), dtype=torch.bfloat16).pin_memory()
    pageable = torch.empty(M * max(K, Nout), dtype=torch.bfloat16)
    L = gb.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(xp, wp, op):
        return L.norm_gemm_fwd(xp, wp, u.data_ptr(), v.data_ptr(), M, K, Nout, EPS, wl.LAYER,
                               op, rstd.data_ptr(), mean.data_ptr(), stream)

    for host in (pinned, pageable):
        assert call(host.data_ptr(), wg.data_ptr(), out.data_ptr()) == 10
        assert call(x.data_ptr(), host.data_ptr(), out.data_ptr()) == 10
        assert call(x.data_ptr(), wg.data_ptr(), host.data_ptr()) == 10
    assert call(x.data_ptr(), wg.data_ptr(), out.data_ptr()) == 0
    torch.cuda.synchronize()
    assert gb.norm_get_device_error() == 0
