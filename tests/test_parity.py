"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Small and medium cases check every row; the shapes span many tiles per CTA
(so the shared-memory ring wraps), ragged last tiles, ragged chunk counts
and every plan regime (sub-warp, warp, multi-warp and cluster rows)."""
import numpy as np
import pytest
import torch

import memory_bound_normalization_rmsnorm_gb300 as gb
from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

import parity_util as pu

pytestmark = pytest.mark.gpu


def _small_cases():
    W = wl.WORKLOADS
    out = [(W["rms_256x1024"], 256, 1024)]
    out.append((W["layer_32768x4096"], 9001, 4096))       # ring wraps (> grid*S tiles)
    for n in (256, 512, 768, 1024):
        out.append((W[f"rms_262144x{n}_outliers"], 4099, n))
    out.append((W["rms_262144x256_outliers"], 70001, 256))  # ring wraps, RT = 64
    for n in (16384, 32768, 65536, 131072):
        out.append((W[f"rms_4096x{n}"], 37, n))
    for n in (24576, 32768, 65536, 131072):  # LayerNorm long rows, exact slices
        out.append((W["layer_32768x4096"], 37, n))
    for mode in ("rms", "layer"):
        for n in (2048, 3072, 5120, 8192):
            out.append((W[f"{mode}_32768x{n}_resid"], 605, n))
    return out


@pytest.mark.parametrize("w,M,N", _small_cases(), ids=lambda v: getattr(v, "name", str(v)))
def test_parity_workload_family(w, M, N):
    case = wl.like(w, M, N)
    x, g, b, dy = [None if t is None else t.cuda() for t in wl.make_inputs(case, "cpu")]
    outs = pu.run_gpu(x, g, b, dy, case.eps, case.mode)
    pu.compare(case.mode, case.eps, x, g, b, dy, outs, label=case.name)


AWKWARD_N = [8, 16, 24, 40, 72, 104, 200, 264, 520, 776, 1000, 1032, 2056, 4104, 12296,
             16392, 40000, 131080, 262144]


@pytest.mark.parametrize("mode", [0, 1], ids=["rms", "layer"])
@pytest.mark.parametrize("N", AWKWARD_N)
def test_parity_awkward_shapes(mode, N):
    base = wl.WORKLOADS["layer_32768x4096" if mode else "rms_256x1024"]
    for M in (1, 3, 50):
        if M * N > 4_000_000 and M > 3:
            continue
        case = wl.like(base, M, N)
        x, g, b, dy = [None if t is None else t.cuda()
                       for t in wl.make_inputs(case, "cpu", seed=N + M)]
        outs = pu.run_gpu(x, g, b, dy, case.eps, case.mode)
        pu.compare(mode, case.eps, x, g, b, dy, outs, label=f"{mode}:{M}x{N}")


@pytest.mark.parametrize("mode", [0, 1], ids=["rms", "layer"])
def test_layer_beta_none_and_dbeta_skipped(mode):
    """LayerNorm with beta omitted (zero shift) and dbeta not requested."""
    if mode == 0:
        pytest.skip("LayerNorm only")
    case = wl.like(wl.WORKLOADS["layer_32768x4096"], 130, 1024)
    x, g, b, dy = [None if t is None else t.cuda() for t in wl.make_inputs(case, "cpu")]
    zero = torch.zeros_like(b)
    y0, r0, m0 = gb.norm_fwd(x, g, None, case.eps, mode)
    y1, r1, m1 = gb.norm_fwd(x, g, zero, case.eps, mode)
    dx0, dg0, db0 = gb.norm_bwd(dy, x, g, r0, m0, mode, want_dbeta=False)
    dx1, dg1, db1 = gb.norm_bwd(dy, x, g, r1, m1, mode)
    torch.cuda.synchronize()
    assert db0 is None
    assert torch.equal(y0, y1) and torch.equal(r0, r1) and torch.equal(m0, m1)
    assert torch.equal(dx0, dx1) and torch.equal(dg0, dg1)


def test_special_rows():
    """Constant rows (RMSNorm -> gamma*sign(c); LayerNorm -> beta), zero rows
    and rows with a single huge outlier, against the oracle."""
    M, N = 64, 2048
    x = torch.randn(M, N)
    x[0] = 0.0
    x[1] = 3.0
    x[2] = -0.5
    x[3, 17] = 1e4
    x[4] = 1e-30
    x = x.to(torch.bfloat16).cuda()
    gen = torch.Generator().manual_seed(3)
    g = (1 + 0.1 * torch.randn(N, generator=gen)).to(torch.bfloat16).cuda()
    b = (0.1 * torch.randn(N, generator=gen)).to(torch.bfloat16).cuda()
    dy = torch.randn(M, N, generator=gen).to(torch.bfloat16).cuda()
    for mode in (0, 1):
        bb = b if mode == 1 else None
        outs = pu.run_gpu(x, g, bb, dy, 1e-6, mode)
        pu.compare(mode, 1e-6, x, g, bb, dy, outs, label=f"special mode={mode}")
    y, _, _ = gb.norm_fwd(x, g, None, 1e-6, 0)
    torch.cuda.synchronize()
    # RMSNorm of a constant row c is gamma * c / sqrt(c^2 + eps) ~ gamma * sign(c)
    assert torch.allclose(y[1].float(), g.float(), rtol=1e-2)
    assert torch.allclose(y[2].float(), -g.float(), rtol=1e-2)
    assert torch.count_nonzero(y[0]) == 0


def test_rows_are_independent():
    """Each output row depends on its own input row only: computing a subset
    of rows alone gives the same bits as inside the full batch."""
    case = wl.like(wl.WORKLOADS["layer_32768x4096"], 2001, 4096)
    x, g, b, dy = [None if t is None else t.cuda() for t in wl.make_inputs(case, "cpu")]
    y, r, m = gb.norm_fwd(x, g, b, case.eps, 1)
    sub = slice(1000, 1013)
    y2, r2, m2 = gb.norm_fwd(x[sub].contiguous(), g, b, case.eps, 1)
    dx, _, _ = gb.norm_bwd(dy, x, g, r, m, 1)
    dx2, _, _ = gb.norm_bwd(dy[sub].contiguous(), x[sub].contiguous(), g, r2, m2, 1)
    torch.cuda.synchronize()
    assert torch.equal(y[sub], y2) and torch.equal(r[sub], r2) and torch.equal(dx[sub], dx2)


@pytest.mark.gpu
@pytest.mark.parametrize("mode,M,N", [(wl.LAYER, 9001, 4096), (wl.RMS, 3001, 2048),
                                      (wl.LAYER, 777, 1024)])
def test_forward_with_wait_hint(mode, M, N, monkeypatch):
    """Forward plans whose stage waits sleep (the LayerNorm 4096 default,
    and others forced with hint=): same results as the oracle."""
    monkeypatch.setenv("GBNORM_PLAN", "hint=2000")
    assert gb.norm_plan(M, N, mode, False)["wait_hint_ns"] == 2000
    base = wl.WORKLOADS["layer_32768x4096" if mode == wl.LAYER else "rms_262144x1024_outliers"]
    case = wl.like(base, M, N)
    x, g, b, dy = [None if t is None else t.cuda()
                   for t in wl.make_inputs(case, "cpu", seed=M + N)]
    outs = pu.run_gpu(x, g, b, dy, case.eps, mode)
    assert gb.norm_get_device_error() == 0
    pu.compare(mode, case.eps, x, g, b, dy, outs, label=f"hint {mode}:{M}x{N}")
