"""CPU check of the T4 rule used for the normalisation-GEMM parity: a float32
emulation of the fused arithmetic (W' = bf16(W * gamma), fp32 contraction,
rstd and the mean correction applied afterwards, bf16 output) passes it, and
plausible mistakes in that arithmetic fail it."""
import numpy as np
import pytest
import torch

from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

import oracle
import tolerances


def _emulate(x, gamma, beta, w, eps, mode, drop_mean=False, gamma_twice=False, no_rstd=False):
    xf = x.float()
    wg = (w.float() * gamma.float()[None, :]).to(torch.bfloat16).float()
    if gamma_twice:
        wg = (wg * gamma.float()[None, :]).to(torch.bfloat16).float()
    u = wg.sum(dim=1)
    acc = xf @ wg.T
    if mode == wl.LAYER:
        mu = xf.mean(dim=1)
        var = ((xf - mu[:, None]) ** 2).mean(dim=1)
        v = w.float() @ beta.float()
    else:
        mu = torch.zeros(x.shape[0])
        var = (xf ** 2).mean(dim=1)
        v = torch.zeros(w.shape[0])
    r = torch.rsqrt(var + eps)
    if no_rstd:
        r = torch.ones_like(r)
    corr = acc if drop_mean else acc - mu[:, None] * u[None, :]
    return (r[:, None] * corr + v[None, :]).to(torch.bfloat16)


def _case(mode, M, K, Nout, off):
    w0 = wl.Workload("t4", mode, M, K, 1e-5, "normal_offset" if off else "normal",
                     "one_plus_0.1n")
    x, gamma, beta, _ = wl.make_inputs(w0, seed=5, with_dy=False)
    if off:
        x = (x.float() + off).to(torch.bfloat16)
    w = wl.make_gemm_weight(w0, Nout, seed=5)
    return x, gamma, beta if mode == wl.LAYER else None, w


def _check(x, gamma, beta, w, out, mode):
    xb, gb_, wb = wl.bf16_bits(x), wl.bf16_bits(gamma), wl.bf16_bits(w)
    bb = None if beta is None else wl.bf16_bits(beta)
    ref, r, m = oracle.norm_gemm_bf16(xb, gb_, bb, wb, float(np.float32(1e-5)), mode)
    f = oracle.bf16_bits_to_f64
    return tolerances.check_t4(out.double().numpy(), ref, f(xb), f(gb_),
                               None if bb is None else f(bb), f(wb), r,
                               m if mode == wl.LAYER else None, "emulated")


@pytest.mark.parametrize("mode,off", [(wl.RMS, 0.0), (wl.LAYER, 0.0), (wl.LAYER, 2.0)])
def test_emulation_passes(mode, off):
    x, gamma, beta, w = _case(mode, 96, 1024, 128, off)
    ratio = _check(x, gamma, beta, w, _emulate(x, gamma, beta, w, 1e-5, mode), mode)
    assert ratio < 1.0


@pytest.mark.parametrize("mistake", ["drop_mean", "gamma_twice", "no_rstd"])
def test_mistakes_fail(mistake):
    mode = wl.RMS if mistake == "no_rstd" else wl.LAYER
    x, gamma, beta, w = _case(mode, 96, 1024, 128, 0.0)
    out = _emulate(x, gamma, beta, w, 1e-5, mode, **{mistake: True})
    with pytest.raises(AssertionError):
        _check(x, gamma, beta, w, out, mode)
