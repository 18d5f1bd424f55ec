"""Parity at the full workload sizes, in the launch configuration bench.py
times (the library's default plan for each shape).

The oracle checks y, dx, rstd and mean on a seeded sample of rows (first,
last and random rows) and dgamma / dbeta on EVERY row (the column sums need
all of them; the oracle streams the rows in fp64).  Every row is also
checked against an identity that holds at any size: for LayerNorm the row
sum of dx is zero, up to the bf16 rounding of dx.
"""
import numpy as np
import pytest
import torch

import memory_bound_normalization_rmsnorm_gb300 as gb
from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

import parity_util as pu

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_full_size_workload(name):
    w = wl.WORKLOADS[name]
    x, g, b, dy = wl.make_inputs(w, "cuda")
    outs = pu.run_gpu(x, g, b, dy, w.eps, w.mode)
    assert gb.norm_get_device_error() == 0
    nsample = 256 if w.N <= 8192 else 48
    rows = pu.sample_rows(w.M, nsample, seed=w.M + w.N)
    pu.compare(w.mode, w.eps, x, g, b, dy, outs, rows=rows, label=name)
    y, rstd, mean, dx, dg, db = outs
    # every row: finite outputs, positive rstd
    assert torch.isfinite(rstd).all() and (rstd > 0).all()
    assert torch.isfinite(y.float()).all() and torch.isfinite(dx.float()).all()
    if w.mode == wl.LAYER:
        dxf = dx.float()
        rowsum = dxf.sum(dim=1, dtype=torch.float64)
        bound = 2.0 ** -7 * dxf.abs().sum(dim=1, dtype=torch.float64) + 1e-30
        bad = (rowsum.abs() > bound).sum().item()
        assert bad == 0, f"{name}: {bad} rows with sum(dx) != 0"
