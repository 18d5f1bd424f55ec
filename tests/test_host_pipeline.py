"""norm_fwd_bwd_host: forward + backward on host tensors, streamed through
device buffers in chunks.  y, rstd, mean and dx must equal the device entry
points' bit for bit; dgamma / dbeta (summed per chunk, then over chunks)
must match the oracle and be reproducible."""
import numpy as np
import pytest
import torch

import memory_bound_normalization_rmsnorm_gb300 as gb
from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

import oracle
import parity_util as pu
import tolerances

pytestmark = pytest.mark.gpu


def _host(t, pin=True):
    t = t.cpu()
    return t.pin_memory() if pin else t


def _device_ref(case, x, g, b, dy):
    y, rs, mu = gb.norm_fwd(x, g, b, case.eps, case.mode)
    dx, dg, db = gb.norm_bwd(dy, x, g, rs, mu, case.mode)
    torch.cuda.synchronize()
    return y, rs, mu, dx, dg, db


@pytest.mark.parametrize("mode", [0, 1], ids=["rms", "layer"])
@pytest.mark.parametrize("M,N,chunk", [(1031, 1024, 100), (257, 4096, 0), (3000, 2048, 1000),
                                       (5, 512, 2), (64, 8192, 64),
                                       # streamed long rows (backward; and the
                                       # RMSNorm forward beyond 262144 columns)
                                       (40, 131072, 16), (10, 524288, 4)])
@pytest.mark.parametrize("pin", [True, False], ids=["pinned", "pageable"])
def test_host_pipeline_matches_device_path(M, N, chunk, mode, pin):
    base = wl.WORKLOADS["layer_32768x4096" if mode else "rms_262144x1024_outliers"]
    case = wl.like(base, M, N)
    x, g, b, dy = [None if t is None else t.cuda() for t in wl.make_inputs(case, "cpu")]
    ref = _device_ref(case, x, g, b, dy)
    outs = gb.norm_fwd_bwd_host(_host(x, pin), _host(dy, pin), _host(g, pin),
                                None if b is None else _host(b, pin), case.eps, mode,
                                chunk_rows=chunk)
    torch.cuda.synchronize()
    y, rs, mu, dx, dg, db = outs
    assert torch.equal(y, ref[0].cpu()) and torch.equal(rs, ref[1].cpu())
    assert torch.equal(dx, ref[3].cpu())
    if mode == 1:
        assert torch.equal(mu, ref[2].cpu())
    # column sums: against the oracle (over all rows), and reproducible
    eps64 = float(np.float32(case.eps))
    dg_ref, db_ref, dg_abs, db_abs = oracle.param_grads_bf16(
        wl.bf16_bits(dy), wl.bf16_bits(x), wl.bf16_bits(g), eps64, mode)
    tolerances.check_t2(dg.double().numpy(), dg_ref, dg_abs, "dgamma")
    if mode == 1:
        tolerances.check_t2(db.double().numpy(), db_ref, db_abs, "dbeta")
    again = gb.norm_fwd_bwd_host(_host(x, pin), _host(dy, pin), _host(g, pin),
                                 None if b is None else _host(b, pin), case.eps, mode,
                                 chunk_rows=chunk)
    torch.cuda.synchronize()
    assert torch.equal(again[4], dg) and (mode == 0 or torch.equal(again[5], db))
    assert gb.norm_get_device_error() == 0


def test_host_pipeline_full_size_headline():
    w = wl.WORKLOADS["layer_32768x4096"]
    x, g, b, dy = wl.make_inputs(w, "cuda")
    ref = _device_ref(w, x, g, b, dy)
    outs = gb.norm_fwd_bwd_host(_host(x), _host(dy), _host(g), _host(b), w.eps, w.mode)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], ref[0].cpu()) and torch.equal(outs[3], ref[3].cpu())
    assert torch.equal(outs[1], ref[1].cpu()) and torch.equal(outs[2], ref[2].cpu())
    rows = pu.sample_rows(w.M, 64, seed=9)
    eps64 = float(np.float32(w.eps))
    y_ref, _, _ = oracle.fwd_bf16(wl.bf16_bits(x), wl.bf16_bits(g), wl.bf16_bits(b), eps64,
                                  w.mode, rows=rows)
    tolerances.check_t1(outs[0][rows].double().numpy(), y_ref, "y")
    dg_ref, db_ref, dg_abs, db_abs = oracle.param_grads_bf16(
        wl.bf16_bits(dy), wl.bf16_bits(x), wl.bf16_bits(g), eps64, w.mode)
    tolerances.check_t2(outs[4].double().numpy(), dg_ref, dg_abs, "dgamma")
    tolerances.check_t2(outs[5].double().numpy(), db_ref, db_abs, "dbeta")


def test_host_pipeline_argument_errors():
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    g = torch.ones(64, dtype=torch.bfloat16)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(gb.NormError) as e:
        gb.norm_fwd_bwd_host(x, x, g, None, 1e-6, 0, workspace=ws)
    assert e.value.status == 5  # workspace too small
    big = torch.empty(gb.norm_host_workspace_bytes(4, 64, 0) + 256, dtype=torch.uint8,
                      device="cuda")
    with pytest.raises(gb.NormError) as e:
        gb.norm_fwd_bwd_host(x, x, g, None, 1e-6, 0, workspace=big[8:])
    assert e.value.status == 3  # misaligned
