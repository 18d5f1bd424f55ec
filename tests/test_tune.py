"""Plan tuning (norm_tune_fwd / norm_tune_bwd): the chosen plan is valid,
installed for later calls and reported by norm_plan, its results match the
oracle and are reproducible, and norm_tune_reset brings the default back."""
import pytest
import torch

import memory_bound_normalization_rmsnorm_gb300 as gb
from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

import launch_check
import parity_util as pu

pytestmark = pytest.mark.gpu

OPTIN = 232448


@pytest.mark.parametrize("mode,M,N", [(1, 8192, 4096), (0, 65536, 1024), (1, 4097, 3072),
                                      (0, 3000, 8192)])
def test_tuned_plans(mode, M, N):
    base = wl.WORKLOADS["layer_32768x4096" if mode else "rms_262144x1024_outliers"]
    case = wl.like(base, M, N)
    x, g, b, dy = [None if t is None else t.cuda() for t in wl.make_inputs(case, "cpu")]
    gb.norm_tune_reset()
    default_f = gb.norm_plan(M, N, mode, False)
    default_b = gb.norm_plan(M, N, mode, True)
    cf = gb.norm_tune_fwd(x, g, b, case.eps, mode, iters=5)
    assert gb.norm_plan(M, N, mode, False) == cf
    y, rs, mu = gb.norm_fwd(x, g, b, case.eps, mode)
    cb = gb.norm_tune_bwd(dy, x, g, rs, mu, mode, iters=5)
    assert gb.norm_plan(M, N, mode, True) == cb
    for p, bwd in ((cf, False), (cb, True)):
        launch_check.check_plan(p, M, N, mode, bwd, OPTIN)
    outs = pu.run_gpu(x, g, b, dy, case.eps, mode)
    pu.compare(mode, case.eps, x, g, b, dy, outs, label=f"tuned {mode} {M}x{N}")
    again = pu.run_gpu(x, g, b, dy, case.eps, mode)
    for u, v in zip(outs, again):
        assert (u is None and v is None) or torch.equal(u, v)
    gb.norm_tune_reset()
    assert gb.norm_plan(M, N, mode, False) == default_f
    assert gb.norm_plan(M, N, mode, True) == default_b
    assert gb.norm_get_device_error() == 0


def test_tuning_refused_under_plan_override(monkeypatch):
    x = torch.zeros(8, 256, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(256, dtype=torch.bfloat16, device="cuda")
    monkeypatch.setenv("GBNORM_PLAN", "S=2")
    with pytest.raises(gb.NormError) as e:
        gb.norm_tune_fwd(x, g, None, 1e-6, 0)
    assert e.value.status == 9
