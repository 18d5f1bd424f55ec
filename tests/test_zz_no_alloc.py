"""norm_bwd_noalloc: the backward pass for callers that may not allocate
device memory (their memory belongs to a framework pool or a pre-reserved
arena, or an allocation's possible device synchronisation is not allowed on
their path).  It runs with the library's fixed 16 MiB device scratch array
instead of a caller workspace.

Called through the C ABI and compared with norm_bwd (which takes a caller
workspace) on two calls in a row, with the same tolerances as the parity
tests; the second call also shows that what the first left in the shared
array does not leak into the result.  This file is collected last so that a
run stopping at the first failure has run every other test before it.
"""
import ctypes

import pytest
import torch

import memory_bound_normalization_rmsnorm_gb300 as gb
from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

import parity_util as pu
import tolerances

pytestmark = pytest.mark.gpu

CASES = [
    ("layer_32768x4096", 4099, 4096),
    ("rms_262144x768_outliers", 20001, 768),
    ("rms_4096x131072", 37, 131072),
    ("layer_32768x5120_resid", 1001, 5120),
    ("layer_32768x4096", 6, 524288),  # rows wide enough for the two-pass path
]


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("name,M,N", CASES)
def test_noalloc_matches_workspace_entry_point(name, M, N, monkeypatch):
    case = wl.like(wl.WORKLOADS[name], M, N)
    x, g, b, dy = [None if t is None else t.cuda() for t in wl.make_inputs(case, "cpu")]
    mode = case.mode
    y, rstd, mean = gb.norm_fwd(x, g, b, case.eps, mode)
    if gb.norm_bwd_workspace_bytes(M, N, mode) > 16 << 20:
        # the streaming backward's partial rows do not fit the array: the
        # entry point runs the resident long-row plan, as stream=0 does
        assert gb.norm_plan(M, N, mode, True)["streamed"] == 1
        monkeypatch.setenv("GBNORM_PLAN", "stream=0")
    dx_ref, dg_ref, db_ref = gb.norm_bwd(dy, x, g, rstd, mean, mode)
    torch.cuda.synchronize()
    assert gb.norm_bwd_workspace_bytes(M, N, mode) <= 16 << 20
    monkeypatch.delenv("GBNORM_PLAN", raising=False)
    L = gb.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        dx = torch.full_like(x, float("nan"))
        dg = torch.full((N,), float("nan"), device="cuda")
        db = torch.full((N,), float("nan"), device="cuda") if mode == wl.LAYER else None
        st = L.norm_bwd_noalloc(_p(dy), _p(x), _p(g), _p(rstd), _p(mean), M, N, mode,
                                _p(dx), _p(dg), _p(db), stream)
        assert st == 0, gb.strerror(st)
        torch.cuda.synchronize()
        tolerances.check_t1(pu.f64(dx), pu.f64(dx_ref), f"{name} call {call} dx")
        tolerances.check_t2(pu.f64(dg), pu.f64(dg_ref), None, f"{name} call {call} dgamma")
        if db is not None:
            tolerances.check_t2(pu.f64(db), pu.f64(db_ref), None, f"{name} call {call} dbeta")
        # Same kernels, same launch plan: the results are in fact identical.
        assert torch.equal(dx, dx_ref) and torch.equal(dg, dg_ref)
        if db is not None:
            assert torch.equal(db, db_ref)
    assert gb.norm_get_device_error() == 0


def test_noalloc_rejects_shapes_beyond_its_array(monkeypatch):
    """A launch plan whose scratch need exceeds 16 MiB is refused with
    NORM_ERR_WORKSPACE before anything is launched.  (With the library's
    default plans every supported shape fits, the streaming backward through
    its fallback; a plan override with one CTA per row and 152+ partial rows
    makes LayerNorm 4096 x 16384 need about 20 MB.)"""
    M, N = 4096, 16384
    monkeypatch.setenv("GBNORM_PLAN", "C=1,tpr=512")
    need = gb.norm_bwd_workspace_bytes(M, N, wl.LAYER)
    assert need > 16 << 20
    L = gb.lib()
    F = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    st = L.norm_bwd_noalloc(F, F, F, F, F, M, N, wl.LAYER, F, F, F, None)
    assert st == 5  # NORM_ERR_WORKSPACE
