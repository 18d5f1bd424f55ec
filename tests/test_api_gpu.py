"""The C ABI on a device: status codes for bad arguments (checked before any
launch, so nothing faults), guard bands around every output, non-default
streams, the workspace contract and the device error word."""
import ctypes

import pytest
import torch

import memory_bound_normalization_rmsnorm_gb300 as gb
from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

L = None


def lib():
    global L
    if L is None:
        L = gb.lib()
    return L


def _p(t, off=0):
    return ctypes.c_void_p(t.data_ptr() + off)


def _inputs(M=64, N=1024, mode=1):
    case = wl.like(wl.WORKLOADS["layer_32768x4096" if mode else "rms_256x1024"], M, N)
    return [None if t is None else t.cuda() for t in wl.make_inputs(case, "cpu")]


def test_status_codes_on_device():
    x, g, b, dy = _inputs()
    M, N = x.shape
    y = torch.empty_like(x)
    r = torch.empty(M, device="cuda")
    m = torch.empty(M, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    f = lib().norm_fwd
    assert f(_p(x), _p(g), _p(b), M, N, 1e-5, 1, _p(y), _p(r), _p(m), s) == 0
    assert f(_p(x, 2), _p(g), _p(b), M, N, 1e-5, 1, _p(y), _p(r), _p(m), s) == 3
    assert f(_p(x), _p(g), _p(b), M, N, 1e-5, 1, _p(y, 8), _p(r), _p(m), s) == 3
    assert f(_p(x), _p(g), _p(b), M, N, 1e-5, 1, _p(y), _p(r, 4), _p(m), s) == 3
    assert f(_p(x), _p(g), _p(b), M, N, 1e-5, 0, _p(y), _p(r), _p(m), s) == 4  # RMS + mean
    assert f(_p(x), _p(g), _p(b), M, N, 1e-5, 1, _p(y), _p(r), None, s) == 4    # LN no mean
    assert f(_p(x), _p(g), _p(b), M, N, 1e-5, 7, _p(y), _p(r), _p(m), s) == 4
    assert f(_p(x), _p(g), _p(b), M, N - 4, 1e-5, 1, _p(y), _p(r), _p(m), s) == 2
    assert f(_p(x), _p(g), _p(b), 0, N, 1e-5, 1, _p(y), _p(r), _p(m), s) == 2
    assert f(_p(x), _p(g), _p(b), M, N, -1.0, 1, _p(y), _p(r), _p(m), s) == 9
    assert f(_p(x), _p(g), _p(b), M, N, float("nan"), 1, _p(y), _p(r), _p(m), s) == 9
    assert f(None, _p(g), _p(b), M, N, 1e-5, 1, _p(y), _p(r), _p(m), s) == 1
    # backward: workspace contract
    need = gb.norm_bwd_workspace_bytes(M, N, 1)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dx = torch.empty_like(x)
    dg = torch.empty(N, device="cuda")
    db = torch.empty(N, device="cuda")
    bw = lib().norm_bwd
    args = [_p(dy), _p(x), _p(g), _p(r), _p(m), M, N, 1, _p(dx), _p(dg), _p(db)]
    assert bw(*args, _p(ws), need, s) == 0
    assert bw(*args, _p(ws), need - 16, s) == 5
    assert bw(*args, None, need, s) == 5
    assert bw(*args, _p(ws, 8), need, s) == 3
    args_rms = [_p(dy), _p(x), _p(g), _p(r), None, M, N, 0, _p(dx), _p(dg), _p(db)]
    assert bw(*args_rms, _p(ws), need, s) == 4  # RMS with dbeta
    torch.cuda.synchronize()
    assert gb.norm_get_device_error() == 0


@pytest.mark.parametrize("mode,N", [(0, 256), (1, 4096), (0, 131072), (1, 776)])
def test_guard_bands(mode, N):
    """Outputs are written inside guard-banded buffers; the bands (4 KB on
    each side, a fixed byte pattern) must be untouched."""
    M = 33 if N < 100000 else 5
    x, g, b, dy = _inputs(M, N, mode)
    G = 4096

    def banded(nbytes):
        buf = torch.full((nbytes + 2 * G,), 0xA5, dtype=torch.uint8, device="cuda")
        return buf, buf[G:G + nbytes]

    yb, y = banded(M * N * 2)
    rb, r = banded(M * 4)
    mb, m = banded(M * 4)
    dxb, dx = banded(M * N * 2)
    dgb, dg = banded(N * 4)
    dbb, db = banded(N * 4)
    need = gb.norm_bwd_workspace_bytes(M, N, mode)
    wsb, ws = banded(need)
    y, dx = y.view(torch.bfloat16).view(M, N), dx.view(torch.bfloat16).view(M, N)
    r, m, dg, db = r.view(torch.float32), m.view(torch.float32), dg.view(torch.float32), db.view(torch.float32)
    gb.norm_fwd(x, g, b, 1e-5, mode, y=y, rstd=r, mean=m if mode else None)
    gb.norm_bwd(dy, x, g, r, m if mode else None, mode, dx=dx, dgamma=dg,
                dbeta=db if mode else None, workspace=ws)
    torch.cuda.synchronize()
    for buf in (yb, rb, mb, dxb, dgb, dbb, wsb):
        assert torch.all(buf[:G] == 0xA5) and torch.all(buf[-G:] == 0xA5)


def test_side_stream_and_error_word():
    x, g, b, dy = _inputs(4096, 2048, 1)
    s = torch.cuda.Stream()
    y0, r0, m0 = gb.norm_fwd(x, g, b, 1e-5, 1)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        y1, r1, m1 = gb.norm_fwd(x, g, b, 1e-5, 1)
        dx1, dg1, db1 = gb.norm_bwd(dy, x, g, r1, m1, 1)
    s.synchronize()
    assert torch.equal(y0, y1) and torch.equal(r0, r1)
    dx0, dg0, db0 = gb.norm_bwd(dy, x, g, r0, m0, 1, stream=s)
    s.synchronize()
    assert torch.equal(dx0, dx1) and torch.equal(dg0, dg1) and torch.equal(db0, db1)
    assert gb.norm_get_device_error(stream=s) == 0


def test_plan_query_matches_device():
    """norm_plan on the device reports a persistent grid within the SM count."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for M, N, mode in ((32768, 4096, 1), (262144, 256, 0), (4096, 131072, 0)):
        for bwd in (False, True):
            p = gb.norm_plan(M, N, mode, bwd)
            assert 1 <= p["grid"] <= 4 * sms and p["grid"] % p["cluster"] == 0


def test_bounded_wait_failure_path():
    """A wait that nothing completes gives up after its poll limit, records
    the timeout in the device error word and lets the kernel return: the
    status is reported once, then cleared, and the context keeps working."""
    L = lib()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert gb.norm_get_device_error() == 0
    assert L.norm_selftest_wait_timeout(1000, s) == 0
    assert gb.norm_get_device_error() == 8  # NORM_ERR_DEVICE_TIMEOUT
    assert gb.norm_get_device_error() == 0  # cleared by the read
    x, g, b, dy = _inputs(64, 1024, 1)
    y, r, m = gb.norm_fwd(x, g, b, 1e-5, 1)
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()
    assert gb.norm_get_device_error() == 0
