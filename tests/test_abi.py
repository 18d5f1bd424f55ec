"""The C ABI library without a GPU: it loads, exports every function that
include/gbnorm.h declares, and rejects bad arguments with the documented
status codes before touching CUDA."""
import ctypes
import os

import pytest
import torch

import memory_bound_normalization_rmsnorm_gb300 as gb


def test_exports_every_declared_symbol():
    names = gb.declared_functions()
    assert set(names) >= {"norm_fwd", "norm_bwd", "norm_bwd_workspace_bytes",
                          "norm_strerror", "norm_get_device_error", "norm_plan",
                          "norm_bwd_noalloc", "norm_selftest_wait_timeout"}
    L = ctypes.CDLL(gb.library_path())
    for n in names:
        assert hasattr(L, n), f"{n} declared in gbnorm.h but not exported"


def test_library_is_in_tree():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    assert os.path.commonpath([gb.library_path(), root]) == root


def test_strerror_covers_all_codes():
    seen = set()
    for code in range(11):
        s = gb.strerror(code)
        assert s and s != "unknown status"
        seen.add(s)
    assert len(seen) == 11
    assert gb.strerror(1234) == "unknown status"


F = 16  # a fake, 16-byte aligned address: validation fails before any use


def test_fwd_validation_codes():
    f = gb.lib().norm_fwd
    ok = dict(x=F, g=F, b=None, M=4, N=16, eps=1e-5, mode=0, y=F, r=F, m=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["x"], a["g"], a["b"], a["M"], a["N"], a["eps"], a["mode"], a["y"],
                 a["r"], a["m"], None)

    assert call(x=None) == 1
    assert call(y=None) == 1
    assert call(r=None) == 1
    assert call(M=0) == 2
    assert call(N=12) == 2
    assert call(N=0) == 2
    assert call(N=(1 << 24) + 8) == 2   # N > NORM_MAX_N
    assert call(mode=2) == 4
    assert call(b=F) == 4              # beta with RMSNorm
    assert call(m=F) == 4              # mean with RMSNorm
    assert call(mode=1) == 4           # LayerNorm without mean
    assert call(eps=-1e-5) == 9
    assert call(eps=float("inf")) == 9
    assert call(x=F + 8) == 3
    assert call(g=F + 2) == 3
    assert call(mode=1, m=F + 4) == 3


def test_fp8_validation_codes():
    f = gb.lib().norm_fwd_fp8
    ok = dict(x=F, res=None, g=F, b=None, M=4, N=64, eps=1e-5, mode=0, sc=0, h=None, q=F,
              s=F, r=F, m=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["x"], a["res"], a["g"], a["b"], a["M"], a["N"], a["eps"], a["mode"], a["sc"],
                 a["h"], a["q"], a["s"], a["r"], a["m"], None)

    assert call(x=None) == 1
    assert call(q=None) == 1
    assert call(s=None) == 1
    assert call(r=None) == 1
    assert call(res=F) == 1            # residual without h
    assert call(h=F) == 9              # h without residual
    assert call(sc=2) == 9             # unknown scaling
    assert call(sc=1, N=48) == 2       # MX needs N % 32 == 0
    assert call(N=262144 + 32) == 2    # above NORM_MAX_N_FUSED
    assert call(N=12) == 2
    assert call(mode=2) == 4
    assert call(b=F) == 4
    assert call(mode=1) == 4           # LayerNorm without mean
    assert call(eps=-1.0) == 9
    assert call(q=F + 8) == 3
    assert call(s=F + 4) == 3
    assert call(res=F + 2, h=F) == 3


def test_host_pipeline_validation_codes():
    f = gb.lib().norm_fwd_bwd_host
    ok = dict(x=F, dy=F, g=F, b=None, M=4, N=64, eps=1e-5, mode=0, y=F, dx=F, r=F, m=None,
              dg=F, db=None, cr=0, ws=F, wsb=1 << 20)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["x"], a["dy"], a["g"], a["b"], a["M"], a["N"], a["eps"], a["mode"], a["y"],
                 a["dx"], a["r"], a["m"], a["dg"], a["db"], a["cr"], a["ws"], a["wsb"], None)

    assert call(x=None) == 1
    assert call(dy=None) == 1
    assert call(dg=None) == 1
    assert call(mode=3) == 4
    assert call(b=F) == 4              # beta with RMSNorm
    assert call(db=F) == 4             # dbeta with RMSNorm
    assert call(mode=1) == 4           # LayerNorm without mean
    assert call(N=12) == 2
    assert call(M=0) == 2
    assert call(cr=-1) == 2
    assert call(eps=float("nan")) == 9
    n = ctypes.c_size_t(0)
    assert gb.lib().norm_host_workspace_bytes(4, 12, 0, 0, ctypes.byref(n)) == 2
    assert gb.lib().norm_host_workspace_bytes(4, 64, 0, 0, None) == 1


def test_tune_validation_codes():
    f = gb.lib().norm_tune_fwd
    assert f(F, F, None, 0, 64, ctypes.c_float(1e-5), 0, F, F, None, 5, None, None) == 2
    assert f(F, F, None, 4, 64, ctypes.c_float(1e-5), 7, F, F, None, 5, None, None) == 4
    assert f(F, F, None, 4, 64, ctypes.c_float(1e-5), 0, F, F, None, 0, None, None) == 9
    fb = gb.lib().norm_tune_bwd
    assert fb(F, F, F, F, None, 4, 12, 0, F, F, None, F, 64, 5, None, None) == 2
    assert fb(F, F, F, F, None, 4, 64, 0, F, F, None, F, 64, -1, None, None) == 9
    assert gb.lib().norm_tune_reset() == 0


def test_bwd_validation_codes():
    f = gb.lib().norm_bwd
    ok = dict(dy=F, x=F, g=F, r=F, m=None, M=4, N=16, mode=0, dx=F, dg=F, db=None, ws=F,
              wsb=1 << 20)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["dy"], a["x"], a["g"], a["r"], a["m"], a["M"], a["N"], a["mode"], a["dx"],
                 a["dg"], a["db"], a["ws"], a["wsb"], None)

    assert call(dy=None) == 1
    assert call(dg=None) == 1
    assert call(M=-1) == 2
    assert call(N=20) == 2
    assert call(db=F) == 4
    assert call(m=F) == 4
    assert call(mode=1) == 4
    assert call(ws=None) == 5
    assert call(ws=F + 4) == 3
    assert call(dx=F + 2) == 3


def test_norm_gemm_validation_codes():
    L = gb.lib()
    pf = L.norm_gemm_prepare
    okp = dict(w=F, g=F, b=None, K=128, Nout=64, mode=0, wg=F, u=None, v=None)

    def prep(**kw):
        a = dict(okp, **kw)
        return pf(a["w"], a["g"], a["b"], a["K"], a["Nout"], a["mode"], a["wg"], a["u"], a["v"],
                  None)

    assert prep(w=None) == 1
    assert prep(wg=None) == 1
    assert prep(mode=3) == 4
    assert prep(b=F) == 4                       # beta with RMSNorm
    assert prep(mode=1) == 4                    # LayerNorm without u, v
    assert prep(mode=1, u=F) == 4
    assert prep(K=96) == 2                      # K % 64
    assert prep(K=0) == 2
    assert prep(Nout=48) == 2                   # Nout % 32
    assert prep(g=F + 8) == 3
    assert prep(mode=1, u=F, v=F + 4) == 3

    ff = L.norm_gemm_fwd
    okf = dict(x=F, wg=F, u=None, v=None, M=5, K=128, Nout=64, eps=1e-5, mode=0, out=F, r=F,
               m=None)

    def fwd(**kw):
        a = dict(okf, **kw)
        return ff(a["x"], a["wg"], a["u"], a["v"], a["M"], a["K"], a["Nout"], a["eps"],
                  a["mode"], a["out"], a["r"], a["m"], None)

    assert fwd(x=None) == 1
    assert fwd(out=None) == 1
    assert fwd(r=None) == 1
    assert fwd(mode=2) == 4
    assert fwd(m=F) == 4                        # mean with RMSNorm
    assert fwd(mode=1, m=F) == 4                # LayerNorm without u, v
    assert fwd(mode=1, u=F, v=F) == 4           # LayerNorm without mean
    assert fwd(M=0) == 2
    assert fwd(M=65535 * 128 + 1) == 2
    assert fwd(K=100) == 2
    assert fwd(K=262144 + 64) == 2
    assert fwd(Nout=16) == 2
    assert fwd(Nout=80) == 2
    assert fwd(Nout=(1 << 20) + 32) == 2       # Nout <= 2^20
    assert fwd(eps=float("nan")) == 9
    assert fwd(eps=-1.0) == 9
    assert fwd(x=F + 2) == 3
    assert fwd(out=F + 8) == 3
    if not torch.cuda.is_available():
        assert fwd() == 7                       # valid arguments, no device


def test_selftest_argument_checks():
    L = gb.lib()
    assert L.norm_selftest_wait_timeout(0, None) == 9
    assert L.norm_selftest_wait_timeout((1 << 20) + 1, None) == 9


def test_plan_is_pure_host_arithmetic():
    """norm_plan for a described device works without any GPU and is
    deterministic."""
    a = gb.norm_plan(32768, 4096, 1, True, 152, 232448)
    b = gb.norm_plan(32768, 4096, 1, True, 152, 232448)
    assert a == b and a["grid"] >= 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device status")
def test_no_device_reports_cuda_error():
    with pytest.raises(gb.NormError) as e:
        gb.norm_bwd_workspace_bytes(128, 1024, 0)
    assert e.value.status == 7
