"""Plain fp64 CPU oracle for RMSNorm / LayerNorm forward and backward.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module; the library and its
binding never do.  The arithmetic lives in ``oracle.c`` (its header gives the
definitions and the page passages they follow: the LayerNorm/RMSNorm and
backward-pass paragraphs of "PyTorch atinge desempenho SOTA em normalizacao
com torch.compile").  This file only compiles that C file with gcc and
marshals numpy arrays to it.

bf16 tensors are passed as their raw uint16 bit patterns.  Outputs are fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

RMS = 0
LAYER = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_lock = threading.Lock()
_default = None

_dp = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u8p = ctypes.POINTER(ctypes.c_uint8)

FP8_ROW = 0
FP8_MX = 1


def compile_c(src: str, out: str) -> str:
    """gcc -O2 without fast-math or FMA contraction, so every operation is an
    IEEE double operation in source order."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.c (skipped when the shared object is newer)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(SRC)):
        return _LIB
    return compile_c(SRC, _LIB)


def _ptr(a, typ):
    if a is None:
        return ctypes.cast(None, typ)
    return a.ctypes.data_as(typ)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs are passed as uint16 bit patterns")
    return a


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what} failed with code {rc}")


def _rows(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r, int(r.size)


class Oracle:
    """ctypes view of one compiled oracle shared object."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oracle_fwd_f64.argtypes = [_dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_double, ctypes.c_int, _dp, _dp, _dp]
        lib.oracle_bwd_f64.argtypes = [_dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_double, ctypes.c_int, _dp, _dp, _dp]
        lib.oracle_fwd_bf16.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_double, ctypes.c_int,
                                        _i64p, ctypes.c_int64, _dp, _dp, _dp]
        lib.oracle_bwd_dx_bf16.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_double, ctypes.c_int,
                                           _i64p, ctypes.c_int64, _dp]
        lib.oracle_param_grads_bf16.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int64,
                                                ctypes.c_int64, ctypes.c_double,
                                                ctypes.c_int, _dp, _dp, _dp, _dp]
        lib.oracle_residual_add_bf16.argtypes = [_u16p, _u16p, ctypes.c_int64,
                                                 ctypes.c_int64, _u16p]
        lib.oracle_add_bwd_dx_bf16.argtypes = [_u16p, _u16p, _u16p, _u16p, ctypes.c_int64,
                                               ctypes.c_int64, ctypes.c_double, ctypes.c_int,
                                               _i64p, ctypes.c_int64, _dp]
        _u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_e4m3_encode.argtypes = [_dp, ctypes.c_int64, _u8p]
        lib.oracle_e4m3_decode.argtypes = [_u8p, ctypes.c_int64, _dp]
        lib.oracle_fwd_fp8_bf16.argtypes = [_u16p, _u16p, _u16p, _u16p, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_double, ctypes.c_int,
                                            ctypes.c_int, _i64p, ctypes.c_int64, _dp, _u8p,
                                            _dp, _dp, _u8p]
        lib.oracle_norm_gemm_bf16.argtypes = [_u16p, _u16p, _u16p, _u16p, ctypes.c_int64,
                                              ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
                                              ctypes.c_int, _i64p, ctypes.c_int64, _dp, _dp,
                                              _dp]
        for f in (lib.oracle_fwd_f64, lib.oracle_bwd_f64, lib.oracle_fwd_bf16,
                  lib.oracle_bwd_dx_bf16, lib.oracle_param_grads_bf16,
                  lib.oracle_residual_add_bf16, lib.oracle_add_bwd_dx_bf16,
                  lib.oracle_e4m3_encode, lib.oracle_e4m3_decode, lib.oracle_fwd_fp8_bf16,
                  lib.oracle_norm_gemm_bf16):
            f.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    # -------------------------------------------------------------- fp64 API
    def fwd_f64(self, x, gamma, beta, eps, mode):
        """Forward on double inputs.  x: [M, N]. Returns (y, rstd, mean)."""
        x = _f64(x)
        M, N = x.shape
        gamma = _f64(gamma)
        beta = None if beta is None else _f64(beta)
        y = np.empty((M, N), np.float64)
        rstd = np.empty(M, np.float64)
        mean = np.empty(M, np.float64)
        _check(self.lib.oracle_fwd_f64(_ptr(x, _dp), _ptr(gamma, _dp), _ptr(beta, _dp),
                                       M, N, float(eps), int(mode), _ptr(y, _dp),
                                       _ptr(rstd, _dp), _ptr(mean, _dp)), "oracle_fwd_f64")
        return y, rstd, mean

    def bwd_f64(self, dy, x, gamma, eps, mode):
        """Backward on double inputs. Returns (dx, dgamma, dbeta); dbeta is the
        column sum of dy in LayerNorm mode and zeros in RMSNorm mode."""
        x = _f64(x)
        dy = _f64(dy)
        M, N = x.shape
        gamma = _f64(gamma)
        dx = np.empty((M, N), np.float64)
        dg = np.empty(N, np.float64)
        db = np.empty(N, np.float64)
        _check(self.lib.oracle_bwd_f64(_ptr(dy, _dp), _ptr(x, _dp), _ptr(gamma, _dp),
                                       M, N, float(eps), int(mode), _ptr(dx, _dp),
                                       _ptr(dg, _dp), _ptr(db, _dp)), "oracle_bwd_f64")
        return dx, dg, db

    # -------------------------------------------------------------- bf16 API
    def fwd_bf16(self, x_bits, gamma_bits, beta_bits, eps, mode, rows=None):
        """Forward on bf16 bit patterns, for all rows or the listed ones.
        Returns (y [R, N], rstd [R], mean [R]) in fp64."""
        x_bits = _u16(x_bits)
        M, N = x_bits.shape
        gamma_bits = _u16(gamma_bits)
        beta_bits = None if beta_bits is None else _u16(beta_bits)
        r, R = _rows(rows, M)
        y = np.empty((R, N), np.float64)
        rstd = np.empty(R, np.float64)
        mean = np.empty(R, np.float64)
        _check(self.lib.oracle_fwd_bf16(_ptr(x_bits, _u16p), _ptr(gamma_bits, _u16p),
                                        _ptr(beta_bits, _u16p), M, N, float(eps),
                                        int(mode), _ptr(r, _i64p), R, _ptr(y, _dp),
                                        _ptr(rstd, _dp), _ptr(mean, _dp)),
               "oracle_fwd_bf16")
        return y, rstd, mean

    def bwd_dx_bf16(self, dy_bits, x_bits, gamma_bits, eps, mode, rows=None):
        """dx on bf16 bit patterns for all rows or the listed ones (fp64)."""
        x_bits = _u16(x_bits)
        dy_bits = _u16(dy_bits)
        M, N = x_bits.shape
        gamma_bits = _u16(gamma_bits)
        r, R = _rows(rows, M)
        dx = np.empty((R, N), np.float64)
        _check(self.lib.oracle_bwd_dx_bf16(_ptr(dy_bits, _u16p), _ptr(x_bits, _u16p),
                                           _ptr(gamma_bits, _u16p), M, N, float(eps),
                                           int(mode), _ptr(r, _i64p), R, _ptr(dx, _dp)),
               "oracle_bwd_dx_bf16")
        return dx

    def param_grads_bf16(self, dy_bits, x_bits, gamma_bits, eps, mode):
        """Column reductions over all rows: (dgamma, dbeta, dgamma_abs,
        dbeta_abs), the last two being sums of |summand| (tolerance scales)."""
        x_bits = _u16(x_bits)
        dy_bits = _u16(dy_bits)
        M, N = x_bits.shape
        gamma_bits = _u16(gamma_bits)
        out = [np.empty(N, np.float64) for _ in range(4)]
        _check(self.lib.oracle_param_grads_bf16(_ptr(dy_bits, _u16p), _ptr(x_bits, _u16p),
                                                _ptr(gamma_bits, _u16p), M, N, float(eps),
                                                int(mode), *[_ptr(o, _dp) for o in out]),
               "oracle_param_grads_bf16")
        return tuple(out)


    # ------------------------------------------------ fused residual add
    def residual_add_bf16(self, x_bits, r_bits):
        """h = bf16(x + r) (sum in binary32, round to nearest even), bits."""
        x_bits = _u16(x_bits)
        r_bits = _u16(r_bits)
        assert x_bits.shape == r_bits.shape
        M, N = x_bits.shape
        h = np.empty((M, N), np.uint16)
        _check(self.lib.oracle_residual_add_bf16(_ptr(x_bits, _u16p), _ptr(r_bits, _u16p),
                                                 M, N, _ptr(h, _u16p)),
               "oracle_residual_add_bf16")
        return h

    def add_fwd_bf16(self, x_bits, r_bits, gamma_bits, beta_bits, eps, mode, rows=None):
        """Fused residual add + norm forward: (h bits, y, rstd, mean)."""
        h = self.residual_add_bf16(x_bits, r_bits)
        y, rstd, mean = self.fwd_bf16(h, gamma_bits, beta_bits, eps, mode, rows=rows)
        return h, y, rstd, mean

    def add_bwd_dx_bf16(self, dy_bits, h_bits, dh_bits, gamma_bits, eps, mode, rows=None):
        """dx = norm backward of dy at h, plus dh (fp64)."""
        h_bits = _u16(h_bits)
        dy_bits = _u16(dy_bits)
        dh_bits = _u16(dh_bits)
        M, N = h_bits.shape
        gamma_bits = _u16(gamma_bits)
        r, R = _rows(rows, M)
        dx = np.empty((R, N), np.float64)
        _check(self.lib.oracle_add_bwd_dx_bf16(_ptr(dy_bits, _u16p), _ptr(h_bits, _u16p),
                                               _ptr(dh_bits, _u16p), _ptr(gamma_bits, _u16p),
                                               M, N, float(eps), int(mode), _ptr(r, _i64p), R,
                                               _ptr(dx, _dp)), "oracle_add_bwd_dx_bf16")
        return dx

    # ------------------------------------------------------------ FP8 (E4M3)
    def e4m3_encode(self, v):
        """Nearest E4M3 codes (uint8) of fp64 values: ties to even,
        saturating at +-448, NaN -> 0x7F."""
        v = _f64(v)
        out = np.empty(v.shape, np.uint8)
        _check(self.lib.oracle_e4m3_encode(_ptr(v, _dp), v.size, _ptr(out, _u8p)),
               "oracle_e4m3_encode")
        return out

    def e4m3_decode(self, codes):
        """Exact fp64 values of E4M3 codes (NaN for S.1111.111)."""
        c = np.ascontiguousarray(codes, dtype=np.uint8)
        out = np.empty(c.shape, np.float64)
        _check(self.lib.oracle_e4m3_decode(_ptr(c, _u8p), c.size, _ptr(out, _dp)),
               "oracle_e4m3_decode")
        return out

    def fwd_fp8_bf16(self, x_bits, r_bits, gamma_bits, beta_bits, eps, mode, scaling,
                     rows=None):
        """Forward with E4M3 output (scaling FP8_ROW or FP8_MX), optionally on
        h = bf16(x + r).  Returns dict y (fp64 [R, N]), q (uint8 [R, N]),
        amax, scale (fp64 [R] or [R, N/32]) and, for MX, ebyte (uint8)."""
        x_bits = _u16(x_bits)
        M, N = x_bits.shape
        r_bits = None if r_bits is None else _u16(r_bits)
        gamma_bits = _u16(gamma_bits)
        beta_bits = None if beta_bits is None else _u16(beta_bits)
        r, R = _rows(rows, M)
        ns = (R,) if scaling == FP8_ROW else (R, N // 32)
        y = np.empty((R, N), np.float64)
        q = np.empty((R, N), np.uint8)
        amax = np.empty(ns, np.float64)
        scale = np.empty(ns, np.float64)
        ebyte = np.zeros(ns, np.uint8)
        _check(self.lib.oracle_fwd_fp8_bf16(
            _ptr(x_bits, _u16p), _ptr(r_bits, _u16p), _ptr(gamma_bits, _u16p),
            _ptr(beta_bits, _u16p), M, N, float(eps), int(mode), int(scaling), _ptr(r, _i64p), R,
            _ptr(y, _dp), _ptr(q, _u8p), _ptr(amax, _dp), _ptr(scale, _dp), _ptr(ebyte, _u8p)),
            "oracle_fwd_fp8_bf16")
        out = {"y": y, "q": q, "amax": amax, "scale": scale}
        if scaling == FP8_MX:
            out["ebyte"] = ebyte
        return out


    # ------------------------------------------- norm feeding a GEMM
    def norm_gemm_bf16(self, x_bits, gamma_bits, beta_bits, w_bits, eps, mode, rows=None):
        """out = norm(x) @ W^T in fp64, W [Nout, K] (one row per output
        feature), for all rows of x or the listed ones.  y = norm(x) is the
        unrounded fp64 forward.  Returns (out [R, Nout], rstd [R], mean [R])."""
        x_bits = _u16(x_bits)
        M, K = x_bits.shape
        w_bits = _u16(w_bits)
        Nout, K2 = w_bits.shape
        if K2 != K:
            raise ValueError("W must be [Nout, K]")
        gamma_bits = _u16(gamma_bits)
        beta_bits = None if beta_bits is None else _u16(beta_bits)
        r, R = _rows(rows, M)
        out = np.empty((R, Nout), np.float64)
        rstd = np.empty(R, np.float64)
        mean = np.empty(R, np.float64)
        _check(self.lib.oracle_norm_gemm_bf16(
            _ptr(x_bits, _u16p), _ptr(gamma_bits, _u16p), _ptr(beta_bits, _u16p),
            _ptr(w_bits, _u16p), M, K, Nout, float(eps), int(mode), _ptr(r, _i64p), R,
            _ptr(out, _dp), _ptr(rstd, _dp), _ptr(mean, _dp)), "oracle_norm_gemm_bf16")
        return out, rstd, mean


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def fwd_f64(*a, **k):
    return default().fwd_f64(*a, **k)


def bwd_f64(*a, **k):
    return default().bwd_f64(*a, **k)


def fwd_bf16(*a, **k):
    return default().fwd_bf16(*a, **k)


def bwd_dx_bf16(*a, **k):
    return default().bwd_dx_bf16(*a, **k)


def param_grads_bf16(*a, **k):
    return default().param_grads_bf16(*a, **k)


def residual_add_bf16(*a, **k):
    return default().residual_add_bf16(*a, **k)


def add_fwd_bf16(*a, **k):
    return default().add_fwd_bf16(*a, **k)


def add_bwd_dx_bf16(*a, **k):
    return default().add_bwd_dx_bf16(*a, **k)


def e4m3_encode(*a, **k):
    return default().e4m3_encode(*a, **k)


def e4m3_decode(*a, **k):
    return default().e4m3_decode(*a, **k)


def fwd_fp8_bf16(*a, **k):
    return default().fwd_fp8_bf16(*a, **k)


def norm_gemm_bf16(*a, **k):
    return default().norm_gemm_bf16(*a, **k)


def bf16_bits_to_f64(bits):
    """Exact widening of bf16 bit patterns to float64 (numpy only)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
