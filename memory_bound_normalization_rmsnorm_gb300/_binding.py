"""ctypes binding of libgbnorm.so (the C ABI of include/gbnorm.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of the library.  PyTorch supplies device memory (outputs and the
backward workspace are allocated with torch when the caller passes none) and
the stream (torch's current stream unless one is given).  There is no
fallback: if the shared library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from . import builder as _build

RMS = 0
LAYER = 1

STATUS = {
    0: "NORM_OK",
    1: "NORM_ERR_NULL",
    2: "NORM_ERR_SHAPE",
    3: "NORM_ERR_ALIGN",
    4: "NORM_ERR_MODE",
    5: "NORM_ERR_WORKSPACE",
    6: "NORM_ERR_UNSUPPORTED",
    7: "NORM_ERR_CUDA",
    8: "NORM_ERR_DEVICE_TIMEOUT",
    9: "NORM_ERR_ARG",
    10: "NORM_ERR_MEMORY",
}

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64


class Plan(ctypes.Structure):
    """Mirror of norm_plan_t."""
    _fields_ = [("cluster", ctypes.c_int32), ("cols_per_cta", ctypes.c_int32),
                ("threads_per_row", ctypes.c_int32), ("chunks_per_thread", ctypes.c_int32),
                ("groups", ctypes.c_int32), ("rows_per_group", ctypes.c_int32),
                ("rows_per_tile", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("tiles", ctypes.c_int64), ("grid", ctypes.c_int32),
                ("partials", ctypes.c_int32), ("exact", ctypes.c_int32),
                ("long_rows", ctypes.c_int32), ("param_smem_bytes", ctypes.c_int32),
                ("split_segments", ctypes.c_int32), ("streamed", ctypes.c_int32),
                ("wait_hint_ns", ctypes.c_int32), ("piece_cols", ctypes.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class NormError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({strerror(status)})")


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded ctypes library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it first "
                    "(python -m memory_bound_normalization_rmsnorm_gb300.builder)")
            L = ctypes.CDLL(path)
            L.norm_fwd.argtypes = [_vp, _vp, _vp, _i64, _i64, ctypes.c_float, ctypes.c_int,
                                   _vp, _vp, _vp, _vp]
            L.norm_fwd.restype = ctypes.c_int
            L.norm_bwd_workspace_bytes.argtypes = [_i64, _i64, ctypes.c_int,
                                                   ctypes.POINTER(ctypes.c_size_t)]
            L.norm_bwd_workspace_bytes.restype = ctypes.c_int
            L.norm_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_int, _vp,
                                   _vp, _vp, _vp, ctypes.c_size_t, _vp]
            L.norm_bwd.restype = ctypes.c_int
            L.norm_bwd_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_int,
                                           _vp, _vp, _vp, _vp]
            L.norm_bwd_noalloc.restype = ctypes.c_int
            L.norm_selftest_wait_timeout.argtypes = [ctypes.c_uint32, _vp]
            L.norm_selftest_wait_timeout.restype = ctypes.c_int
            L.norm_add_fwd.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_float,
                                       ctypes.c_int, _vp, _vp, _vp, _vp, _vp]
            L.norm_add_fwd.restype = ctypes.c_int
            L.norm_add_bwd_workspace_bytes.argtypes = [_i64, _i64, ctypes.c_int,
                                                       ctypes.POINTER(ctypes.c_size_t)]
            L.norm_add_bwd_workspace_bytes.restype = ctypes.c_int
            L.norm_add_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_int,
                                       _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
            L.norm_fwd_fp8.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_float,
                                       ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp]
            L.norm_fwd_fp8.restype = ctypes.c_int
            L.norm_tune_fwd.argtypes = [_vp, _vp, _vp, _i64, _i64, ctypes.c_float, ctypes.c_int,
                                        _vp, _vp, _vp, ctypes.c_int, ctypes.POINTER(Plan), _vp]
            L.norm_tune_fwd.restype = ctypes.c_int
            L.norm_tune_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_int, _vp,
                                        _vp, _vp, _vp, ctypes.c_size_t, ctypes.c_int,
                                        ctypes.POINTER(Plan), _vp]
            L.norm_tune_bwd.restype = ctypes.c_int
            L.norm_tune_reset.argtypes = []
            L.norm_tune_reset.restype = ctypes.c_int
            L.norm_host_workspace_bytes.argtypes = [_i64, _i64, ctypes.c_int, _i64,
                                                    ctypes.POINTER(ctypes.c_size_t)]
            L.norm_host_workspace_bytes.restype = ctypes.c_int
            L.norm_fwd_bwd_host.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_float,
                                            ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp, _i64,
                                            _vp, ctypes.c_size_t, _vp]
            L.norm_fwd_bwd_host.restype = ctypes.c_int
            L.norm_add_bwd.restype = ctypes.c_int
            L.norm_gemm_prepare.argtypes = [_vp, _vp, _vp, _i64, _i64, ctypes.c_int, _vp, _vp,
                                            _vp, _vp]
            L.norm_gemm_prepare.restype = ctypes.c_int
            L.norm_gemm_fwd.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_float,
                                        ctypes.c_int, _vp, _vp, _vp, _vp]
            L.norm_gemm_fwd.restype = ctypes.c_int
            L.norm_plan.argtypes = [_i64, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.POINTER(Plan)]
            L.norm_plan.restype = ctypes.c_int
            L.norm_strerror.argtypes = [ctypes.c_int]
            L.norm_strerror.restype = ctypes.c_char_p
            L.norm_get_device_error.argtypes = [_vp]
            L.norm_get_device_error.restype = ctypes.c_int
            _lib = L
    return _lib


def declared_functions():
    """Names of the functions include/gbnorm.h declares."""
    hdr = os.path.join(_build.INCLUDE, "gbnorm.h")
    text = open(hdr).read()
    return sorted(set(re.findall(r"^(?:norm_status_t|const char \*)\s*(norm_\w+)\(",
                                 text, flags=re.M)))


def strerror(status: int) -> str:
    try:
        return lib().norm_strerror(int(status)).decode()
    except RuntimeError:
        return STATUS.get(status, "unknown")


def _ptr(t):
    return None if t is None else _vp(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        return _vp(torch.cuda.current_stream(device).cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return _vp(stream.cuda_stream)
    return _vp(int(stream))


def _check_tensor(t, name, dtype, shape, device):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _rows(x):
    if x.dim() < 1:
        raise ValueError("x must have at least one dimension")
    N = x.shape[-1]
    M = x.numel() // N if N else 0
    return M, N


def norm_fwd(x, gamma, beta=None, eps=1e-5, mode=RMS, *, y=None, rstd=None, mean=None,
             stream=None):
    """Forward pass over the last dimension of x (bf16, contiguous).

    Returns (y, rstd, mean); mean is None for RMSNorm.  rstd/mean have the
    shape of x without its last dimension."""
    mode = int(mode)
    M, N = _rows(x)
    dev = x.device
    bf, f32 = torch.bfloat16, torch.float32
    _check_tensor(x, "x", bf, x.shape, dev)
    _check_tensor(gamma, "gamma", bf, (N,), dev)
    _check_tensor(beta, "beta", bf, (N,), dev)
    if y is None:
        y = torch.empty_like(x)
    if rstd is None:
        rstd = torch.empty(x.shape[:-1], dtype=f32, device=dev)
    if mode == LAYER and mean is None:
        mean = torch.empty(x.shape[:-1], dtype=f32, device=dev)
    _check_tensor(y, "y", bf, x.shape, dev)
    _check_tensor(rstd, "rstd", f32, x.shape[:-1], dev)
    _check_tensor(mean, "mean", f32, x.shape[:-1], dev)
    st = lib().norm_fwd(_ptr(x), _ptr(gamma), _ptr(beta), M, N, float(eps), mode, _ptr(y),
                        _ptr(rstd), _ptr(mean), _stream(stream, dev))
    if st != 0:
        raise NormError(st, "norm_fwd")
    return y, rstd, mean


def norm_bwd_workspace_bytes(M, N, mode=RMS) -> int:
    out = ctypes.c_size_t(0)
    st = lib().norm_bwd_workspace_bytes(int(M), int(N), int(mode), ctypes.byref(out))
    if st != 0:
        raise NormError(st, "norm_bwd_workspace_bytes")
    return int(out.value)


def norm_bwd(dy, x, gamma, rstd, mean=None, mode=RMS, *, dx=None, dgamma=None, dbeta=None,
             want_dbeta=True, workspace=None, stream=None):
    """Backward pass.  Returns (dx, dgamma, dbeta); dbeta is None for RMSNorm
    (or when want_dbeta is False)."""
    mode = int(mode)
    M, N = _rows(x)
    dev = x.device
    bf, f32 = torch.bfloat16, torch.float32
    _check_tensor(x, "x", bf, x.shape, dev)
    _check_tensor(dy, "dy", bf, x.shape, dev)
    _check_tensor(gamma, "gamma", bf, (N,), dev)
    _check_tensor(rstd, "rstd", f32, x.shape[:-1], dev)
    _check_tensor(mean, "mean", f32, x.shape[:-1], dev)
    if dx is None:
        dx = torch.empty_like(x)
    if dgamma is None:
        dgamma = torch.empty(N, dtype=f32, device=dev)
    if mode == LAYER and want_dbeta and dbeta is None:
        dbeta = torch.empty(N, dtype=f32, device=dev)
    _check_tensor(dx, "dx", bf, x.shape, dev)
    _check_tensor(dgamma, "dgamma", f32, (N,), dev)
    _check_tensor(dbeta, "dbeta", f32, (N,), dev)
    if workspace is None:
        with torch.cuda.device(dev):
            nbytes = norm_bwd_workspace_bytes(M, N, mode)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    st = lib().norm_bwd(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(rstd), _ptr(mean), M, N, mode,
                        _ptr(dx), _ptr(dgamma), _ptr(dbeta), _ptr(workspace),
                        workspace.numel() * workspace.element_size(), _stream(stream, dev))
    if st != 0:
        raise NormError(st, "norm_bwd")
    return dx, dgamma, dbeta


def norm_add_fwd(x, r, gamma, beta=None, eps=1e-5, mode=RMS, *, h=None, y=None, rstd=None,
                 mean=None, stream=None):
    """Fused residual add + norm forward: h = bf16(x + r), y = norm(h).
    Returns (h, y, rstd, mean)."""
    mode = int(mode)
    M, N = _rows(x)
    dev = x.device
    bf, f32 = torch.bfloat16, torch.float32
    _check_tensor(x, "x", bf, x.shape, dev)
    _check_tensor(r, "r", bf, x.shape, dev)
    _check_tensor(gamma, "gamma", bf, (N,), dev)
    _check_tensor(beta, "beta", bf, (N,), dev)
    h = torch.empty_like(x) if h is None else h
    y = torch.empty_like(x) if y is None else y
    if rstd is None:
        rstd = torch.empty(x.shape[:-1], dtype=f32, device=dev)
    if mode == LAYER and mean is None:
        mean = torch.empty(x.shape[:-1], dtype=f32, device=dev)
    for t, n in ((h, "h"), (y, "y")):
        _check_tensor(t, n, bf, x.shape, dev)
    _check_tensor(rstd, "rstd", f32, x.shape[:-1], dev)
    _check_tensor(mean, "mean", f32, x.shape[:-1], dev)
    st = lib().norm_add_fwd(_ptr(x), _ptr(r), _ptr(gamma), _ptr(beta), M, N, float(eps), mode,
                            _ptr(h), _ptr(y), _ptr(rstd), _ptr(mean), _stream(stream, dev))
    if st != 0:
        raise NormError(st, "norm_add_fwd")
    return h, y, rstd, mean


FP8_ROW = 0
FP8_MX = 1


def norm_fwd_fp8(x, gamma, beta=None, eps=1e-5, mode=RMS, scaling=FP8_ROW, *, r=None, h=None,
                 q=None, scale=None, rstd=None, mean=None, stream=None):
    """Forward with E4M3 output (norm_fwd_fp8 in gbnorm.h).  With r given,
    the norm is taken of h = bf16(x + r) (written to h).  Returns
    (q, scale, rstd, mean, h): q uint8 [..., N] E4M3 codes; scale fp32
    [...] (FP8_ROW) or uint8 [..., N // 32] E8M0 exponents (FP8_MX)."""
    mode = int(mode)
    scaling = int(scaling)
    M, N = _rows(x)
    dev = x.device
    bf, f32, u8 = torch.bfloat16, torch.float32, torch.uint8
    lead = x.shape[:-1]
    _check_tensor(x, "x", bf, x.shape, dev)
    _check_tensor(r, "r", bf, x.shape, dev)
    _check_tensor(gamma, "gamma", bf, (N,), dev)
    _check_tensor(beta, "beta", bf, (N,), dev)
    if r is not None and h is None:
        h = torch.empty_like(x)
    if q is None:
        q = torch.empty(x.shape, dtype=u8, device=dev)
    sshape = lead if scaling == FP8_ROW else (*lead, N // 32)
    sdtype = f32 if scaling == FP8_ROW else u8
    if scale is None:
        scale = torch.empty(sshape, dtype=sdtype, device=dev)
    if rstd is None:
        rstd = torch.empty(lead, dtype=f32, device=dev)
    if mode == LAYER and mean is None:
        mean = torch.empty(lead, dtype=f32, device=dev)
    _check_tensor(h, "h", bf, x.shape, dev)
    _check_tensor(q, "q", u8, x.shape, dev)
    _check_tensor(scale, "scale", sdtype, sshape, dev)
    _check_tensor(rstd, "rstd", f32, lead, dev)
    _check_tensor(mean, "mean", f32, lead, dev)
    st = lib().norm_fwd_fp8(_ptr(x), _ptr(r), _ptr(gamma), _ptr(beta), M, N, float(eps), mode,
                            scaling, _ptr(h), _ptr(q), _ptr(scale), _ptr(rstd), _ptr(mean),
                            _stream(stream, dev))
    if st != 0:
        raise NormError(st, "norm_fwd_fp8")
    return q, scale, rstd, mean, h


def norm_tune_fwd(x, gamma, beta=None, eps=1e-5, mode=RMS, *, iters=20, stream=None):
    """Measure the forward plans of this shape on these buffers and keep the
    fastest (norm_tune_fwd in gbnorm.h).  Returns the chosen plan (dict)."""
    mode = int(mode)
    M, N = _rows(x)
    dev = x.device
    _check_tensor(x, "x", torch.bfloat16, x.shape, dev)
    _check_tensor(gamma, "gamma", torch.bfloat16, (N,), dev)
    _check_tensor(beta, "beta", torch.bfloat16, (N,), dev)
    y = torch.empty_like(x)
    rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=dev)
    mean = torch.empty_like(rstd) if mode == LAYER else None
    out = Plan()
    st = lib().norm_tune_fwd(_ptr(x), _ptr(gamma), _ptr(beta), M, N, float(eps), mode, _ptr(y),
                             _ptr(rstd), _ptr(mean), int(iters), ctypes.byref(out),
                             _stream(stream, dev))
    if st != 0:
        raise NormError(st, "norm_tune_fwd")
    return out.as_dict()


def norm_tune_bwd(dy, x, gamma, rstd, mean=None, mode=RMS, *, iters=20, stream=None):
    """Measure the backward plans of this shape on these buffers and keep the
    fastest (norm_tune_bwd in gbnorm.h).  Returns the chosen plan (dict)."""
    mode = int(mode)
    M, N = _rows(x)
    dev = x.device
    for t, n in ((x, "x"), (dy, "dy")):
        _check_tensor(t, n, torch.bfloat16, x.shape, dev)
    _check_tensor(gamma, "gamma", torch.bfloat16, (N,), dev)
    _check_tensor(rstd, "rstd", torch.float32, x.shape[:-1], dev)
    _check_tensor(mean, "mean", torch.float32, x.shape[:-1], dev)
    dx = torch.empty_like(x)
    dg = torch.empty(N, dtype=torch.float32, device=dev)
    db = torch.empty(N, dtype=torch.float32, device=dev) if mode == LAYER else None
    ws = torch.empty(max(norm_bwd_workspace_bytes(M, N, mode), 16), dtype=torch.uint8,
                     device=dev)
    out = Plan()
    st = lib().norm_tune_bwd(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(rstd), _ptr(mean), M, N, mode,
                             _ptr(dx), _ptr(dg), _ptr(db), _ptr(ws), ws.numel(), int(iters),
                             ctypes.byref(out), _stream(stream, dev))
    if st != 0:
        raise NormError(st, "norm_tune_bwd")
    return out.as_dict()


def norm_tune_reset():
    """Drop every cached plan (tuned or default)."""
    st = lib().norm_tune_reset()
    if st != 0:
        raise NormError(st, "norm_tune_reset")


def norm_host_workspace_bytes(M, N, mode=RMS, chunk_rows=0) -> int:
    out = ctypes.c_size_t(0)
    st = lib().norm_host_workspace_bytes(int(M), int(N), int(mode), int(chunk_rows),
                                         ctypes.byref(out))
    if st != 0:
        raise NormError(st, "norm_host_workspace_bytes")
    return int(out.value)


def _check_host(t, name, dtype, shape):
    if t is None:
        return
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if t.dtype != dtype or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected contiguous {dtype} {tuple(shape)}")


def norm_fwd_bwd_host(x, dy, gamma, beta=None, eps=1e-5, mode=RMS, *, chunk_rows=0, out=None,
                      workspace=None, stream=None, device=None):
    """Forward + backward on host tensors (norm_fwd_bwd_host in gbnorm.h).
    x, dy, gamma, beta are CPU tensors (pinned for overlap); returns CPU
    tensors (y, rstd, mean, dx, dgamma, dbeta), complete once `stream`
    (default: the current stream of `device`) is synchronised.  `out` may
    pass preallocated (pinned) outputs in that order, `workspace` a device
    uint8 tensor of norm_host_workspace_bytes bytes."""
    mode = int(mode)
    M, N = _rows(x)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    bf, f32 = torch.bfloat16, torch.float32
    lead = x.shape[:-1]
    _check_host(x, "x", bf, x.shape)
    _check_host(dy, "dy", bf, x.shape)
    _check_host(gamma, "gamma", bf, (N,))
    _check_host(beta, "beta", bf, (N,))
    if out is None:
        pin = x.is_pinned()
        out = (torch.empty(x.shape, dtype=bf, pin_memory=pin),
               torch.empty(lead, dtype=f32, pin_memory=pin),
               torch.empty(lead, dtype=f32, pin_memory=pin) if mode == LAYER else None,
               torch.empty(x.shape, dtype=bf, pin_memory=pin),
               torch.empty(N, dtype=f32, pin_memory=pin),
               torch.empty(N, dtype=f32, pin_memory=pin) if mode == LAYER else None)
    y, rstd, mean, dx, dg, db = out
    for t, n, dt, sh in ((y, "y", bf, x.shape), (rstd, "rstd", f32, lead), (mean, "mean", f32, lead),
                         (dx, "dx", bf, x.shape), (dg, "dgamma", f32, (N,)), (db, "dbeta", f32, (N,))):
        _check_host(t, n, dt, sh)
    nbytes = norm_host_workspace_bytes(M, N, mode, chunk_rows)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    _check_tensor(workspace, "workspace", torch.uint8, (workspace.numel(),), dev)
    st = lib().norm_fwd_bwd_host(_ptr(x), _ptr(dy), _ptr(gamma), _ptr(beta), M, N, float(eps),
                                 mode, _ptr(y), _ptr(dx), _ptr(rstd), _ptr(mean), _ptr(dg),
                                 _ptr(db), int(chunk_rows), _ptr(workspace),
                                 workspace.numel(), _stream(stream, dev))
    if st != 0:
        raise NormError(st, "norm_fwd_bwd_host")
    return y, rstd, mean, dx, dg, db


def norm_add_bwd_workspace_bytes(M, N, mode=RMS) -> int:
    out = ctypes.c_size_t(0)
    st = lib().norm_add_bwd_workspace_bytes(int(M), int(N), int(mode), ctypes.byref(out))
    if st != 0:
        raise NormError(st, "norm_add_bwd_workspace_bytes")
    return int(out.value)


def norm_add_bwd(dy, dh, h, gamma, rstd, mean=None, mode=RMS, *, dx=None, dgamma=None,
                 dbeta=None, want_dbeta=True, workspace=None, stream=None):
    """Fused residual add + norm backward: dx = norm backward at h + dh (the
    gradient of both x and r).  Returns (dx, dgamma, dbeta)."""
    mode = int(mode)
    M, N = _rows(h)
    dev = h.device
    bf, f32 = torch.bfloat16, torch.float32
    for t, n in ((dy, "dy"), (dh, "dh"), (h, "h")):
        _check_tensor(t, n, bf, h.shape, dev)
    _check_tensor(gamma, "gamma", bf, (N,), dev)
    _check_tensor(rstd, "rstd", f32, h.shape[:-1], dev)
    _check_tensor(mean, "mean", f32, h.shape[:-1], dev)
    dx = torch.empty_like(h) if dx is None else dx
    dgamma = torch.empty(N, dtype=f32, device=dev) if dgamma is None else dgamma
    if mode == LAYER and want_dbeta and dbeta is None:
        dbeta = torch.empty(N, dtype=f32, device=dev)
    _check_tensor(dx, "dx", bf, h.shape, dev)
    _check_tensor(dgamma, "dgamma", f32, (N,), dev)
    _check_tensor(dbeta, "dbeta", f32, (N,), dev)
    if workspace is None:
        with torch.cuda.device(dev):
            nbytes = norm_add_bwd_workspace_bytes(M, N, mode)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    st = lib().norm_add_bwd(_ptr(dy), _ptr(dh), _ptr(h), _ptr(gamma), _ptr(rstd), _ptr(mean), M,
                            N, mode, _ptr(dx), _ptr(dgamma), _ptr(dbeta), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream, dev))
    if st != 0:
        raise NormError(st, "norm_add_bwd")
    return dx, dgamma, dbeta


def norm_gemm_prepare(w, gamma, beta=None, mode=RMS, *, wg=None, u=None, v=None,
                      stream=None):
    """Weights of the normalisation-GEMM: W' = bf16(W * gamma) (gamma scales
    the columns of W [Nout, K]), u = row sums of W' and v = W beta (fp32).
    Returns (wg, u, v); u and v are None for RMSNorm unless given."""
    mode = int(mode)
    if w.dim() != 2:
        raise ValueError("w must be [Nout, K]")
    Nout, K = w.shape
    dev = w.device
    bf, f32 = torch.bfloat16, torch.float32
    _check_tensor(w, "w", bf, (Nout, K), dev)
    _check_tensor(gamma, "gamma", bf, (K,), dev)
    _check_tensor(beta, "beta", bf, (K,), dev)
    if wg is None:
        wg = torch.empty_like(w)
    if mode == LAYER:
        if u is None:
            u = torch.empty(Nout, dtype=f32, device=dev)
        if v is None:
            v = torch.empty(Nout, dtype=f32, device=dev)
    _check_tensor(wg, "wg", bf, (Nout, K), dev)
    _check_tensor(u, "u", f32, (Nout,), dev)
    _check_tensor(v, "v", f32, (Nout,), dev)
    st = lib().norm_gemm_prepare(_ptr(w), _ptr(gamma), _ptr(beta), K, Nout, mode, _ptr(wg),
                                 _ptr(u), _ptr(v), _stream(stream, dev))
    if st != 0:
        raise NormError(st, "norm_gemm_prepare")
    return wg, u, v


def norm_gemm_fwd(x, wg, u=None, v=None, eps=1e-5, mode=RMS, *, out=None, rstd=None,
                  mean=None, stream=None):
    """out = norm(x) W^T through the fused tensor-core GEMM, with (wg, u, v)
    from norm_gemm_prepare.  x is [..., K]; returns (out [..., Nout], rstd,
    mean), mean None for RMSNorm."""
    mode = int(mode)
    M, K = _rows(x)
    if wg.dim() != 2 or wg.shape[1] != K:
        raise ValueError("wg must be [Nout, K]")
    Nout = wg.shape[0]
    dev = x.device
    bf, f32 = torch.bfloat16, torch.float32
    _check_tensor(x, "x", bf, x.shape, dev)
    _check_tensor(wg, "wg", bf, (Nout, K), dev)
    _check_tensor(u, "u", f32, (Nout,), dev)
    _check_tensor(v, "v", f32, (Nout,), dev)
    oshape = tuple(x.shape[:-1]) + (Nout,)
    if out is None:
        out = torch.empty(oshape, dtype=bf, device=dev)
    if rstd is None:
        rstd = torch.empty(x.shape[:-1], dtype=f32, device=dev)
    if mode == LAYER and mean is None:
        mean = torch.empty(x.shape[:-1], dtype=f32, device=dev)
    _check_tensor(out, "out", bf, oshape, dev)
    _check_tensor(rstd, "rstd", f32, x.shape[:-1], dev)
    _check_tensor(mean, "mean", f32, x.shape[:-1], dev)
    st = lib().norm_gemm_fwd(_ptr(x), _ptr(wg), _ptr(u), _ptr(v), M, K, Nout, float(eps), mode,
                             _ptr(out), _ptr(rstd), _ptr(mean), _stream(stream, dev))
    if st != 0:
        raise NormError(st, "norm_gemm_fwd")
    return out, rstd, mean


def norm_plan(M, N, mode=RMS, backward=False, sm_count=0, smem_optin=0, residual=False,
              fp8=False, other_pass=False) -> dict:
    """Launch plan of one pass (see norm_plan in gbnorm.h).  sm_count > 0
    plans for a hypothetical device without touching CUDA; residual=True
    plans the fused residual add variant, fp8=True the E4M3-output forward;
    other_pass=True gives, for rows on the two-pass path, the forward's
    output pass or the backward's dot-product pass."""
    out = Plan()
    which = ((1 if backward else 0) | (2 if residual else 0) | (4 if fp8 else 0)
             | (8 if other_pass else 0))
    st = lib().norm_plan(int(M), int(N), int(mode), which, int(sm_count), int(smem_optin),
                         ctypes.byref(out))
    if st != 0:
        raise NormError(st, "norm_plan")
    return out.as_dict()


def norm_get_device_error(stream=None, device=None):
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    return lib().norm_get_device_error(_stream(stream, dev))
