"""The E4M3 comparison rule (tests/fp8_check.py) on the CPU: it accepts a
binary32 computation of the forward followed by round-to-nearest-even E4M3
conversion (done here with numpy float32 and torch's float8_e4m3fn), keeps
the share of non-unique codes small, and rejects truncated codes, a wrong
MX exponent and a wrong row scale."""
import numpy as np
import pytest
import torch

from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

import fp8_check
import oracle


def _f32_forward(x, g, b, eps, mode):
    xf, gf = x.float().numpy(), g.float().numpy()
    e = np.float32(eps)
    if mode == 1:
        mu = xf.mean(axis=1, dtype=np.float32, keepdims=True)
        var = ((xf - mu) ** 2).mean(axis=1, dtype=np.float32, keepdims=True)
    else:
        mu = np.float32(0)
        var = (xf * xf).mean(axis=1, dtype=np.float32, keepdims=True)
    rs = (np.float32(1) / np.sqrt(var + e)).astype(np.float32)
    y = (xf - mu) * rs * gf
    if b is not None:
        y = y + b.float().numpy()
    return y.astype(np.float32)


def _e4m3(v32):
    v = torch.from_numpy(np.clip(v32, -448, 448).astype(np.float32))
    return v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("mode,N", [(0, 64), (0, 1024), (1, 256), (1, 4096)])
def test_rule_on_binary32_forward(mode, N):
    base = wl.WORKLOADS["layer_32768x4096" if mode else "rms_262144x1024_outliers"]
    case = wl.like(base, 96, N)
    x, g, b, _ = wl.make_inputs(case, "cpu", with_dy=False)
    y = _f32_forward(x, g, b, case.eps, mode)
    bb = None if b is None else wl.bf16_bits(b)
    eps = float(np.float32(case.eps))
    # per row
    ref = oracle.fwd_fp8_bf16(wl.bf16_bits(x), None, wl.bf16_bits(g), bb, eps, mode,
                              oracle.FP8_ROW)
    am = np.abs(y).max(axis=1)
    inv = (np.float32(448) / am).astype(np.float32)
    q = _e4m3((y * inv[:, None]).astype(np.float32))
    s = (am / np.float32(448)).astype(np.float32)
    assert fp8_check.check_fp8(q, s, ref, oracle.FP8_ROW, mode) < 0.01
    v = (y * inv[:, None]).astype(np.float64)
    with pytest.raises(AssertionError):
        fp8_check.check_fp8(_e4m3(np.trunc(v * 8) / 8), s, ref, oracle.FP8_ROW, mode)
    with pytest.raises(AssertionError):
        fp8_check.check_fp8(q, s * np.float32(1.001), ref, oracle.FP8_ROW, mode)
    # MX blocks
    ref = oracle.fwd_fp8_bf16(wl.bf16_bits(x), None, wl.bf16_bits(g), bb, eps, mode,
                              oracle.FP8_MX)
    yb = y.reshape(96, -1, 32)
    amb = np.abs(yb).max(axis=2)
    ebits = (amb.view(np.uint32) >> 23) & 0xFF
    e = np.where(ebits == 0, -127, np.maximum(ebits.astype(np.int64) - 135, -127))
    qm = _e4m3((yb * np.exp2(-e)[:, :, None].astype(np.float32)).reshape(96, N))
    eb = (e + 127).astype(np.uint8)
    assert fp8_check.check_fp8(qm, eb, ref, oracle.FP8_MX, mode) < 0.01
    with pytest.raises(AssertionError):
        fp8_check.check_fp8(qm, (eb + 1).astype(np.uint8), ref, oracle.FP8_MX, mode)
