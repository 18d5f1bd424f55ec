"""Host-side pieces of the normalisation-GEMM row, without a GPU: the seeded
weight generator follows its stated recipe, and the benchmark's CPU
baseline times the oracle on a bounded sample."""
import numpy as np
import torch

from memory_bound_normalization_rmsnorm_gb300 import workloads as wl

import bench


def test_gemm_weight_recipe():
    """W [Nout, K] ~ N(0, 1/K) in bf16, reproducible for a seed, from its own
    generator (seed + 2): independent of the x / gamma / beta draws."""
    w0 = wl.Workload("g", wl.LAYER, 8, 1024, 1e-5, "normal", "one_plus_0.1n")
    a = wl.make_gemm_weight(w0, 512)
    b = wl.make_gemm_weight(w0, 512)
    c = wl.make_gemm_weight(w0, 512, seed=7)
    assert a.shape == (512, 1024) and a.dtype == torch.bfloat16
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a.view(torch.int16), c.view(torch.int16))
    std = a.float().std().item()
    assert abs(std * 1024 ** 0.5 - 1.0) < 0.01
    assert abs(a.float().mean().item()) < 5e-4
    # drawing the activations does not move the weights
    wl.make_inputs(w0, with_dy=False)
    assert torch.equal(wl.make_gemm_weight(w0, 512).view(torch.int16), a.view(torch.int16))


def test_gemm_cpu_baseline_sample():
    w0 = wl.Workload("norm_gemm_layer_64x256x128", wl.LAYER, 64, 256, 1e-5, "normal_offset",
                     "one_plus_0.1n")
    cb = bench.gemm_cpu_baseline(w0, 128, seconds=0.2)
    assert cb["kind"] == "oracle" and cb["unit"] == "TFLOP/s" and cb["cores"] == 1
    assert np.isfinite(cb["value"]) and cb["value"] > 0
    assert "rows" in cb["sample"] and "K=256" in cb["sample"]
