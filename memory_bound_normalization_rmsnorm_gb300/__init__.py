"""GB300 (sm_103a) RMSNorm / LayerNorm forward and backward, and the
normalisation fused into a tensor-core GEMM.

The computation runs in hand-written CUDA kernels behind the C ABI of
include/gbnorm.h (libgbnorm.so); this package is its thin Python binding plus
the seeded synthetic workloads used by the tests and the benchmark.
"""
from ._binding import (FP8_MX, FP8_ROW, LAYER, RMS, NormError, declared_functions, lib,
                       library_path, norm_add_bwd, norm_add_bwd_workspace_bytes, norm_add_fwd,
                       norm_bwd, norm_bwd_workspace_bytes, norm_fwd, norm_fwd_bwd_host,
                       norm_fwd_fp8, norm_gemm_fwd, norm_gemm_prepare, norm_get_device_error,
                       norm_host_workspace_bytes, norm_plan, norm_tune_bwd, norm_tune_fwd, norm_tune_reset, strerror)
from .builder import build

__all__ = [
    "RMS", "LAYER", "NormError", "norm_fwd", "norm_bwd", "norm_bwd_workspace_bytes",
    "norm_get_device_error", "norm_plan", "norm_add_fwd", "norm_add_bwd",
    "norm_add_bwd_workspace_bytes", "norm_fwd_fp8", "FP8_ROW", "FP8_MX",
    "norm_fwd_bwd_host", "norm_host_workspace_bytes", "norm_tune_fwd", "norm_tune_bwd",
    "norm_tune_reset", "norm_gemm_prepare", "norm_gemm_fwd", "strerror", "lib", "library_path", "declared_functions", "build",
]
