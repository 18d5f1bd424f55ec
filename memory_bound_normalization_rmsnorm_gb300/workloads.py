"""Seeded synthetic inputs for the normalisation workloads.

This module only draws random tensors; it holds none of the normalisation
arithmetic, so both the CUDA path's callers and the fp64 oracle's callers can
use it without sharing any of the method.

The workloads are the five shape families the benchmark and the parity tests
run.  The 16,384-token sequence length (M = 2 x 16384) comes from the page
"Extraindo 2x de MFU dos nossos treinamentos" (building.nu.com), section
"Introducao".  Distribution notation N(a, s) is read as mean a and standard
deviation s.  Every tensor is drawn in fp32 from ONE generator seeded with
`seed`, in the fixed order x, (outlier mask or channel offset), gamma, beta,
dy, and then rounded to bf16 once; the same bf16 bits feed the GPU and the
oracle.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

RMS = 0
LAYER = 1


@dataclass(frozen=True)
class Workload:
    name: str
    mode: int  # RMS or LAYER
    M: int
    N: int
    eps: float
    x_dist: str  # "normal" | "normal_outliers" | "normal2" | "normal_offset"
    gamma_dist: str  # "one_plus_0.1n" | "uniform_0.5_1.5"
    dy_scale: float = 1.0
    seed: int = 0
    tags: tuple = field(default=())

    @property
    def mode_name(self) -> str:
        return "rms" if self.mode == RMS else "layer"


def _family():
    w = []
    # Small RMSNorm case (fits the oracle in well under a second).
    w.append(Workload("rms_256x1024", RMS, 256, 1024, 1e-6, "normal", "one_plus_0.1n"))
    # LayerNorm at a transformer width: the headline workload.
    w.append(Workload("layer_32768x4096", LAYER, 32768, 4096, 1e-5, "normal",
                      "one_plus_0.1n"))
    # Small-row sweep with 0.5% x50 outliers.
    for n in (256, 512, 768, 1024):
        w.append(Workload(f"rms_262144x{n}_outliers", RMS, 262144, n, 1e-6,
                          "normal_outliers", "one_plus_0.1n"))
    # Very long rows.
    for n in (16384, 32768, 65536, 131072):
        w.append(Workload(f"rms_4096x{n}", RMS, 4096, n, 1e-6, "normal2",
                          "uniform_0.5_1.5"))
    # Transformer-block shapes, batch 2 x 16384 tokens, residual-stream-like x.
    for mode in (RMS, LAYER):
        for n in (2048, 3072, 5120, 8192):
            tag = "rms" if mode == RMS else "layer"
            w.append(Workload(f"{tag}_32768x{n}_resid", mode, 32768, n, 1e-5,
                              "normal_offset", "one_plus_0.1n", dy_scale=1e-2))
    return {x.name: x for x in w}


WORKLOADS = _family()
HEADLINE = "layer_32768x4096"


def _wide():
    """Rows wider than one thread-block cluster holds in shared memory
    (streamed row slices or the two-pass path): the very-long-row family
    carried past 262144 columns, RMSNorm with its distributions and
    LayerNorm with the headline's."""
    w = [Workload("rms_4096x524288", RMS, 4096, 524288, 1e-6, "normal2", "uniform_0.5_1.5"),
         Workload("rms_1024x1048576", RMS, 1024, 1048576, 1e-6, "normal2", "uniform_0.5_1.5"),
         Workload("layer_2048x524288", LAYER, 2048, 524288, 1e-5, "normal", "one_plus_0.1n")]
    return {x.name: x for x in w}


WIDE = _wide()
ALL = {**WORKLOADS, **WIDE}


def like(w: Workload, M: int, N: int) -> Workload:
    """Same distributions as `w` at another shape (for small parity cases)."""
    return Workload(f"{w.name}@{M}x{N}", w.mode, M, N, w.eps, w.x_dist, w.gamma_dist,
                    w.dy_scale, w.seed)


def make_inputs(w: Workload, device="cpu", seed=None, with_dy=True):
    """Draw (x, gamma, beta, dy) as bf16 tensors on `device`.

    beta is None for RMSNorm.  All draws use one torch.Generator on `device`
    seeded with `seed` (default: the workload's), in the order x, mask or
    offset, gamma, beta, dy.  A CPU generator and a CUDA generator give
    different (but each reproducible) bits.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed if seed is None else seed)
    M, N = w.M, w.N
    f32 = dict(dtype=torch.float32, device=dev, generator=g)

    x = torch.randn(M, N, **f32)
    if w.x_dist == "normal_outliers":
        # Bernoulli(0.005) mask; selected entries are scaled by 50.
        mask = torch.rand(M, N, **f32) < 0.005
        x = torch.where(mask, x * 50.0, x)
        del mask
    elif w.x_dist == "normal2":
        x.mul_(2.0)
    elif w.x_dist == "normal_offset":
        offset = torch.randn(N, **f32) * 0.5
        x.add_(offset)
    elif w.x_dist != "normal":
        raise ValueError(w.x_dist)
    x = x.to(torch.bfloat16)

    if w.gamma_dist == "one_plus_0.1n":
        gamma = 1.0 + 0.1 * torch.randn(N, **f32)
    elif w.gamma_dist == "uniform_0.5_1.5":
        gamma = 0.5 + torch.rand(N, **f32)
    else:
        raise ValueError(w.gamma_dist)
    gamma = gamma.to(torch.bfloat16)

    beta = None
    if w.mode == LAYER:
        beta = (0.1 * torch.randn(N, **f32)).to(torch.bfloat16)

    dy = None
    if with_dy:
        dy = torch.randn(M, N, **f32)
        if w.dy_scale != 1.0:
            dy.mul_(w.dy_scale)
        dy = dy.to(torch.bfloat16)
    return x, gamma, beta, dy


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a bf16 tensor's bit patterns (copies to host)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def make_residual_inputs(w: Workload, device="cpu", seed=None):
    """Inputs of the fused residual add + norm: (x, r, gamma, beta, dy, dh).

    x, gamma, beta and dy as make_inputs; then, from a second generator
    seeded with seed + 1, the residual r ~ N(0, 1) (the update added to the
    residual stream) and the residual-path gradient dh drawn like dy.
    """
    x, gamma, beta, dy = make_inputs(w, device, seed=seed)
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed((w.seed if seed is None else seed) + 1)
    f32 = dict(dtype=torch.float32, device=dev, generator=g)
    r = torch.randn(w.M, w.N, **f32).to(torch.bfloat16)
    dh = torch.randn(w.M, w.N, **f32)
    if w.dy_scale != 1.0:
        dh.mul_(w.dy_scale)
    dh = dh.to(torch.bfloat16)
    return x, r, gamma, beta, dy, dh


def make_gemm_weight(w: Workload, Nout: int, device="cpu", seed=None):
    """Weight [Nout, K = w.N] of the linear layer that consumes the
    normalised rows: N(0, 1/K) entries (the usual fan-in scaled
    initialisation), drawn in fp32 from a generator seeded with seed + 2 and
    rounded to bf16."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed((w.seed if seed is None else seed) + 2)
    wt = torch.randn(Nout, w.N, dtype=torch.float32, device=dev, generator=g)
    return (wt * (1.0 / w.N ** 0.5)).to(torch.bfloat16)
