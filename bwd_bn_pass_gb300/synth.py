"""Seeded synthetic inputs for the normalization workloads.

This module only draws random numbers with a CPU ``torch.Generator`` and
rounds them to the storage dtype.  It holds none of the normalization
arithmetic: the saved LayerNorm / RMSNorm statistics that a backward needs
are computed by whoever consumes these tensors.  Both the test suite and
``bench.py`` use it, so the CUDA path and the float64 oracle always see the
same stored values.

Workloads (the pages' shapes and value distributions):

* BatchNorm2d training, NCHW.  ``x = mu_c + sigma_c * N(0, 1)`` per channel,
  gamma ~ U(0.5, 1.5), beta ~ N(0, 0.1), dy ~ N(0, 1), running_mean = 0,
  running_var = 1, eps = 1e-5, momentum = 0.1.  gamma/beta/running stats are
  fp32; x/dy take the workload dtype.
* RMSNorm backward [R, H]: x, dy ~ N(0, 1), weight ~ U(0.5, 1.5), eps = 1e-5.
* LayerNorm backward fused with bias+dropout+add [R, H]: input, residual,
  bias, dy ~ N(0, 1); keep-mask ~ Bernoulli(0.9); dropout scale fl32(1/0.9);
  gamma ~ U(0.5, 1.5); beta ~ N(0, 0.1) (unused by the backward); eps = 1e-5.
"""

from dataclasses import dataclass
from typing import Optional, Tuple

import torch

SEED_BASE = 20241202

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class BNCase:
    name: str
    shape: Tuple[int, ...]
    dtype: str
    mu_range: Optional[Tuple[float, float]] = None
    sigma_range: Optional[Tuple[float, float]] = None
    eps: float = 1e-5
    momentum: float = 0.1
    seed: int = SEED_BASE


@dataclass(frozen=True)
class RMSCase:
    name: str
    rows: int
    hidden: int
    dtype: str
    eps: float = 1e-5
    seed: int = SEED_BASE + 2


@dataclass(frozen=True)
class LNCase:
    name: str
    rows: int
    hidden: int
    dtype: str
    fused: bool = True
    keep_prob: float = 0.9
    eps: float = 1e-5
    with_dz_extra: bool = False
    seed: int = SEED_BASE + 3


CASES = {
    c.name: c
    for c in [
        BNCase("bn_tiny_f32", (8, 4, 8, 8), "f32", seed=SEED_BASE + 0),
        BNCase("bn_offset_f32", (256, 32, 32, 32), "f32",
               mu_range=(-1000.0, 1000.0), seed=SEED_BASE + 1),
        BNCase("bn_ragged_f32", (3, 37, 41, 40), "f32",
               mu_range=(-1000.0, 1000.0), seed=SEED_BASE + 1),
        RMSCase("rms_bf16", 2048, 8192, "bf16"),
        RMSCase("rms_f32", 2048, 8192, "f32"),
        LNCase("ln_fused_bf16", 16 * 512, 1600, "bf16"),
        BNCase("bn_offset_bf16", (128, 256, 56, 56), "bf16",
               mu_range=(-100.0, 100.0), sigma_range=(0.01, 10.0),
               seed=SEED_BASE + 4),
    ]
}


def _uniform(g, n, lo, hi, dtype=torch.float32):
    return lo + (hi - lo) * torch.rand(n, generator=g, dtype=dtype)


def bn_inputs(case: BNCase):
    """Return dict of CPU tensors: x, dy (case dtype), gamma, beta,
    running_mean, running_var (fp32 [C]), plus eps and momentum."""
    g = torch.Generator().manual_seed(case.seed)
    C = case.shape[1]
    view = (1, C) + (1,) * (len(case.shape) - 2)
    mu = (torch.zeros(C) if case.mu_range is None
          else _uniform(g, C, *case.mu_range))
    sigma = (torch.ones(C) if case.sigma_range is None
             else _uniform(g, C, *case.sigma_range))
    noise = torch.randn(case.shape, generator=g, dtype=torch.float32)
    x = (mu.view(view) + sigma.view(view) * noise).to(DTYPES[case.dtype])
    del noise
    gamma = _uniform(g, C, 0.5, 1.5)
    beta = 0.1 * torch.randn(C, generator=g)
    dy = torch.randn(case.shape, generator=g,
                     dtype=torch.float32).to(DTYPES[case.dtype])
    return {
        "x": x.contiguous(), "dy": dy.contiguous(),
        "gamma": gamma, "beta": beta,
        "running_mean": torch.zeros(C), "running_var": torch.ones(C),
        "eps": case.eps, "momentum": case.momentum,
    }


def rms_inputs(case: RMSCase):
    """Return dict of CPU tensors x, dy [R, H] and w [H] (case dtype)."""
    g = torch.Generator().manual_seed(case.seed)
    dt = DTYPES[case.dtype]
    x = torch.randn(case.rows, case.hidden, generator=g).to(dt)
    dy = torch.randn(case.rows, case.hidden, generator=g).to(dt)
    w = _uniform(g, case.hidden, 0.5, 1.5).to(dt)
    return {"x": x, "dy": dy, "w": w, "eps": case.eps}


def ln_inputs(case: LNCase):
    """Return dict of CPU tensors for the (fused) LayerNorm backward.

    Keys: inp, residual, dy [R, H] and bias, gamma, beta [H] in the case
    dtype; mask uint8 [R, H] (1 = kept); dropout_scale (a Python float that
    is exactly representable in fp32); dz_extra fp32 [R, H] or None; eps.
    For an unfused case residual/bias/mask are None and inp is the LayerNorm
    input itself.
    """
    g = torch.Generator().manual_seed(case.seed)
    dt = DTYPES[case.dtype]
    R, H = case.rows, case.hidden
    inp = torch.randn(R, H, generator=g).to(dt)
    residual = torch.randn(R, H, generator=g).to(dt)
    bias = torch.randn(H, generator=g).to(dt)
    mask = (torch.rand(R, H, generator=g) < case.keep_prob).to(torch.uint8)
    gamma = _uniform(g, H, 0.5, 1.5).to(dt)
    beta = (0.1 * torch.randn(H, generator=g)).to(dt)
    dy = torch.randn(R, H, generator=g).to(dt)
    dz_extra = (torch.randn(R, H, generator=g) if case.with_dz_extra
                else None)
    scale = float(torch.tensor(1.0 / case.keep_prob, dtype=torch.float32))
    if not case.fused:
        residual = bias = mask = None
        scale = 1.0
    return {
        "inp": inp, "residual": residual, "bias": bias, "mask": mask,
        "gamma": gamma, "beta": beta, "dy": dy, "dz_extra": dz_extra,
        "dropout_scale": scale, "eps": case.eps,
    }
