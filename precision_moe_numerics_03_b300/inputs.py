"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds none of the method's arithmetic: it only draws random numbers and rounds them
to bf16 storage (torch's own nearest-even cast).  Both the CUDA path and the oracle read the same
bytes that it produces.

Recipe (the pages publish no data; the shapes follow the Inkling 2 Small model card: 384
experts, top-8 routing, d_model 4096, SwiGLU expert width 2048):
  * host generator: numpy PCG64 seeded with 1000 + workload number;
  * device generator (for tensors too large to draw on the host): torch's CUDA generator seeded
    with the same number; every element is a pure function of the seed;
  * activations N(0, 1), optionally with Student-t(nu=3) tails rescaled to unit standard
    deviation (t3 / sqrt(3)), optionally with 1% of entries multiplied by 20 (outliers);
  * expert weights N(0, 0.02);
  * router logits N(0, 1) plus a per-expert bias N(0, 1) (skewed load) where the workload says so;
  * upstream gradients N(0, 1).
"""
from __future__ import annotations

import math

import numpy as np
import torch


def seed_of(workload: int) -> int:
    return 1000 + int(workload)


def host_rng(workload: int, stream: int = 0) -> np.random.Generator:
    """numpy PCG64 generator of a workload; `stream` separates tensors of one workload."""
    return np.random.Generator(np.random.PCG64([seed_of(workload), stream]))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """binary32 -> bf16 bit patterns (uint16) with torch's nearest-even cast."""
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def host_normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def host_student_t(rng: np.random.Generator, shape, nu: float = 3.0) -> np.ndarray:
    """Student-t(nu) rescaled to unit standard deviation."""
    t = rng.standard_t(nu, size=shape)
    return (t / math.sqrt(nu / (nu - 2.0))).astype(np.float32)


def host_outliers(rng: np.random.Generator, x: np.ndarray, frac: float = 0.01,
                  factor: float = 20.0) -> np.ndarray:
    mask = rng.random(x.shape) < frac
    return np.where(mask, x * np.float32(factor), x).astype(np.float32)


# ---------------------------------------------------------------------------------------------
# Device-side draws (large workloads).  torch's generator on the given device; deterministic.
# ---------------------------------------------------------------------------------------------
def device_generator(workload: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed_of(workload) * 1000 + int(stream))
    return g


def device_normal(shape, std: float, gen: torch.Generator, device, dtype=torch.bfloat16):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def device_student_t(shape, gen: torch.Generator, device, nu: int = 3, dtype=torch.bfloat16):
    """Student-t with integer nu: Z / sqrt(chi2_nu / nu), chi2_nu a sum of nu squared normals;
    rescaled to unit standard deviation.  Drawn in slices to bound temporary memory."""
    out = torch.empty(shape, device=device, dtype=dtype)
    flat = out.view(-1)
    n = flat.numel()
    step = 1 << 26
    scale = 1.0 / math.sqrt(nu / (nu - 2.0))
    for s in range(0, n, step):
        m = min(step, n - s)
        z = torch.randn(m, generator=gen, device=device)
        chi = torch.zeros(m, device=device)
        for _ in range(nu):
            w = torch.randn(m, generator=gen, device=device)
            chi.addcmul_(w, w)
        z.mul_(torch.rsqrt(chi.div_(nu))).mul_(scale)
        flat[s:s + m] = z.to(dtype)
    return out
