"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers and rounds them to bf16 with torch; it
holds none of the quantiser's or the matmul's arithmetic, so the oracle and
the CUDA path can both be fed from it without sharing any method code.

The workloads it imitates are the ones the source pages measure on (Llama-3
projection shapes, activations with outliers, a scaled FP8 KV cache); the
pages' own datasets and checkpoints are not available, so these seeded
tensors stand in for them:

* activations: N(0, 1) with a Bernoulli(rate) fraction of elements scaled by
  ``outlier_mult`` (default 1 % x 20);
* weights: N(0, std) with ``std = 0.02``;
* "heavy-tailed" activations: N(0, 1) with one column in ``every`` drawn from
  Student-t(nu = 4) instead, built as Z / sqrt(chi2_4 / 4) with
  chi2_4 = -2 ln(U1 U2);
* KV cache: N(0, 1) with rare spikes (rate 1e-4) scaled by 50.

All tensors are drawn in fp32 and rounded to bf16 (or fp16) by torch.
"""
from __future__ import annotations

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, std: float = 1.0, dtype=torch.bfloat16, device="cpu"):
    g = _gen(seed, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def normal_with_outliers(shape, seed: int, rate: float = 0.01, outlier_mult: float = 20.0,
                         std: float = 1.0, dtype=torch.bfloat16, device="cpu"):
    g = _gen(seed, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if rate > 0:
        u = torch.rand(*shape, generator=g, device=device, dtype=torch.float32)
        x = torch.where(u < rate, x * outlier_mult, x)
    return x.to(dtype)


def student_t_columns(shape, seed: int, every: int = 32, nu4: bool = True,
                      dtype=torch.bfloat16, device="cpu"):
    """N(0,1) rows x cols, with one column in ``every`` (chosen by the seed)
    replaced by Student-t(4) draws."""
    rows, cols = shape
    g = _gen(seed, device)
    x = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
    ncols = max(1, cols // every)
    perm = torch.randperm(cols, generator=g, device=device)[:ncols]
    z = torch.randn(rows, ncols, generator=g, device=device, dtype=torch.float32)
    u1 = torch.rand(rows, ncols, generator=g, device=device, dtype=torch.float32)
    u2 = torch.rand(rows, ncols, generator=g, device=device, dtype=torch.float32)
    # keep the uniforms away from 0 so the logarithm stays finite
    u1 = u1.clamp_min(1e-12)
    u2 = u2.clamp_min(1e-12)
    chi2 = -2.0 * torch.log(u1 * u2)
    t = z / torch.sqrt(chi2 / 4.0)
    x[:, perm] = t
    return x.to(dtype)


def kv_with_spikes(tokens: int, heads: int, head_dim: int, seed: int,
                   rate: float = 1e-4, spike_mult: float = 50.0,
                   dtype=torch.bfloat16, device="cpu"):
    return normal_with_outliers((tokens, heads, head_dim), seed, rate=rate,
                                outlier_mult=spike_mult, dtype=dtype, device=device)


def bits16(t: torch.Tensor):
    """numpy uint16 view of a bf16/fp16 CPU tensor (same bytes)."""
    import numpy as np
    t = t.detach().to("cpu").contiguous()
    return t.view(torch.int16).numpy().view(np.uint16)


def random_codes(shape, seed: int, device="cpu"):
    """Uniform random bytes (every e4m3 / int8 code, NaN codes included)."""
    g = _gen(seed, device)
    return torch.randint(0, 256, shape, generator=g, device=device, dtype=torch.int32).to(torch.uint8)
