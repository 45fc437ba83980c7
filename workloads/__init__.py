"""Seeded synthetic inputs for the MX-scaled FP8 ``wo_a`` path.

This module holds no arithmetic of the method itself (no RoPE, no
quantisation, no GEMM).  It draws the raw inputs -- BF16 activations,
positions, the BF16 cos/sin cache and FP32 weights -- and it is the only
code that both the oracle side and the CUDA side of the tests consume.

Recipe (deterministic on any machine with numpy and torch):

* activations: numpy ``Generator(PCG64(seed)).standard_normal`` in float32,
  times ``std``; with ``outlier_frac`` > 0 a Bernoulli mask drawn from the
  same generator multiplies that fraction of elements by ``outlier_mult``;
  then one round-to-nearest-even to BF16 (torch's float32 -> bfloat16).
* positions: ``arange`` for prefill chunks, or uniform integers in
  ``[0, max_pos)`` drawn from PCG64(seed).
* cos/sin cache: theta_i = base^(-2i/R) and angle = pos * theta_i in float64,
  cos/sin in float64, rounded to float32 and then to BF16 (both RNE).
  This is the forward-rotation cache a model keeps; the operator applies
  the inverse rotation itself.
* weights: float32 N(0, std) from PCG64(seed); the E4M3 codes and E8M0
  scales are made from these by whichever quantiser a side uses.

The *_cuda variants draw the same distributions on the GPU with a seeded
torch generator (different numbers, same recipe) for the throughput bench,
where no oracle value is compared.
"""

from __future__ import annotations

import numpy as np
import torch

# Shapes of the operator's workloads (tokens T, groups G, row length D = K,
# output features N, RoPE width R).
WO_A = dict(G=8, D=4096, N=1024, R=64)
TINY = dict(T=16, G=2, D=256, N=128, R=64)
DECODE_T = (1, 8, 32, 64)
PREFILL_T = 8192
LINEAR_N = 5120
LINEAR_K = (576, 288, 2304)
LINEAR_M = (1, 8)
STREAM_CHUNKS = (8192,) * 12 + (1696,)
STREAM_LAYERS = 61
ROPE_BASE = 10000.0


def bf16_normal(shape, seed: int, std: float = 1.0, outlier_frac: float = 0.0,
                outlier_mult: float = 50.0) -> torch.Tensor:
    """BF16 CPU tensor of N(0, std) samples (with optional x`outlier_mult`
    outliers), one RNE rounding from float32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    v = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    if outlier_frac > 0.0:
        mask = rng.random(size=shape, dtype=np.float32) < np.float32(outlier_frac)
        v[mask] *= np.float32(outlier_mult)
    return torch.from_numpy(v).to(torch.bfloat16)


def f32_normal(shape, seed: int, std: float = 1.0) -> torch.Tensor:
    """float32 CPU tensor of N(0, std) samples."""
    rng = np.random.Generator(np.random.PCG64(seed))
    v = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    return torch.from_numpy(v)


def positions_arange(start: int, T: int) -> torch.Tensor:
    return torch.arange(start, start + T, dtype=torch.int64)


def positions_uniform(T: int, seed: int, max_pos: int) -> torch.Tensor:
    rng = np.random.Generator(np.random.PCG64(seed))
    return torch.from_numpy(rng.integers(0, max_pos, size=T, dtype=np.int64))


def rope_cache(max_pos: int, R: int, base: float = ROPE_BASE):
    """(cos, sin) BF16 CPU tensors [max_pos, R/2] of the forward rotation."""
    half = R // 2
    i = np.arange(half, dtype=np.float64)
    theta = base ** (-2.0 * i / R)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * theta[None, :]
    cos = torch.from_numpy(np.cos(ang).astype(np.float32)).to(torch.bfloat16)
    sin = torch.from_numpy(np.sin(ang).astype(np.float32)).to(torch.bfloat16)
    return cos.contiguous(), sin.contiguous()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a BF16 tensor (numpy has no bfloat16)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------- GPU side
def bf16_normal_cuda(shape, seed: int, std: float = 1.0, outlier_frac: float = 0.0,
                     outlier_mult: float = 50.0, device="cuda") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        v *= std
    if outlier_frac > 0.0:
        mask = torch.rand(shape, generator=g, device=device) < outlier_frac
        v[mask] *= outlier_mult
    return v.to(torch.bfloat16)


def f32_normal_cuda(shape, seed: int, std: float = 1.0, device="cuda") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        v *= std
    return v


def positions_uniform_cuda(T: int, seed: int, max_pos: int, device="cuda") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randint(0, max_pos, (T,), generator=g, device=device, dtype=torch.int64)
