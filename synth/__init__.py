"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers in the shapes and distributions of the
workloads the pages measure ("[AMD] Small-M FP8 block-scale GEMM with fused
activation quant for gfx950 (Qwen3.5)", sections "Modifications" and "Kernel
microbenchmarks": the projection shapes 5120x4096, 4608x4096, 4096x2048 at
1..32 tokens).  It holds none of the method's arithmetic: no quantisation, no
scales, no GEMM.  Both the CUDA library's callers and the CPU oracle's callers
take their inputs from here, so both sides see identical bytes.

Recipes:
  x  -- bf16 [M, K]: fp32 N(0, 1), optionally with each entry independently
        chosen with probability 1% and multiplied by 20 (outliers), then
        rounded to bf16 (nearest even).
  W  -- fp32 [N, K]: N(0, 0.02).
  gamma -- bf16 [K], the RMSNorm weight of the producer: fp32 1 + 0.25 * N(0, 1),
        rounded to bf16 (nearest even).
  MoE routing -- per token S slots: S-1 distinct routed experts drawn uniformly
        from experts 0 .. E-2 with weights exp(N(0, 1)) normalised to sum 1,
        and the shared expert E-1 in the last slot with weight 1 (Qwen3.5's
        11 slots per token: 10 routed + 1 shared, out of 513 experts).
Seeds: ``seed = 1000 * workload + copy`` by convention of the callers.
"""

from __future__ import annotations

import numpy as np

OUTLIER_FRACTION = 0.01
OUTLIER_SCALE = 20.0
WEIGHT_STD = 0.02


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def x_bf16(M: int, K: int, seed: int, outliers: bool = True) -> np.ndarray:
    """Activations as bf16 bit patterns, uint16 [M, K]."""
    rng = _rng(seed)
    v = rng.standard_normal((M, K), dtype=np.float32)
    if outliers:
        pick = rng.random((M, K)) < OUTLIER_FRACTION
        v = np.where(pick, v * np.float32(OUTLIER_SCALE), v).astype(np.float32)
    return f32_to_bf16_bits(v)


def w_f32(N: int, K: int, seed: int) -> np.ndarray:
    """Weights before block quantisation, float32 [N, K] ~ N(0, 0.02)."""
    rng = _rng(seed)
    return (rng.standard_normal((N, K), dtype=np.float32) * np.float32(WEIGHT_STD)).astype(
        np.float32)


GAMMA_STD = 0.25


def gamma_bf16(K: int, seed: int) -> np.ndarray:
    """RMSNorm weight as bf16 bit patterns, uint16 [K] ~ 1 + N(0, 0.25)."""
    rng = _rng(seed)
    v = (np.float32(1.0) + rng.standard_normal(K, dtype=np.float32) * np.float32(GAMMA_STD))
    return f32_to_bf16_bits(v.astype(np.float32))


def moe_routing(M: int, S: int, E: int, seed: int):
    """(ids int32 [M, S], weights float32 [M, S]) per the routing recipe."""
    rng = _rng(seed)
    ids = np.empty((M, S), dtype=np.int32)
    w = np.empty((M, S), dtype=np.float32)
    for m in range(M):
        ids[m, :S - 1] = rng.choice(E - 1, size=S - 1, replace=False)
        ids[m, S - 1] = E - 1
        g = np.exp(rng.standard_normal(S - 1)).astype(np.float64)
        w[m, :S - 1] = (g / g.sum()).astype(np.float32)
        w[m, S - 1] = 1.0
    return ids, w


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Device-side draws for the benchmark's large rotated weight sets.  These use
# torch's CUDA generator: the same recipe, a different stream of numbers, so
# they never stand in for an oracle comparison.
# ---------------------------------------------------------------------------

def x_bf16_torch(M: int, K: int, seed: int, device, outliers: bool = True):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    v = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    if outliers:
        pick = torch.rand((M, K), generator=g, device=device) < OUTLIER_FRACTION
        v = torch.where(pick, v * OUTLIER_SCALE, v)
    return v.to(torch.bfloat16)


def w_f32_torch(N: int, K: int, seed: int, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn((N, K), generator=g, device=device, dtype=torch.float32) * WEIGHT_STD
