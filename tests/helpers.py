"""Shared test helpers: seeded inputs (from synth), oracle references, and the
accuracy criterion for the bf16 output.

Tolerance (bf16 Y vs the oracle's bf16 Y, both widened to fp32):
    max |dY| <= 1e-2 * max |Y_ref|   and   ||dY||_2 <= 2e-3 * ||Y_ref||_2.
The GPU accumulates in fp32 and rounds once to bf16; the oracle accumulates
exactly in fp64 and rounds once to bf16, so most elements agree bit for bit
and the rest differ by one bf16 ulp (relative 2^-8) at rounding boundaries.
The pages report 3.1e-3 max relative difference against their library and a
rel 2e-2 unit-test bound ("[AMD] Small-M FP8 block-scale GEMM with fused
activation quant for gfx950 (Qwen3.5)", "Modifications" and "Kernel
microbenchmarks").
"""

from __future__ import annotations

import os

import numpy as np

import synth

MAX_ABS_FRAC = 1e-2
REL_L2 = 2e-3


def threads() -> int:
    return max(1, os.cpu_count() or 1)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(h)


def check_y(y_gpu_bits: np.ndarray, y_ref_bits: np.ndarray, what: str = "") -> dict:
    a = bf16_to_f32(y_gpu_bits).astype(np.float64)
    b = bf16_to_f32(y_ref_bits).astype(np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    assert np.all(np.isfinite(a)), f"{what}: non-finite GPU output"
    d = np.abs(a - b)
    max_ref = float(np.abs(b).max()) if b.size else 0.0
    l2_ref = float(np.sqrt((b * b).sum()))
    stats = {
        "max_abs": float(d.max()) if d.size else 0.0,
        "max_ref": max_ref,
        "rel_l2": float(np.sqrt((d * d).sum()) / l2_ref) if l2_ref > 0 else 0.0,
        "frac_exact": float((d == 0).mean()) if d.size else 1.0,
    }
    assert stats["max_abs"] <= MAX_ABS_FRAC * max_ref, f"{what}: {stats}"
    assert stats["rel_l2"] <= REL_L2, f"{what}: {stats}"
    return stats


def weight(oracle, N: int, K: int, kind: int, seed: int):
    """Seeded fp32 weight, block-quantised by the oracle: (wq, ws) numpy."""
    w = synth.w_f32(N, K, seed=seed)
    return oracle.quant_weight_128x128(w, kind)


def torch_u16_to_np(t) -> np.ndarray:
    return t.contiguous().view(__import__("torch").int16).cpu().numpy().view(np.uint16)
