"""Seeded synthetic inputs for the quantized-linear path.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark.  It produces bf16 activation and weight matrices (as uint16 bit
patterns) and holds none of the quantization arithmetic: no scales, no codecs,
no rounding onto a low-precision grid.  The only conversion here is fp32 ->
bf16 round-to-nearest-even, which is how the inputs themselves are made.

Distributions follow the workloads the pages describe ("FP8 and FP4
inference, SmoothQuant and activation quantization", section "Measured: a 0.5B
instruct model on a laptop": a handful of input channels hundreds or thousands
of times the median, fixed across tokens; "Low-bit LLM Weights and
Activations", section 4.1: fewer than 0.1% of channels carry the outliers, the
same channels for every token).
"""
from __future__ import annotations

import math

import numpy as np

# Seeds: X = 1000 + config, W = 2000 + config, calibration batch = 3000,
# outlier-channel choice = 4000 (+ config).
SEED_X = 1000
SEED_W = 2000
SEED_CAL = 3000
SEED_OUTLIER = 4000


def bf16_bits_from_f32(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even; NaN kept quiet."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    nan = np.isnan(x)
    out = rounded.astype(np.uint16)
    if nan.any():
        out[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return out


def f32_from_bf16_bits(b) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp32 values."""
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def outlier_channels(K: int, count: int, seed: int) -> np.ndarray:
    """`count` distinct input channels in [0, K), sorted."""
    if count <= 0:
        return np.zeros(0, dtype=np.int64)
    return np.sort(_rng(seed).choice(K, size=count, replace=False)).astype(np.int64)


def activations(M: int, K: int, seed: int, *, n_outlier: int | None = None,
                outlier_seed: int = SEED_OUTLIER, lo: float = 50.0, hi: float = 500.0,
                log_uniform: bool = False, fixed_factor: float | None = None,
                sigma: float = 1.0) -> np.ndarray:
    """X ~ N(0, sigma^2) [M, K] with a few input channels scaled up for every token.

    n_outlier defaults to round(0.001 K) (0.1% of channels, at least 1).
    Each outlier channel j gets one factor f_j, drawn U[lo, hi] (or
    log-uniform on [lo, hi]), or `fixed_factor` for all of them.
    Returns bf16 bit patterns, shape [M, K].
    """
    if n_outlier is None:
        n_outlier = max(1, int(round(0.001 * K)))
    x = _rng(seed).standard_normal((M, K)) * sigma
    ch = outlier_channels(K, n_outlier, outlier_seed)
    if len(ch):
        r = _rng(outlier_seed + 1)
        if fixed_factor is not None:
            f = np.full(len(ch), fixed_factor)
        elif log_uniform:
            f = np.exp(r.uniform(math.log(lo), math.log(hi), size=len(ch)))
        else:
            f = r.uniform(lo, hi, size=len(ch))
        x[:, ch] *= f[None, :]
    return bf16_bits_from_f32(x.astype(np.float32))


def weights(N: int, K: int, seed: int, sigma: float = 0.02) -> np.ndarray:
    """W ~ N(0, sigma^2), [N, K] (out, in), as bf16 bit patterns."""
    w = _rng(seed).standard_normal((N, K)) * sigma
    return bf16_bits_from_f32(w.astype(np.float32))


def uniform_bits(shape, seed: int, lo: float, hi: float) -> np.ndarray:
    """U[lo, hi] values as bf16 bit patterns (edge-case tests)."""
    return bf16_bits_from_f32(_rng(seed).uniform(lo, hi, size=shape).astype(np.float32))


def all_bf16_finite() -> np.ndarray:
    """Every finite bf16 bit pattern (65536 minus the inf/NaN ones)."""
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    exp = (b >> 7) & 0xFF
    return b[exp != 0xFF]


def random_f32_bits(n: int, seed: int) -> np.ndarray:
    """n uniformly random finite fp32 values drawn by bit pattern."""
    u = _rng(seed).integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    return f[np.isfinite(f)]

from . import configs  # noqa: E402  (workload table; imports this module lazily)
