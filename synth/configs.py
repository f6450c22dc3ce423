"""The five synthetic workloads of the quantized-linear path, by name and shape.

Shapes are Llama-8B-like projections (qkv, o, gate+up, down) for FP8 decode and
block-scaled prefill, the INT8 SmoothQuant case, and the NVFP4/MXFP4 W4A4 case.
Every K and N is a multiple of 128.
"""
from __future__ import annotations

from dataclasses import dataclass, field

# (K, N) of the four projections: qkv, o, gate+up, down.
LLAMA8B_PROJ = {
    "qkv": (4096, 6144),
    "o": (4096, 4096),
    "gate_up": (4096, 28672),
    "down": (14336, 4096),
}


@dataclass(frozen=True)
class Workload:
    name: str
    fmt: str                      # "fp8" | "fp8_block" | "int8" | "nvfp4" | "mxfp4"
    Ms: tuple
    KNs: tuple                    # ((K, N), ...)
    x_sigma: float = 1.0
    w_sigma: float = 0.02
    outlier: dict = field(default_factory=dict)   # kwargs for synth.activations
    index: int = 0


TINY_FP8 = Workload("tiny_fp8_w8a8_16x256x256", "fp8", (16,), ((256, 256),),
                    outlier=dict(n_outlier=4, fixed_factor=100.0), index=0)

DECODE_FP8 = Workload("llama8b_decode_fp8_w8a8", "fp8", (1, 16, 64, 256),
                      tuple(LLAMA8B_PROJ.values()),
                      outlier=dict(lo=50.0, hi=500.0), index=1)

PREFILL_FP8_BLOCK = Workload("llama8b_prefill_fp8_block1x128_128x128", "fp8_block", (2048, 8192),
                             tuple(LLAMA8B_PROJ.values()),
                             outlier=dict(lo=50.0, hi=500.0), index=2)

INT8_SMOOTHQUANT = Workload("int8_w8a8_smoothquant_a0.5", "int8", (256, 4096),
                            ((4096, 4096), (4096, 28672)),
                            outlier=dict(lo=50.0, hi=500.0), index=3)
INT8_CALIB_TOKENS = 512
SMOOTH_ALPHA = 0.5

NVFP4_W4A4 = Workload("nvfp4_w4a4", "nvfp4", (512, 8192), ((8192, 8192), (8192, 28672)),
                      w_sigma=0.015, outlier=dict(lo=10.0, hi=2000.0, log_uniform=True), index=4)
MXFP4_W4A4 = Workload("mxfp4_w4a4", "mxfp4", (512, 8192), ((8192, 8192), (8192, 28672)),
                      w_sigma=0.015, outlier=dict(lo=10.0, hi=2000.0, log_uniform=True), index=4)

ALL = (TINY_FP8, DECODE_FP8, PREFILL_FP8_BLOCK, INT8_SMOOTHQUANT, NVFP4_W4A4, MXFP4_W4A4)


def make_x(w: Workload, M: int, K: int, salt: int = 0):
    """Activation bits [M, K] for workload w (seed 1000 + config index)."""
    from . import activations, SEED_X, SEED_OUTLIER
    return activations(M, K, SEED_X + w.index + 17 * salt, outlier_seed=SEED_OUTLIER + w.index,
                       sigma=w.x_sigma, **w.outlier)


def make_w(w: Workload, N: int, K: int, salt: int = 0):
    """Weight bits [N, K] for workload w (seed 2000 + config index)."""
    from . import weights, SEED_W
    return weights(N, K, SEED_W + w.index + 17 * salt, sigma=w.w_sigma)


def make_calib(w: Workload, K: int, tokens: int = INT8_CALIB_TOKENS):
    """SmoothQuant calibration batch [tokens, K] (seed 3000), same outlier channels."""
    from . import activations, SEED_CAL, SEED_OUTLIER
    return activations(tokens, K, SEED_CAL, outlier_seed=SEED_OUTLIER + w.index,
                       sigma=w.x_sigma, **w.outlier)
