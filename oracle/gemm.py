"""GEMM references: the dequantized product in fp64, the factored epilogue, and
the exact INT8 product.  Test infrastructure only.

The product the path computes is Y = X^ W^T with X^ and W^ the dequantized
operands; with per-row scales it factors as
    X^ W^T = diag(s_X) (X_q W_q^T) diag(s_W)
("FP8 and FP4 inference, SmoothQuant and activation quantization", section
"Scale granularity"; "Low-bit LLM Weights and Activations", section 3.4).
Block-scaled operands (1x128 / 128x128 FP8, NVFP4, MXFP4) do not factor; their
reference is the dequantized product itself.

Products of decoded codes (at most 4 significant bits) and fp32 scales are
exact in fp64, so `dequant` is exact; the fp64 matmul (a library primitive) adds
only fp64 rounding.
"""
from __future__ import annotations

import numpy as np

from .codecs import bf16_ulp, bf16_round


def matmul_ref(xh, wh):
    """Y_ref = X^ W^T in fp64, and B = |X^| |W^|^T (the tolerance's scale)."""
    xh = np.asarray(xh, dtype=np.float64)
    wh = np.asarray(wh, dtype=np.float64)
    return xh @ wh.T, np.abs(xh) @ np.abs(wh).T


def factored_ref(xq_vals, wq_vals, sx, sw):
    """diag(s_X) (X_q W_q^T) diag(s_W): decoded codes multiplied first, the
    per-row scales applied after the reduction (the epilogue form)."""
    acc = np.asarray(xq_vals, np.float64) @ np.asarray(wq_vals, np.float64).T
    return np.asarray(sx, np.float64)[:, None] * acc * np.asarray(sw, np.float64)[None, :]


def int8_exact(xq, wq):
    """INT8 x INT8 -> exact integer accumulation (int64)."""
    return np.asarray(xq, np.int64) @ np.asarray(wq, np.int64).T


def int8_epilogue_fp32(acc, sx, sw):
    """bf16((fp32(acc) * s_x[t]) * s_w[n]) in fp32, left to right, RNE to bf16
    ("FP8 and INT8 Inference", section 5 "INT8 in practice":
    Y = Y_int32 x s_x[token] x s_w[channel])."""
    a = np.asarray(acc, dtype=np.float32)
    y = (a * np.asarray(sx, np.float32)[:, None]) * np.asarray(sw, np.float32)[None, :]
    return bf16_round(y)


def tolerance(y_ref, abs_sum, rel: float = 1e-3):
    """|y - y_ref| <= rel * sum_k |x^_k||w^_k| + one bf16 ulp of y_ref."""
    return rel * np.asarray(abs_sum, np.float64) + bf16_ulp(y_ref)


def check(y, y_ref, abs_sum, rel: float = 1e-3):
    """Boolean mask of outputs within tolerance, and the worst ratio err / tol."""
    err = np.abs(np.asarray(y, np.float64) - y_ref)
    tol = tolerance(y_ref, abs_sum, rel)
    return err <= tol, float(np.max(err / tol)) if err.size else 0.0


def sampled_ref(xh_rows, wh_rows):
    """Row-by-row references for sampled (m, n) pairs: inputs are the sampled
    dequantized rows [S, K] of X and W; returns y_ref[S] and abs_sum[S]."""
    xh = np.asarray(xh_rows, np.float64)
    wh = np.asarray(wh_rows, np.float64)
    return np.einsum("sk,sk->s", xh, wh), np.einsum("sk,sk->s", np.abs(xh), np.abs(wh))
