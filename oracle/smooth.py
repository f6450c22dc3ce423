"""SmoothQuant calibration.  Test infrastructure only.

"Low-bit LLM Weights and Activations", section 4.2: for Y = X W (W here stored
[out, in], so input channel j is column j of W),
    s_j = max|X_:j|^alpha / max|W_:j|^(1 - alpha),
with the maxima clamped below at 1e-5 as in the emulation of "FP8 and FP4
inference, SmoothQuant and activation quantization", section "Implementation
sketch" (smooth).  Reading r9: the power is taken in fp64 and the result
rounded once to fp32.
"""
from __future__ import annotations

import numpy as np

CLAMP = np.float32(1e-5)


def channel_absmax(x, running=None):
    """max_t |X_tj| per input channel j (fp32, exact), folded into `running`."""
    a = np.max(np.abs(np.asarray(x, dtype=np.float32)), axis=0)
    return a if running is None else np.maximum(np.asarray(running, np.float32), a)


def smooth_factors(act_amax, w, alpha: float = 0.5):
    """s_j = max(ax_j, 1e-5)^alpha / max(aw_j, 1e-5)^(1 - alpha), aw_j = max_n |W_nj|."""
    ax = np.maximum(np.asarray(act_amax, dtype=np.float32), CLAMP).astype(np.float64)
    aw = np.maximum(np.max(np.abs(np.asarray(w, dtype=np.float32)), axis=0), CLAMP).astype(np.float64)
    a = float(np.float32(alpha))
    return (np.power(ax, a) / np.power(aw, 1.0 - a)).astype(np.float32)


def smooth_factors_from_maxima(ax, aw, alpha: float):
    """The same formula on given channel maxima (fp64, no clamp needed for
    positive inputs); used for the pages' worked numbers."""
    ax = np.asarray(ax, dtype=np.float64)
    aw = np.asarray(aw, dtype=np.float64)
    return np.power(ax, alpha) / np.power(aw, 1.0 - alpha)
