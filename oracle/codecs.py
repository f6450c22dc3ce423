"""Number-format codecs, defined from the bit layouts.  Test infrastructure only.

Decoding follows the field definitions of "Low-bit LLM Weights and
Activations", section 2.2 ("FP8 Format Comparison (OCP OFP8 1.0)" table and the
E4M3FN / E5M2 details) and section 2.4 (E2M1 element, E8M0 scale), with the
value formula (-1)^S 2^(E-bias) (1 + M/2^m) and subnormals M 2^(1-bias-m) from
"FP8 and FP4 inference, SmoothQuant and activation quantization", section "The
number formats".

Encoding is defined as: nearest value of the decoded finite grid, ties to the
code whose mantissa LSB is 0 (round-to-nearest-even), magnitudes beyond the
largest finite value saturate to it (the OCP saturating conversion mode, which
the pages' emulation also uses: its clamp to +-max).  The sign of zero is kept.
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------------------
# generic minifloat decode from (exponent bits, mantissa bits, bias)
# ----------------------------------------------------------------------------
def _minifloat_value(code: int, ebits: int, mbits: int, bias: int) -> float:
    sign = -1.0 if (code >> (ebits + mbits)) & 1 else 1.0
    E = (code >> mbits) & ((1 << ebits) - 1)
    M = code & ((1 << mbits) - 1)
    if E == 0:                                     # subnormal: M * 2^(1 - bias - m)
        return sign * M * 2.0 ** (1 - bias - mbits)
    return sign * (1.0 + M / 2.0 ** mbits) * 2.0 ** (E - bias)


def _table(ebits, mbits, bias, special):
    """value of every code; `special(code)` returns inf/nan or None."""
    n = 1 << (1 + ebits + mbits)
    vals = np.empty(n, dtype=np.float64)
    for c in range(n):
        s = special(c)
        vals[c] = _minifloat_value(c, ebits, mbits, bias) if s is None else s
    return vals


def _e4m3fn_special(c):
    # E4M3FN: no infinities; exponent 1111 with mantissa 111 is NaN (0x7F, 0xFF).
    return float("nan") if (c & 0x7F) == 0x7F else None


def _e5m2_special(c):
    # E5M2: IEEE-style; S.11111.00 = +-inf, S.11111.{01,10,11} = NaN.
    if (c & 0x7C) == 0x7C:
        if (c & 0x03) == 0:
            return float("-inf") if c & 0x80 else float("inf")
        return float("nan")
    return None


E4M3FN_VALUES = _table(4, 3, 7, _e4m3fn_special)      # 256 entries
E5M2_VALUES = _table(5, 2, 15, _e5m2_special)         # 256 entries
E2M1_VALUES = _table(2, 1, 1, lambda c: None)         # 16 entries: +-{0,.5,1,1.5,2,3,4,6}

E4M3FN_MAX = 448.0
E5M2_MAX = 57344.0
E2M1_MAX = 6.0


def _encode_nearest_even(v, pos_values: np.ndarray, sign_bit: int) -> np.ndarray:
    """Round |v| to the nearest entry of the ascending non-negative grid
    `pos_values` (index == code), ties to the even code, saturating at the top;
    then OR in the sign bit taken from v (so -0.0 and negative underflow keep it).
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    top = len(pos_values) - 1
    hi = np.searchsorted(pos_values, a, side="left")          # first grid value >= a
    hi = np.minimum(hi, top)
    lo = np.maximum(hi - 1, 0)
    mid = (pos_values[lo] + pos_values[hi]) * 0.5             # exact: few significant bits
    take_hi = (a > mid) | ((a == mid) & (lo % 2 == 1))
    code = np.where(take_hi, hi, lo)
    code = np.where(a >= pos_values[top], top, code)          # saturate
    code = np.where(pos_values[hi] == a, hi, code)            # exact hits
    neg = np.signbit(v)
    out = code.astype(np.uint16) | np.where(neg, sign_bit, 0).astype(np.uint16)
    return out


# ---------------------------------------------------------------- E4M3FN ----
_E4M3_POS = E4M3FN_VALUES[:0x7F]          # codes 0x00..0x7E, ascending, 0 .. 448


def e4m3fn_decode(codes) -> np.ndarray:
    return E4M3FN_VALUES[np.asarray(codes, dtype=np.uint8)]


def e4m3fn_encode(v) -> np.ndarray:
    """fp values -> E4M3FN codes (uint8), RNE, saturating to +-448; NaN -> 0x7F."""
    v = np.asarray(v)
    out = _encode_nearest_even(v, _E4M3_POS, 0x80).astype(np.uint8)
    nan = np.isnan(v)
    if np.any(nan):
        out = np.where(nan, np.uint8(0x7F), out)
    return out


# ------------------------------------------------------------------ E5M2 ----
_E5M2_POS = E5M2_VALUES[:0x7C]            # codes 0x00..0x7B, 0 .. 57344


def e5m2_decode(codes) -> np.ndarray:
    return E5M2_VALUES[np.asarray(codes, dtype=np.uint8)]


def e5m2_encode(v, saturate: bool = True) -> np.ndarray:
    """fp values -> E5M2 codes, RNE.  saturate=False sends overflow to +-inf
    (the IEEE-like mode); saturate=True clamps to +-57344."""
    v = np.asarray(v, dtype=np.float64)
    out = _encode_nearest_even(v, _E5M2_POS, 0x80).astype(np.uint8)
    if not saturate:
        # RNE would carry |v| >= 57344 + half a step (61440) to the next binade: inf.
        over = np.abs(v) >= 61440.0
        out = np.where(over, np.where(np.signbit(v), 0xFC, 0x7C), out).astype(np.uint8)
    nan = np.isnan(v)
    if np.any(nan):
        out = np.where(nan, np.uint8(0x7F), out)
    return out


# ------------------------------------------------------------------ E2M1 ----
_E2M1_POS = E2M1_VALUES[:8]               # 0, .5, 1, 1.5, 2, 3, 4, 6


def e2m1_decode(codes) -> np.ndarray:
    return E2M1_VALUES[np.asarray(codes, dtype=np.uint8) & 0xF]


def e2m1_encode(v) -> np.ndarray:
    """fp values -> E2M1 codes (uint8 in 0..15, bit 3 = sign), RNE, saturating at 6."""
    return _encode_nearest_even(v, _E2M1_POS, 0x8).astype(np.uint8)


# ------------------------------------------------------------------ E8M0 ----
def e8m0_decode(codes) -> np.ndarray:
    """8-bit pure exponent, bias 127: 2^(c - 127); 0xFF is NaN."""
    c = np.asarray(codes, dtype=np.int64)
    return np.where(c == 0xFF, np.nan, np.ldexp(1.0, c - 127))


# ------------------------------------------------------------------ INT8 ----
def int8_encode(v) -> np.ndarray:
    """Symmetric INT8 code: round half to even, clamp to [-127, 127] (the
    symmetric range of S = max|x|/127; two's complement -128 is left unused)."""
    return np.clip(np.rint(np.asarray(v, dtype=np.float64)), -127, 127).astype(np.int8)


# ------------------------------------------------------------------ bf16 ----
def bf16_round(v) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returns fp32 values.
    Used for the epilogue's output rounding in the INT8 one-ulp check."""
    x = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32)
    return np.where(np.isnan(x), x, out)


def bf16_ulp(v) -> np.ndarray:
    """Spacing of bf16 at |v| (8 significant bits); the subnormal spacing 2^-133 at 0."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, ex = np.frexp(a)                                   # a = m 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, -126)
    return np.where(a == 0, 2.0 ** -133, np.ldexp(1.0, e - 7))
