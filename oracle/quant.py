"""Dynamic quantizers, in fp32, in the pages' order of operations.  Test infrastructure only.

Inputs are fp32 arrays holding bf16 values (exact).  Every function returns the
codes and scales the stored artefact holds, in a plain logical layout:

* codes: one code per element, same shape as the input (E2M1 codes unpacked,
  one per uint8);
* scales: fp32 for FP8 / INT8, [rows, K / block] codes for NVFP4 / MXFP4.

Readings of points the pages leave open:

* r1 ties round to even (the emulation's `torch.round`);
* r2 `x / s` is a correctly rounded fp32 division, never a reciprocal multiply;
* r3 the 1e-8 floor of the FP8 activation scale (emulation `clamp(min=1e-8)`)
  is used for every FP8 and INT8 scale, so an all-zero row gets s = 1e-8 / qmax
  and codes 0;
* r4 overflow saturates to +-448 / +-6, never NaN (E4M3FN has no infinity;
  the saturating OCP mode);
* r5 the sign of zero is kept;
* r6 the NVFP4 tensor scale g is computed per whole tensor, for activations
  and weights alike; an all-zero tensor gets g = 1;
* r7 an NVFP4 block whose E4M3 scale code rounds to 0 is stored as all-zero
  codes (a zero scale code decodes every element of the block to 0 anyway);
* r8 the MXFP4 scale is the OCP MX shared exponent
  floor(log2 amax_block) - 2 (2 = largest exponent of E2M1), clamped to
  [-127, 127]; an all-zero block gets exponent -127;
* r10 SmoothQuant factors are applied inside the INT8 quantizers: activations
  divided, weights multiplied, in fp32, with no bf16 rounding in between;
* r11 INT8 codes are symmetric, +-127.
"""
from __future__ import annotations

import numpy as np

from .codecs import (e4m3fn_encode, e4m3fn_decode, e2m1_encode, int8_encode)

F32 = np.float32
SCALE_FLOOR = F32(1e-8)      # "FP8 and FP4 inference ...", Implementation sketch: clamp(min=1e-8)
E4M3_MAX = F32(448.0)
E2M1_MAX = F32(6.0)
INT8_MAX = F32(127.0)
NVFP4_GLOBAL_DIV = F32(448.0 * 6.0)    # 2688
NVFP4_BLOCK = 16
MXFP4_BLOCK = 32
FP8_ACT_GROUP = 128
FP8_WEIGHT_BLOCK = 128


def _f32(x):
    return np.asarray(x, dtype=np.float32)


# ------------------------------------------------------------------- FP8 ----
def fp8_per_row(x):
    """Per-row (per-token activation, per-output-channel weight) FP8 E4M3FN.

    s = max(max_k |x|, 1e-8) / 448, q = E4M3FN(x / s).
    "FP8 and FP4 inference, SmoothQuant and activation quantization",
    section "Implementation sketch" (fp8_per_token) and section "Scale
    granularity" (per-channel weights = one scale per output row).
    Returns (codes uint8 [R, K], s float32 [R]).
    """
    x = _f32(x)
    amax = np.max(np.abs(x), axis=-1)
    s = np.maximum(amax, SCALE_FLOOR) / E4M3_MAX
    q = e4m3fn_encode(x / s[..., None])
    return q, s.astype(np.float32)


def fp8_per_group_1x128(x, group: int = FP8_ACT_GROUP):
    """Activations scaled per 1x128 K-group (DeepSeek-V3 style).

    The per-token rule applied to each run of 128 consecutive K elements of a
    row ("FP8 and FP4 inference ...", section "Scale granularity";
    "FP8 and INT8 Inference", section 5 "What DeepSeek did").
    Returns (codes uint8 [R, K], s float32 [R, K/128]).
    """
    x = _f32(x)
    R, K = x.shape
    assert K % group == 0
    xg = x.reshape(R, K // group, group)
    amax = np.max(np.abs(xg), axis=-1)
    s = np.maximum(amax, SCALE_FLOOR) / E4M3_MAX
    q = e4m3fn_encode(xg / s[..., None]).reshape(R, K)
    return q, s.astype(np.float32)


def fp8_per_block_128x128(w, block: int = FP8_WEIGHT_BLOCK):
    """Weights scaled per 128x128 block (DeepSeek-V3 style), same rule per block.
    Returns (codes uint8 [N, K], s float32 [N/128, K/128]).  N and K must be
    multiples of 128 here; the GPU path also accepts a ragged last block, which
    `fp8_per_block_128x128_ragged` covers.
    """
    return fp8_per_block_128x128_ragged(w, block)


def fp8_per_block_128x128_ragged(w, block: int = FP8_WEIGHT_BLOCK):
    w = _f32(w)
    N, K = w.shape
    nb, kb = -(-N // block), -(-K // block)
    s = np.empty((nb, kb), dtype=np.float32)
    q = np.empty((N, K), dtype=np.uint8)
    for i in range(nb):
        for j in range(kb):
            blk = w[i * block:(i + 1) * block, j * block:(j + 1) * block]
            a = np.max(np.abs(blk))
            sc = np.maximum(a, SCALE_FLOOR) / E4M3_MAX
            s[i, j] = sc
            q[i * block:(i + 1) * block, j * block:(j + 1) * block] = e4m3fn_encode(blk / sc)
    return q, s


def fp8_static(x, s):
    """Static (calibrated) per-tensor FP8: q = E4M3FN(x / s) with a given s
    ("FP8 and FP4 inference ...", section "Scale granularity", static)."""
    return e4m3fn_encode(_f32(x) / F32(s))


def fp8_dequant(q, s):
    return e4m3fn_decode(q) * np.asarray(s, dtype=np.float64)


# ------------------------------------------------------------------ INT8 ----
def int8_per_row(x, smooth=None, *, weight: bool = False):
    """Symmetric per-row INT8 with optional SmoothQuant factors.

    Activation rows: x~ = x / s_j (per input channel j); weight rows:
    w~ = w * s_j ("Low-bit LLM Weights and Activations", section 4.2, the
    identity X diag(s)^-1 . diag(s) W).  Then S = max(max|x~|, 1e-8) / 127 and
    q = clamp(round(x~ / S), +-127) ("Low-bit LLM Weights and Activations",
    section 2.1; "FP8 and INT8 Inference", section 4 int8PerTensor, applied
    per token / per output channel as in section 5 "INT8 in practice").
    Returns (codes int8 [R, K], S float32 [R]).
    """
    x = _f32(x)
    if smooth is not None:
        sm = _f32(smooth)
        x = x * sm if weight else x / sm
    amax = np.max(np.abs(x), axis=-1)
    S = np.maximum(amax, SCALE_FLOOR) / INT8_MAX
    q = int8_encode(x / S[..., None])
    return q, S.astype(np.float32)


def int8_per_tensor(x):
    """One scale for the whole tensor, S = max|x| / 127 (the pages' tiny
    example, "FP8 and INT8 Inference", section 4)."""
    x = _f32(x)
    S = np.max(np.abs(x)) / INT8_MAX
    return int8_encode(x / S), F32(S)


def int_symmetric(x, qmax: int):
    """Per-tensor symmetric integer quantizer with levels -qmax..qmax, in fp64
    (the 4-bit hand example of "FP8 and FP4 inference ...", section "Worked
    example: three channels, one outlier", uses qmax = 7)."""
    x = np.asarray(x, dtype=np.float64)
    step = np.max(np.abs(x)) / qmax
    return np.clip(np.rint(x / step), -qmax, qmax), step


# ----------------------------------------------------------------- NVFP4 ----
def nvfp4(x):
    """NVFP4: E2M1 elements, one E4M3 scale per 16, one fp32 tensor scale.

    Steps of "FP8 and FP4 inference ...", section "Implementation sketch"
    (nvfp4), in fp32:
      g  = max|x| / (448 * 6)                         (tensor scale)
      c  = E4M3FN((max_block |x| / 6) / g)            (block scale code)
      s  = dec(c) * g ;  q = E2M1(x / s)
    Readings r6 (g = 1 for an all-zero tensor) and r7 (c == 0 -> codes 0).
    Returns (codes uint8 [R, K] unpacked 0..15, sf uint8 [R, K/16], amax f32, g f32).
    """
    x = _f32(x)
    R, K = x.shape
    assert K % NVFP4_BLOCK == 0
    amax = F32(np.max(np.abs(x))) if x.size else F32(0)
    g = amax / NVFP4_GLOBAL_DIV if amax > 0 else F32(1.0)
    g = F32(g)
    xb = x.reshape(R, K // NVFP4_BLOCK, NVFP4_BLOCK)
    amax_b = np.max(np.abs(xb), axis=-1)
    t = (amax_b / F32(6.0)) / g
    c = e4m3fn_encode(t)
    s = (e4m3fn_decode(c).astype(np.float32) * g).astype(np.float32)
    s_safe = np.where(c == 0, F32(1.0), s).astype(np.float32)
    q = e2m1_encode(xb / s_safe[..., None])
    q = np.where((c == 0)[..., None], np.uint8(0), q).astype(np.uint8)
    return q.reshape(R, K), c.astype(np.uint8), F32(amax), g


def nvfp4_dequant(q, sf, g):
    """x^ = E2M1(q) * E4M3(sf) * g, exactly, in fp64."""
    from .codecs import e2m1_decode
    R, K = q.shape
    v = e2m1_decode(q).reshape(R, K // NVFP4_BLOCK, NVFP4_BLOCK)
    return (v * e4m3fn_decode(sf)[..., None] * float(g)).reshape(R, K)


# ----------------------------------------------------------------- MXFP4 ----
def _floor_log2(a):
    """floor(log2 a) for finite a > 0, exactly, from the binary exponent."""
    _, ex = np.frexp(np.asarray(a, dtype=np.float64))     # a = m 2^ex, m in [0.5, 1)
    return ex - 1


def mxfp4(x):
    """MXFP4: E2M1 elements with one power-of-two (E8M0) scale per 32.

    Scale rule (reading r8, OCP MX): e = clamp(floor(log2 max_block|x|) - 2,
    -127, 127), stored code e + 127, q = E2M1(x * 2^-e) (exact scaling).
    "FP8 and FP4 inference ...", section "Scale granularity" (16- and 32-element
    blocks); "Low-bit LLM Weights and Activations", section 2.4 (E8M0, bias 127,
    32 elements).
    Returns (codes uint8 [R, K] unpacked, sf uint8 [R, K/32]).
    """
    x = _f32(x)
    R, K = x.shape
    assert K % MXFP4_BLOCK == 0
    xb = x.reshape(R, K // MXFP4_BLOCK, MXFP4_BLOCK).astype(np.float64)
    amax_b = np.max(np.abs(xb), axis=-1)
    e = np.where(amax_b > 0, _floor_log2(np.where(amax_b > 0, amax_b, 1.0)) - 2, -127)
    e = np.clip(e, -127, 127).astype(np.int64)
    q = e2m1_encode(np.ldexp(xb, -e[..., None]))
    return q.reshape(R, K).astype(np.uint8), (e + 127).astype(np.uint8)


def mxfp4_dequant(q, sf):
    from .codecs import e2m1_decode, e8m0_decode
    R, K = q.shape
    v = e2m1_decode(q).reshape(R, K // MXFP4_BLOCK, MXFP4_BLOCK)
    return (v * e8m0_decode(sf)[..., None]).reshape(R, K)
