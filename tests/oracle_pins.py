"""Pin checks for the oracle, written as functions of the oracle routine they
check, so that the mutation tests can hand them a deliberately broken routine
and see them fail.  Each pin is something the pages or mathematics fix.
"""
import json
import os

import numpy as np

from conftest import GOLDEN
from oracle import codecs as C
from oracle import quant as Q
from oracle import smooth as S
from oracle import gemm as G
import synth


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _r4(v):
    return np.round(np.asarray(v, np.float64), 4)


# ----------------------------------------------------------------- codecs --
def pin_e4m3_table(values=None):
    g = golden("e4m3fn_e5m2_table.json")["e4m3fn"]
    V = C.E4M3FN_VALUES if values is None else values
    assert V[0x7E] == g["max_finite"] and V[0xFE] == -g["max_finite"]
    assert V[0x08] == g["min_positive_normal"]
    assert V[0x38] == 1.0 and V[0x39] - V[0x38] == g["ulp_at_one"]
    assert sorted(np.flatnonzero(np.isnan(V)).tolist()) == [0x7F, 0xFF]


# ------------------------------------------------------ the tiny example --
def pin_tiny_example(fp8_encode=None, int8_per_tensor=None):
    """FP8 (unit scale) and per-tensor INT8 on [60, 0.5, 2, 0.05, 30]."""
    g = golden("tiny_example_fp8_vs_int8.json")
    enc = fp8_encode or C.e4m3fn_encode
    i8 = int8_per_tensor or Q.int8_per_tensor
    x0 = np.array(g["input"], np.float64)          # the program's float64 inputs
    # the same inputs as fp32 and as bf16 (what the GPU path receives) give the
    # same codes; relative errors are taken against the printed inputs
    for x in (x0.astype(np.float32),
              synth.f32_from_bf16_bits(synth.bf16_bits_from_f32(x0.astype(np.float32)))):
        f8 = C.e4m3fn_decode(enc(x))
        assert np.array_equal(_r4(f8), g["fp8_e4m3_dequant_4dp"]), f8
        assert np.array_equal(np.round(np.abs(f8 - x0) / x0, 3), g["fp8_rel_err_3dp"])
        q, s = i8(x)
        d = q.astype(np.float64) * float(s)
        assert np.array_equal(_r4(d), g["int8_per_tensor_dequant_4dp"]), d
        assert np.array_equal(np.round(np.abs(d - x0) / x0, 3), g["int8_rel_err_3dp"])


# ------------------------------------------------------------ per-row FP8 --
def pin_fp8_rows(fn=None, seed=5):
    """Per-row invariants: each row's max element encodes to +-448 (0x7E/0xFE),
    s = max|x| / 448, every value within half a grid step of x / s."""
    fn = fn or Q.fp8_per_row
    x = synth.f32_from_bf16_bits(synth.activations(37, 384, seed, n_outlier=3, fixed_factor=300.0))
    q, s = fn(x)
    amax = np.abs(x).max(1)
    assert np.array_equal(s, (amax / np.float32(448)).astype(np.float32))
    idx = np.abs(x).argmax(1)
    top = q[np.arange(len(q)), idx]
    assert np.all(np.where(x[np.arange(len(q)), idx] > 0, top == 0x7E, top == 0xFE))
    xs = x.astype(np.float64) / s[:, None]
    v = C.e4m3fn_decode(q)
    # within the binade's half step: 2^-4 relative in the normal range, 2^-10 absolute below
    assert np.all(np.abs(v - xs) <= np.maximum(np.abs(xs) / 16, 2.0 ** -10) + 1e-12)


def pin_fp8_groups(fn=None):
    """1x128 groups behave as rows of 128: same codes and scales."""
    fn = fn or Q.fp8_per_group_1x128
    x = synth.f32_from_bf16_bits(synth.activations(9, 512, 6, n_outlier=2, fixed_factor=90.0))
    q, s = fn(x)
    q2, s2 = Q.fp8_per_row(x.reshape(-1, 128))
    assert np.array_equal(q.reshape(-1, 128), q2) and np.array_equal(s.reshape(-1), s2)
    assert s.shape == (9, 4)


def pin_fp8_blocks(fn=None):
    """128x128 weight blocks: one scale per block, block max -> +-448."""
    fn = fn or Q.fp8_per_block_128x128
    w = synth.f32_from_bf16_bits(synth.weights(256, 384, 7))
    q, s = fn(w)
    assert s.shape == (2, 3)
    for i in range(2):
        for j in range(3):
            blk = w[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            assert s[i, j] == np.float32(np.abs(blk).max()) / np.float32(448)
            qb = q[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            assert (C.e4m3fn_decode(qb) == 448.0).sum() + (C.e4m3fn_decode(qb) == -448.0).sum() >= 1


# ------------------------------------------------------------------ INT8 --
def pin_int8_rows(fn=None):
    fn = fn or Q.int8_per_row
    x = synth.f32_from_bf16_bits(synth.activations(11, 256, 8, n_outlier=2, fixed_factor=70.0))
    x[3] = 0.0                                           # an all-zero row
    q, s = fn(x)
    assert s[3] == np.float32(1e-8) / np.float32(127) and not q[3].any()
    rows = [r for r in range(11) if r != 3]
    idx = np.abs(x[rows]).argmax(1)
    assert np.all(np.abs(q[rows, idx]) == 127)
    assert q.min() >= -127
    xs = x.astype(np.float64) / s[:, None]
    assert np.all(np.abs(q - xs) <= 0.5 + 1e-9)


def pin_int8_smoothing_exact(fn=None):
    """X diag(s)^-1 . diag(s) W = X W: with power-of-two factors the smoothed
    operands are exact, so smoothing then quantizing equals quantizing the
    pre-scaled tensors."""
    fn = fn or Q.int8_per_row
    x = synth.f32_from_bf16_bits(synth.activations(8, 256, 9, n_outlier=2, fixed_factor=64.0))
    w = synth.f32_from_bf16_bits(synth.weights(16, 256, 10))
    sm = np.ldexp(1.0, np.random.Generator(np.random.PCG64(3)).integers(-4, 5, 256)).astype(np.float32)
    qx, sx = fn(x, sm)
    qw, sw = fn(w, sm, weight=True)
    qx2, sx2 = fn(x / sm, None)
    qw2, sw2 = fn(w * sm, None, weight=True)
    assert np.array_equal(qx, qx2) and np.array_equal(sx, sx2)
    assert np.array_equal(qw, qw2) and np.array_equal(sw, sw2)
    # the product identity, bitwise for power-of-two factors
    assert np.array_equal((x / sm).astype(np.float64) @ (w * sm).astype(np.float64).T,
                          x.astype(np.float64) @ w.astype(np.float64).T)


# ----------------------------------------------------------------- NVFP4 --
def pin_nvfp4(fn=None):
    """g = amax / 2688; the block holding the tensor max gets scale code 0x7E
    (448); every block with a normal scale code sends its max element to +-6;
    an all-zero tensor gets g = 1 and zero codes."""
    fn = fn or Q.nvfp4
    x = synth.f32_from_bf16_bits(synth.activations(6, 256, 11, n_outlier=2, lo=10, hi=2000, log_uniform=True))
    q, sf, amax, g = fn(x)
    assert amax == np.abs(x).max() and g == np.float32(amax) / np.float32(2688)
    r, c = np.unravel_index(np.abs(x).argmax(), x.shape)
    assert sf[r, c // 16] == 0x7E
    xb = x.reshape(6, 16, 16)
    qb = q.reshape(6, 16, 16)
    normal = sf >= 0x08
    idx = np.abs(xb).argmax(-1)
    top = np.take_along_axis(qb, idx[..., None], -1)[..., 0]
    assert np.all((top[normal] & 7) == 7)               # |E2M1| = 6
    qz, sfz, az, gz = fn(np.zeros((2, 32), np.float32))
    assert gz == 1.0 and not qz.any() and not sfz.any()
    # dequantized value within the E2M1 half step (relative 1/4) of x, or the subnormal half step
    d = Q.nvfp4_dequant(q, sf, g)
    s = (C.e4m3fn_decode(sf) * float(g))[..., None]
    assert np.all(np.abs(d.reshape(6, 16, 16) - xb) <= np.maximum(np.abs(xb) / 4, s / 4) + 1e-12)


def pin_nvfp4_flush_block(fn=None):
    """Reading r7: a block whose scale code rounds to 0 stores zero codes."""
    fn = fn or Q.nvfp4
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 3.0e6                  # g = 1116
    x[0, 16] = 0.3                   # (0.3/6)/g ~ 4.5e-5 < 2^-10 -> code 0
    q, sf, amax, g = fn(x)
    assert sf[0, 1] == 0 and not q[0, 16:].any() and sf[0, 0] == 0x7E


# ----------------------------------------------------------------- MXFP4 --
def pin_mxfp4(fn=None):
    """Power-of-two scales; the block max lands on +-4 or +-6; the scale code
    is floor(log2 amax_block) - 2 + 127; a zero block gets code 0, zero codes."""
    fn = fn or Q.mxfp4
    x = synth.f32_from_bf16_bits(synth.activations(5, 256, 12, n_outlier=2, lo=10, hi=2000, log_uniform=True))
    x[2, 64:96] = 0.0
    q, sf = fn(x)
    xb = x.reshape(5, 8, 32)
    qb = q.reshape(5, 8, 32)
    amax = np.abs(xb).max(-1)
    nz = amax > 0
    assert np.all(sf[~nz] == 0) and not qb[~nz].any()
    expect = np.floor(np.log2(amax[nz].astype(np.float64))) - 2 + 127
    assert np.array_equal(sf[nz].astype(np.float64), expect)
    idx = np.abs(xb).argmax(-1)
    top = np.take_along_axis(qb, idx[..., None], -1)[..., 0]
    assert np.all(np.isin(C.e2m1_decode(top[nz]), [4.0, 6.0, -4.0, -6.0]))


# -------------------------------------------------------------- smoothing --
def pin_smoothquant_three_channel(fn=None):
    g = golden("smoothquant_worked.json")["three_channel"]
    fn = fn or S.smooth_factors_from_maxima
    s = fn(g["act_channel_max"], g["weight_channel_max"], g["alpha"])
    assert np.allclose(s, g["s_3dp_or_4sf"], atol=6e-3, rtol=0)
    ax = np.array(g["act_channel_max"]) / s
    aw = np.array(g["weight_channel_max"]) * s
    assert np.allclose(ax, aw)                           # equal ranges at alpha = 0.5
    step = max(ax.max(), aw.max()) / g["levels"]
    assert round(step, 3) == g["smoothed_step_3dp"]
    assert round(58.0 / 7, 2) == g["unsmoothed_act_step_2dp"]
    assert round(0.55 / 7, 3) == g["unsmoothed_weight_step_3dp"]
    # the channel-max entries of the two tokens land on the printed codes
    for (tok, ch, val) in ((0, 0, 1.3), (1, 1, 0.9), (0, 2, 58.0)):
        k = int(np.rint(val / s[ch] / step))
        assert round(k * step, 3) == g["smoothed_act_dequant_3dp"][tok][ch]
    # every printed activation is an integer number of steps (the 4-bit grid)
    ks = np.array(g["smoothed_act_dequant_3dp"]) / step
    assert np.allclose(ks, np.rint(ks), atol=0.01)
    assert np.rint(ks).tolist() == [[5, -2, 7], [-3, 5, -5]]


def pin_smoothquant_channel112(fn=None):
    g = golden("smoothquant_worked.json")["channel_112"]
    fn = fn or S.smooth_factors_from_maxima
    for a, s_exp, xm, wm in zip(g["alpha"], g["s_2dp"], g["smoothed_act_max_2dp"], g["scaled_weight_max_2dp"]):
        s = float(fn(g["act_max"], g["weight_max"], a))
        assert abs(s - s_exp) <= 6e-3, (a, s)
        assert abs(g["act_max"] / s - xm) <= 0.01
        assert abs(g["weight_max"] * s - wm) <= 0.01


def pin_smooth_factors_calibration(fn=None):
    """The calibrated factors on matrices: alpha = 0.5 equalises the channel
    ranges (max |X~_j| = max |W~_j| = sqrt(ax aw)); alpha = 1 gives s = ax,
    alpha = 0 gives 1 / aw."""
    fn = fn or S.smooth_factors
    x = synth.f32_from_bf16_bits(synth.activations(64, 256, 13, n_outlier=2, fixed_factor=80.0))
    w = synth.f32_from_bf16_bits(synth.weights(32, 256, 14))
    ax = S.channel_absmax(x)
    s = fn(ax, w, 0.5).astype(np.float64)
    aw = np.abs(w).max(0).astype(np.float64)
    assert np.allclose(ax / s, aw * s, rtol=1e-6)
    assert np.allclose(ax / s, np.sqrt(ax * aw), rtol=1e-6)
    assert np.allclose(fn(ax, w, 1.0), ax, rtol=1e-7)
    assert np.allclose(fn(ax, w, 0.0), 1.0 / aw, rtol=1e-7)


# ------------------------------------------------------------------ GEMM --
def pin_gemm_bruteforce(fn=None, seed=21):
    """fp64 matmul of dequantized operands vs an exact rational triple loop."""
    from fractions import Fraction
    fn = fn or G.matmul_ref
    r = np.random.Generator(np.random.PCG64(seed))
    M, N, K = 3, 5, 7
    xh = C.e4m3fn_decode(r.integers(0, 256, (M, K)) & 0xF7) * 0.375
    wh = C.e4m3fn_decode(r.integers(0, 256, (N, K)) & 0xF7) * 1.25
    y, b = fn(xh, wh)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(xh[m, k])) * Fraction(float(wh[n, k])) for k in range(K))
            assert abs(Fraction(float(y[m, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200)
            assert float(b[m, n]) == float(sum(abs(Fraction(float(xh[m, k])) * Fraction(float(wh[n, k]))) for k in range(K)))


def pin_factored_epilogue(fn=None):
    """diag(s_X)(X_q W_q^T)diag(s_W) equals the dequantized product."""
    fn = fn or G.factored_ref
    x = synth.f32_from_bf16_bits(synth.activations(6, 128, 15, n_outlier=1, fixed_factor=50.0))
    w = synth.f32_from_bf16_bits(synth.weights(10, 128, 16))
    qx, sx = Q.fp8_per_row(x)
    qw, sw = Q.fp8_per_row(w)
    y1 = fn(C.e4m3fn_decode(qx), C.e4m3fn_decode(qw), sx, sw)
    y2, _ = G.matmul_ref(Q.fp8_dequant(qx, sx[:, None]), Q.fp8_dequant(qw, sw[:, None]))
    assert np.allclose(y1, y2, rtol=1e-14, atol=0)


def pin_int8_exact(fn=None):
    fn = fn or G.int8_exact
    r = np.random.Generator(np.random.PCG64(22))
    a = r.integers(-127, 128, (4, 9)).astype(np.int8)
    b = r.integers(-127, 128, (6, 9)).astype(np.int8)
    acc = fn(a, b)
    for m in range(4):
        for n in range(6):
            assert acc[m, n] == sum(int(a[m, k]) * int(b[n, k]) for k in range(9))
    # the largest magnitude K = 4096 can reach stays inside int32
    assert 127 * 127 * 4096 < 2 ** 31
