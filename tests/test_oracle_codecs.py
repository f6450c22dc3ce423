"""Pins for the oracle's codecs against what the pages fix (CPU only).

* every E4M3FN / E5M2 table value the pages print (section 2.2 of "Low-bit LLM
  Weights and Activations", exercise 05);
* the E2M1 value set implied by the emulation's fp_round(x, 1, 0, 6);
* an independent restatement of the pages' fp_round emulation ("FP8 and FP4
  inference, SmoothQuant and activation quantization", "Implementation
  sketch"), with an exact floor(log2) from the binary exponent, checked against
  the table encoder on every finite bf16 value, on fp32 values around every
  rounding midpoint and on random fp32 bit patterns;
* the relative-error bound 2^-(m+1) of section "The number formats".
"""
import json
import os

import numpy as np
import pytest

from conftest import GOLDEN
from oracle import codecs as C
import synth


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def fp_round_restated(x, mbits, emin, maxv):
    """The emulation's rule, restated: e = max(floor(log2|x|), emin),
    step = 2^(e - mbits), round half to even of x/step, times step, clamped."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(ex - 1, emin)
    step = np.ldexp(1.0, e - mbits)
    q = np.rint(x / step) * step
    q = np.where(a > 0, q, x)
    return np.clip(q, -maxv, maxv)


# ------------------------------------------------------------------ tables --
def test_e4m3fn_printed_table():
    g = _golden("e4m3fn_e5m2_table.json")["e4m3fn"]
    V = C.E4M3FN_VALUES
    assert V[int(g["max_code_pos"], 16)] == g["max_finite"]
    assert V[int(g["max_code_neg"], 16)] == -g["max_finite"]
    assert V[int(g["min_normal_code"], 16)] == g["min_positive_normal"]
    one = int(g["one_code"], 16)
    assert V[one] == 1.0 and V[one + 1] - V[one] == g["ulp_at_one"]
    nan_codes = sorted(int(c, 16) for c in g["nan_codes"])
    assert sorted(np.flatnonzero(np.isnan(V)).tolist()) == nan_codes
    assert not np.any(np.isinf(V))                       # FN: no infinities
    for z in g["zero_codes"]:
        assert V[int(z, 16)] == 0.0
    assert np.signbit(V[0x80]) and not np.signbit(V[0x00])
    fin = V[np.isfinite(V)]
    assert fin.max() == g["max_finite"] and fin.min() == -g["max_finite"]
    # max = 1.75 * 2^8 from the bit layout (exponent 15, mantissa 6)
    assert (1 + 6 / 8) * 2.0 ** (15 - g["bias"]) == g["max_finite"]
    # smallest subnormal 2^-9 and the IEEE-style E4M3 maximum the FN variant exceeds
    assert V[0x01] == 2.0 ** -9
    assert (1 + 7 / 8) * 2.0 ** (14 - 7) == g["ieee_e4m3_would_stop_at"]


def test_e5m2_printed_table():
    g = _golden("e4m3fn_e5m2_table.json")["e5m2"]
    V = C.E5M2_VALUES
    assert V[int(g["max_code_pos"], 16)] == g["max_finite"]
    assert V[0x04] == g["min_positive_normal"]
    one = int(g["one_code"], 16)
    assert V[one] == 1.0 and V[one + 1] - V[one] == g["ulp_at_one"]
    for c in g["inf_codes"]:
        assert np.isinf(V[int(c, 16)])
    assert sorted(np.flatnonzero(np.isnan(V)).tolist()) == sorted(int(c, 16) for c in g["nan_codes"])
    assert (1 + 3 / 4) * 2.0 ** (30 - g["bias"]) == g["max_finite"]


def test_e2m1_value_set():
    g = _golden("e2m1_and_error_bounds.json")
    assert C.E2M1_VALUES[:8].tolist() == g["e2m1_nonnegative_values"]
    assert C.E2M1_VALUES[8:].tolist() == [-v for v in g["e2m1_nonnegative_values"]]


def test_e8m0_and_int8():
    assert C.e8m0_decode([127, 128, 0, 254]).tolist() == [1.0, 2.0, 2.0 ** -127, 2.0 ** 127]
    assert np.isnan(C.e8m0_decode([255])[0])
    assert C.int8_encode([0.5, 1.5, 2.5, -0.5, -2.5, 200.0, -200.0]).tolist() == [0, 2, 2, 0, -2, 127, -127]


# --------------------------------------- table encoder vs fp_round restated --
def _e4m3_midpoints_and_grid():
    pos = C.E4M3FN_VALUES[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    pts = np.concatenate([pos, mids, [464.0, 480.0, 1e4]]).astype(np.float32)
    # fp32 neighbours: +-64 ulps around each point, both signs
    u = pts.view(np.uint32).astype(np.int64)
    offs = np.arange(-64, 65)
    near = (u[:, None] + offs[None, :]).clip(0, 0x7F7FFFFF).astype(np.uint32).view(np.float32).ravel()
    return np.concatenate([near, -near])


@pytest.mark.parametrize("name,mbits,emin,maxv,enc,dec", [
    ("e4m3fn", 3, -6, 448.0, C.e4m3fn_encode, C.e4m3fn_decode),
    ("e2m1", 1, 0, 6.0, C.e2m1_encode, C.e2m1_decode),
])
def test_encoder_matches_fp_round(name, mbits, emin, maxv, enc, dec):
    xs = [synth.f32_from_bf16_bits(synth.all_bf16_finite()),
          synth.random_f32_bits(1 << 21, seed=7)]
    if name == "e4m3fn":
        xs.append(_e4m3_midpoints_and_grid())
    else:
        grid = C.E2M1_VALUES[:8]
        pts = np.concatenate([grid, (grid[:-1] + grid[1:]) / 2, [7.0, 8.0]]).astype(np.float32)
        u = pts.view(np.uint32).astype(np.int64)
        near = (u[:, None] + np.arange(-64, 65)[None, :]).clip(0, 0x7F7FFFFF).astype(np.uint32).view(np.float32).ravel()
        xs.append(np.concatenate([near, -near]))
    x = np.concatenate(xs)
    got = dec(enc(x))
    want = fp_round_restated(x, mbits, emin, maxv)
    bad = got != want
    assert not bad.any(), (name, x[bad][:8], got[bad][:8], want[bad][:8])
    # the sign of zero is kept
    assert np.array_equal(np.signbit(got[got == 0]), np.signbit(x[got == 0]))


def test_e5m2_encoder_matches_fp_round():
    x = np.concatenate([synth.f32_from_bf16_bits(synth.all_bf16_finite()),
                        synth.random_f32_bits(1 << 20, seed=8)])
    got = C.e5m2_decode(C.e5m2_encode(x))
    want = fp_round_restated(x, 2, -14, 57344.0)
    assert np.array_equal(got, want)
    # non-saturating mode: overflow goes to inf, as the IEEE-style layout allows
    y = C.e5m2_decode(C.e5m2_encode(np.array([61439.0, 61440.0, -7e4]), saturate=False))
    assert y[0] == 57344.0 and np.isinf(y[1]) and y[2] == -np.inf


def test_saturation_never_nan():
    big = np.array([448.0, 449.0, 463.99, 464.0, 479.0, 480.0, 1e30, 3.4e38], np.float32)
    codes = C.e4m3fn_encode(np.concatenate([big, -big]))
    assert set(codes.tolist()) == {0x7E, 0xFE}
    assert set(C.e2m1_encode(np.array([6.0, 6.5, 7.0, 1e9, -1e9])).tolist()) == {0x7, 0xF}


def test_e2m1_ties_to_even():
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0])
    assert C.e2m1_decode(C.e2m1_encode(x)).tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, -0.0, -4.0]


@pytest.mark.parametrize("name,enc,dec,mbits,lo,hi", [
    ("e4m3fn", C.e4m3fn_encode, C.e4m3fn_decode, 3, 2.0 ** -6, 448.0),
    ("e5m2", C.e5m2_encode, C.e5m2_decode, 2, 2.0 ** -14, 57344.0),
    ("e2m1", C.e2m1_encode, C.e2m1_decode, 1, 1.0, 6.0),
])
def test_relative_error_bound(name, enc, dec, mbits, lo, hi):
    bound = _golden("e2m1_and_error_bounds.json")["relative_error_bound"][name]
    assert bound == 2.0 ** -(mbits + 1)
    r = np.random.Generator(np.random.PCG64(11))
    x = np.exp(r.uniform(np.log(lo), np.log(hi), 200000)).astype(np.float32)
    x = np.concatenate([x, -x])
    rel = np.abs(dec(enc(x)) - x) / np.abs(x)
    assert rel.max() <= bound
    # the worst case sits at a midpoint just above a power of two:
    # half a step over 2^e (1 + 2^-(m+1)), so the bound is approached
    sup = bound / (1 + bound)
    assert sup * 0.97 < rel.max() <= sup
