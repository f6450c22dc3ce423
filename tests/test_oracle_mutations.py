"""Plant plausible mistakes in copies of the oracle's routines (on the CPU) and
check that at least one pin catches each: a wrong constant, a dropped term, a
swapped exponent, a transposed operand, truncation instead of rounding."""
import numpy as np
import pytest

import oracle_pins as P
from oracle import codecs as C
from oracle import quant as Q
from oracle import smooth as S
from oracle import gemm as G

F32 = np.float32


def _fp8_rows_div447(x):
    x = np.asarray(x, np.float32)
    s = np.maximum(np.abs(x).max(-1), F32(1e-8)) / F32(447)
    return C.e4m3fn_encode(x / s[:, None]), s


def _fp8_rows_truncate(x):
    x = np.asarray(x, np.float32)
    s = np.maximum(np.abs(x).max(-1), F32(1e-8)) / F32(448)
    xs = (x / s[:, None]).astype(np.float64)
    a = np.abs(xs)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    step = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)
    return C.e4m3fn_encode(np.trunc(xs / step) * step), s


def _fp8_groups_64(x):
    x = np.asarray(x, np.float32)
    R, K = x.shape
    q, s = Q.fp8_per_row(x.reshape(-1, 64))
    return q.reshape(R, K), s.reshape(R, K // 64)


def _int8_rows_128(x, smooth=None, *, weight=False):
    x = np.asarray(x, np.float32)
    S_ = np.maximum(np.abs(x).max(-1), F32(1e-8)) / F32(128)
    return C.int8_encode(x / S_[:, None]), S_


def _int8_rows_smooth_wrong_side(x, smooth=None, *, weight=False):
    x = np.asarray(x, np.float32)
    if smooth is not None:
        x = x / smooth                       # weights divided instead of multiplied
    S_ = np.maximum(np.abs(x).max(-1), F32(1e-8)) / F32(127)
    return C.int8_encode(x / S_[:, None]), S_


def _nvfp4_g_without_6(x):
    x = np.asarray(x, np.float32)
    R, K = x.shape
    amax = F32(np.abs(x).max())
    g = amax / F32(448) if amax > 0 else F32(1)
    xb = x.reshape(R, K // 16, 16)
    c = C.e4m3fn_encode((np.abs(xb).max(-1) / F32(6)) / g)
    s = np.where(c == 0, F32(1), (C.e4m3fn_decode(c).astype(np.float32) * g)).astype(np.float32)
    q = np.where((c == 0)[..., None], 0, C.e2m1_encode(xb / s[..., None]))
    return q.reshape(R, K).astype(np.uint8), c, amax, g


def _nvfp4_block_without_6(x):
    x = np.asarray(x, np.float32)
    R, K = x.shape
    amax = F32(np.abs(x).max())
    g = amax / F32(2688) if amax > 0 else F32(1)
    xb = x.reshape(R, K // 16, 16)
    c = C.e4m3fn_encode(np.abs(xb).max(-1) / g)
    s = np.where(c == 0, F32(1), (C.e4m3fn_decode(c).astype(np.float32) * g)).astype(np.float32)
    q = np.where((c == 0)[..., None], 0, C.e2m1_encode(xb / s[..., None]))
    return q.reshape(R, K).astype(np.uint8), c, amax, g


def _mxfp4_emax1(x):
    x = np.asarray(x, np.float32)
    R, K = x.shape
    xb = x.reshape(R, K // 32, 32).astype(np.float64)
    a = np.abs(xb).max(-1)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.clip(np.where(a > 0, ex - 1 - 1, -127), -127, 127)
    return C.e2m1_encode(np.ldexp(xb, -e[..., None])).reshape(R, K), (e + 127).astype(np.uint8)


def _smooth_swapped(ax, aw, alpha):
    return S.smooth_factors_from_maxima(ax, aw, 1.0 - alpha)


def _smooth_no_weight_term(ax, aw, alpha):
    return np.power(np.asarray(ax, np.float64), alpha)


def _matmul_transposed_output(xh, wh):
    y, b = G.matmul_ref(xh, wh)
    return y[::-1, ::-1], b


def _matmul_dropped_last_k(xh, wh):
    return G.matmul_ref(np.asarray(xh)[:, :-1], np.asarray(wh)[:, :-1])


def _factored_scales_swapped(xq, wq, sx, sw):
    acc = np.asarray(xq, np.float64) @ np.asarray(wq, np.float64).T
    return np.asarray(sw, np.float64)[:acc.shape[0], None] * acc * np.asarray(sx, np.float64)[None, :acc.shape[1]].mean()


def _int8_exact_in_int16(a, b):
    return (np.asarray(a, np.int16) @ np.asarray(b, np.int16).T).astype(np.int64)


def _e4m3_values_bias8():
    return C._table(4, 3, 8, C._e4m3fn_special)


MUTANTS = [
    ("e4m3 bias 8", lambda: P.pin_e4m3_table(_e4m3_values_bias8())),
    ("fp8 divisor 447", lambda: P.pin_fp8_rows(_fp8_rows_div447)),
    ("fp8 truncation", lambda: P.pin_fp8_rows(_fp8_rows_truncate)),
    ("fp8 group of 64", lambda: P.pin_fp8_groups(_fp8_groups_64)),
    ("int8 divisor 128", lambda: P.pin_int8_rows(_int8_rows_128)),
    ("int8 smoothing on the wrong side", lambda: P.pin_int8_smoothing_exact(_int8_rows_smooth_wrong_side)),
    ("nvfp4 tensor scale without the 6", lambda: P.pin_nvfp4(_nvfp4_g_without_6)),
    ("nvfp4 block scale without the 6", lambda: P.pin_nvfp4(_nvfp4_block_without_6)),
    ("mxfp4 emax 1", lambda: P.pin_mxfp4(_mxfp4_emax1)),
    ("smooth alpha swapped", lambda: P.pin_smoothquant_channel112(_smooth_swapped)),
    ("smooth weight term dropped", lambda: P.pin_smoothquant_three_channel(_smooth_no_weight_term)),
    ("gemm output transposed", lambda: P.pin_gemm_bruteforce(_matmul_transposed_output)),
    ("gemm dropped a k term", lambda: P.pin_gemm_bruteforce(_matmul_dropped_last_k)),
    ("epilogue scales swapped", lambda: P.pin_factored_epilogue(_factored_scales_swapped)),
    ("int8 accumulate in int16", lambda: P.pin_int8_exact(_int8_exact_in_int16)),
]


@pytest.mark.parametrize("name,run", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pin_catches_mutant(name, run):
    with pytest.raises((AssertionError, ValueError, IndexError)):
        run()
