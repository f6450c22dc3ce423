"""GPU quantizers vs the CPU oracle, bit-exact codes and scales (through the C ABI)."""
import numpy as np
import pytest
import torch

import synth
from oracle import quant as Q
from oracle import smooth as S
from gpu_util import lpq, dev_bf16, dev, host, unpack_nibbles, sf_to_logical

pytestmark = pytest.mark.gpu


def _x(M, K, seed, **kw):
    kw.setdefault("n_outlier", max(1, K // 1000))
    kw.setdefault("lo", 50.0)
    kw.setdefault("hi", 500.0)
    return synth.activations(M, K, seed, **kw)


def _f32(bits):
    return synth.f32_from_bf16_bits(bits)


ROW_SHAPES = [(1, 16), (3, 256), (16, 4096), (64, 14336), (257, 1040), (5, 20480)]


@pytest.mark.parametrize("M,K", ROW_SHAPES)
def test_fp8_per_token(M, K):
    L = lpq()
    xb = _x(M, K, 100 + M + K)
    q, s = L.quantize_act_fp8(dev_bf16(xb), L.GRAN_ROW)
    qo, so = Q.fp8_per_row(_f32(xb))
    assert np.array_equal(host(s), so)
    assert np.array_equal(host(q), qo)


def test_fp8_every_bf16_value():
    """All finite bf16 bit patterns, 256 per row, each row with its own scale."""
    L = lpq()
    b = synth.all_bf16_finite()
    pad = (-len(b)) % 256
    b = np.concatenate([b, np.zeros(pad, np.uint16)]).reshape(-1, 256)
    b = b[np.random.Generator(np.random.PCG64(1)).permutation(b.shape[0])]
    q, s = L.quantize_act_fp8(dev_bf16(b), L.GRAN_ROW)
    qo, so = Q.fp8_per_row(_f32(b))
    assert np.array_equal(host(s), so)
    assert np.array_equal(host(q), qo)
    # and with one scale for everything (static): every bf16 value through x / s
    st = torch.tensor([0.37], dtype=torch.float32, device="cuda")
    q2, _ = L.quantize_act_fp8(dev_bf16(b), L.GRAN_TENSOR_STATIC, static_scale=st)
    assert np.array_equal(host(q2), Q.fp8_static(_f32(b), np.float32(0.37)))


def _many_scales(M, K, seed):
    """Rows whose magnitudes span 2^-40 .. 2^40 (a different divisor per row, per
    1x128 group and per 16-block), some rows holding small integer multiples of
    a power of two so that many quotients are exact or sit on rounding ties."""
    g = np.random.Generator(np.random.PCG64(seed))
    e = g.integers(-40, 41, size=(M, 1)).astype(np.float64)
    x = g.standard_normal((M, K)) * np.exp2(e)
    ints = g.integers(-448, 449, size=(M, K)).astype(np.float64) * np.exp2(e - 6)
    pick = (np.arange(M) % 3 == 1)[:, None]
    x = np.where(pick, ints, x).astype(np.float32)
    return synth.bf16_bits_from_f32(x)


def test_shared_divisor_quantizers_many_scales():
    """Codes of every quantizer whose divisor is shared by a row, a 1x128 group
    or a 16-element block (FP8 per token, FP8 1x128, INT8, NVFP4), over 2048
    rows with different magnitudes: each code must equal the oracle's, which
    divides exactly."""
    L = lpq()
    M, K = 2048, 1024
    xb = _many_scales(M, K, 77)
    xf = _f32(xb)
    X = dev_bf16(xb)
    q, s = L.quantize_act_fp8(X, L.GRAN_ROW)
    qo, so = Q.fp8_per_row(xf)
    assert np.array_equal(host(s), so) and np.array_equal(host(q), qo)
    q, s = L.quantize_act_fp8(X, L.GRAN_BLOCK_1x128)
    qo, so = Q.fp8_per_group_1x128(xf)
    assert np.array_equal(host(q), qo) and np.array_equal(host(s).reshape(K // 128, M).T, so)
    q, s = L.quantize_act_int8(X, None)
    qo, so = Q.int8_per_row(xf)
    assert np.array_equal(host(s), so) and np.array_equal(host(q), qo)
    q, sf, gs = L.quantize_nvfp4(X)
    qo, sfo, amax, gg = Q.nvfp4(xf)
    assert host(gs)[1] == gg
    assert np.array_equal(unpack_nibbles(host(q)), qo)
    assert np.array_equal(sf_to_logical(L, L.FMT_NVFP4, host(sf), M, K, 16), sfo)


@pytest.mark.parametrize("M,K", [(1, 128), (7, 4096), (130, 14336)])
def test_fp8_1x128(M, K):
    L = lpq()
    xb = _x(M, K, 200 + M)
    q, s = L.quantize_act_fp8(dev_bf16(xb), L.GRAN_BLOCK_1x128)
    qo, so = Q.fp8_per_group_1x128(_f32(xb))
    assert np.array_equal(host(q), qo)
    assert np.array_equal(host(s), so.T)          # stored K-group major


@pytest.mark.parametrize("N,K", [(128, 128), (300, 384), (256, 4096)])
def test_fp8_weight_128x128(N, K):
    L = lpq()
    wb = synth.weights(N, K, 300 + N)
    q, s = L.quantize_weight_fp8(dev_bf16(wb), L.GRAN_BLOCK_128x128)
    qo, so = Q.fp8_per_block_128x128_ragged(_f32(wb))
    assert np.array_equal(host(q), qo)
    assert np.array_equal(host(s), so)


def test_fp8_weight_per_channel():
    L = lpq()
    wb = synth.weights(1000, 4096, 301)
    q, s = L.quantize_weight_fp8(dev_bf16(wb), L.GRAN_ROW)
    qo, so = Q.fp8_per_row(_f32(wb))
    assert np.array_equal(host(q), qo) and np.array_equal(host(s), so)


@pytest.mark.parametrize("M,K,smooth", [(3, 256, False), (256, 4096, True), (33, 20480, True)])
def test_int8_act(M, K, smooth):
    L = lpq()
    xb = _x(M, K, 400 + M)
    sm = None
    if smooth:
        sm = np.exp(np.random.Generator(np.random.PCG64(K)).uniform(-3, 3, K)).astype(np.float32)
    q, s = L.quantize_act_int8(dev_bf16(xb), None if sm is None else dev(sm))
    qo, so = Q.int8_per_row(_f32(xb), sm)
    assert np.array_equal(host(s), so)
    assert np.array_equal(host(q), qo)


@pytest.mark.parametrize("N,K,smooth", [(5, 64, False), (512, 4096, True)])
def test_int8_weight(N, K, smooth):
    L = lpq()
    wb = synth.weights(N, K, 500 + N)
    sm = np.exp(np.random.Generator(np.random.PCG64(K + 1)).uniform(-3, 3, K)).astype(np.float32) if smooth else None
    q, s = L.quantize_weight_int8(dev_bf16(wb), None if sm is None else dev(sm))
    qo, so = Q.int8_per_row(_f32(wb), sm, weight=True)
    assert np.array_equal(host(s), so)
    assert np.array_equal(host(q), qo)


def test_int8_zero_row_and_saturation():
    L = lpq()
    x = np.zeros((4, 64), np.float32)
    x[1] = 3.0
    x[2, 5] = -1e30
    x[3, :] = np.linspace(-2, 2, 64)
    xb = synth.bf16_bits_from_f32(x)
    q, s = L.quantize_act_int8(dev_bf16(xb))
    qo, so = Q.int8_per_row(_f32(xb))
    assert np.array_equal(host(q), qo) and np.array_equal(host(s), so)


@pytest.mark.parametrize("R,K", [(7, 64), (130, 512), (512, 8192), (3, 96)])
def test_nvfp4(R, K):
    L = lpq()
    xb = _x(R, K, 600 + R, lo=10.0, hi=2000.0, log_uniform=True)
    q, sf, gs = L.quantize_nvfp4(dev_bf16(xb))
    qo, sfo, amax, g = Q.nvfp4(_f32(xb))
    gsh = host(gs)
    assert gsh[0] == amax and gsh[1] == g
    assert np.array_equal(unpack_nibbles(host(q)), qo)
    sfh = host(sf)
    assert np.array_equal(sf_to_logical(L, L.FMT_NVFP4, sfh, R, K, 16), sfo)
    # padding of the scale layout is zero
    used = np.zeros(sfh.size, bool)
    used[_sf_offsets(R, K, 16)] = True
    assert not sfh[~used].any()


def _sf_offsets(R, K, blk):
    kb = K // blk
    r = np.arange(R)[:, None]
    k = np.arange(kb)[None, :]
    kb4 = (kb + 3) // 4
    return (((r // 128) * kb4 + k // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + k % 4).ravel()


def test_nvfp4_zero_tensor_and_flushed_block():
    L = lpq()
    z = np.zeros((2, 64), np.uint16)
    q, sf, gs = L.quantize_nvfp4(dev_bf16(z))
    assert host(gs)[1] == 1.0 and not host(q).any() and not host(sf).any()
    x = np.zeros((1, 64), np.float32)
    x[0, 0] = 3.0e6
    x[0, 16] = 0.3
    xb = synth.bf16_bits_from_f32(x)
    q, sf, gs = L.quantize_nvfp4(dev_bf16(xb))
    qo, sfo, _, _ = Q.nvfp4(_f32(xb))
    assert np.array_equal(unpack_nibbles(host(q)), qo)
    assert np.array_equal(sf_to_logical(L, L.FMT_NVFP4, host(sf), 1, 64, 16), sfo)


@pytest.mark.parametrize("R,K", [(7, 64), (130, 512), (512, 8192), (2, 96)])
def test_mxfp4(R, K):
    L = lpq()
    xb = _x(R, K, 700 + R, lo=10.0, hi=2000.0, log_uniform=True)
    if R > 2:
        xb[1, :32] = 0                       # a zero block
    q, sf = L.quantize_mxfp4(dev_bf16(xb))
    qo, sfo = Q.mxfp4(_f32(xb))
    assert np.array_equal(unpack_nibbles(host(q)), qo)
    assert np.array_equal(sf_to_logical(L, L.FMT_MXFP4, host(sf), R, K, 32), sfo)


def test_mxfp4_every_bf16_value():
    L = lpq()
    b = synth.all_bf16_finite()
    pad = (-len(b)) % 256
    b = np.concatenate([b, np.zeros(pad, np.uint16)]).reshape(-1, 256)
    q, sf = L.quantize_mxfp4(dev_bf16(b))
    qo, sfo = Q.mxfp4(_f32(b))
    assert np.array_equal(unpack_nibbles(host(q)), qo)
    assert np.array_equal(sf_to_logical(L, L.FMT_MXFP4, host(sf), b.shape[0], 256, 32), sfo)


def test_nvfp4_every_bf16_value():
    L = lpq()
    b = synth.all_bf16_finite()
    b = b[np.abs(_f32(b)) < 1e30]            # keep g finite for the whole tensor
    pad = (-len(b)) % 256
    b = np.concatenate([b, np.zeros(pad, np.uint16)]).reshape(-1, 256)
    q, sf, gs = L.quantize_nvfp4(dev_bf16(b))
    qo, sfo, amax, g = Q.nvfp4(_f32(b))
    assert host(gs)[1] == g
    assert np.array_equal(unpack_nibbles(host(q)), qo)
    assert np.array_equal(sf_to_logical(L, L.FMT_NVFP4, host(sf), b.shape[0], 256, 16), sfo)


@pytest.mark.parametrize("alpha", [0.5, 0.8])
def test_smoothquant_calibration(alpha):
    L = lpq()
    w = synth.configs.INT8_SMOOTHQUANT
    K = 4096
    cal = synth.configs.make_calib(w, K)
    wb = synth.configs.make_w(w, 512, K)
    amax = torch.zeros(K, dtype=torch.float32, device="cuda")
    L.lpq_act_absmax_update(dev_bf16(cal[:300]), amax)       # two calibration chunks
    L.lpq_act_absmax_update(dev_bf16(cal[300:]), amax)
    ax = S.channel_absmax(_f32(cal))
    assert np.array_equal(host(amax), ax)
    s = L.smooth_calibrate(amax, dev_bf16(wb), alpha)
    so = S.smooth_factors(ax, _f32(wb), alpha)
    assert np.array_equal(host(s), so)


def test_int8_smoothquant_end_to_end_codes():
    """Calibrate on the GPU, then quantize activations and weights with the
    oracle's factors on both sides: identical codes and scales."""
    L = lpq()
    w = synth.configs.INT8_SMOOTHQUANT
    K = 4096
    cal = synth.configs.make_calib(w, K)
    xb = synth.configs.make_x(w, 256, K)
    wb = synth.configs.make_w(w, 256, K)
    so = S.smooth_factors(S.channel_absmax(_f32(cal)), _f32(wb), 0.5)
    qx, sx = L.quantize_act_int8(dev_bf16(xb), dev(so))
    qw, sw = L.quantize_weight_int8(dev_bf16(wb), dev(so))
    qxo, sxo = Q.int8_per_row(_f32(xb), so)
    qwo, swo = Q.int8_per_row(_f32(wb), so, weight=True)
    assert np.array_equal(host(qx), qxo) and np.array_equal(host(sx), sxo)
    assert np.array_equal(host(qw), qwo) and np.array_equal(host(sw), swo)


def test_invalid_arguments_rejected_on_host():
    L = lpq()
    X = dev_bf16(np.zeros((4, 64), np.uint16))
    Xq = torch.empty((4, 64), dtype=torch.uint8, device="cuda")
    sx = torch.empty(4, dtype=torch.float32, device="cuda")
    lib = L._lib()
    st = L._stream(None)
    assert lib.lpq_quantize_act_fp8(None, 4, 64, 64, 0, L._ptr(Xq), L._ptr(sx), st) == L.LPQ_ERR_NULL
    assert lib.lpq_quantize_act_fp8(L._ptr(X), 4, 60, 64, 0, L._ptr(Xq), L._ptr(sx), st) == L.LPQ_ERR_SHAPE
    assert lib.lpq_quantize_act_fp8(L._ptr(X), 4, 64, 32, 0, L._ptr(Xq), L._ptr(sx), st) == L.LPQ_ERR_SHAPE
    assert lib.lpq_quantize_act_fp8(L._ptr(X), 0, 64, 64, 0, L._ptr(Xq), L._ptr(sx), st) == L.LPQ_ERR_SHAPE
    assert lib.lpq_quantize_act_fp8(L._ptr(X), 4, 64, 64, 1, L._ptr(Xq), L._ptr(sx), st) == L.LPQ_ERR_SHAPE
    mis = ctypes_ptr_plus(X, 2)
    assert lib.lpq_quantize_act_fp8(mis, 4, 64, 64, 0, L._ptr(Xq), L._ptr(sx), st) == L.LPQ_ERR_ALIGN
    assert lib.lpq_quantize_act_fp8(L._ptr(X), 4, 64, 64, 7, L._ptr(Xq), L._ptr(sx), st) == L.LPQ_ERR_UNSUPPORTED
    assert lib.lpq_quantize_act_nvfp4(L._ptr(X), 4, 48, 64, L._ptr(Xq), L._ptr(Xq), L._ptr(sx), st) == L.LPQ_ERR_SHAPE
    torch.cuda.synchronize()
    assert L.lpq_read_error_word() == 0


def ctypes_ptr_plus(t, nbytes):
    import ctypes
    return ctypes.c_void_p(t.data_ptr() + nbytes)


def test_bounded_wait_records_timeout_and_context_survives():
    """The failure path of every kernel wait, made to run out on purpose: a
    barrier nothing completes, a 50 ms limit.  The kernel records its code in
    the device error word and returns; the context keeps working."""
    L = lpq()
    L.lpq_clear_error_word()
    L.lpq_selftest_bounded_wait(50_000_000)
    torch.cuda.synchronize()
    assert L.lpq_read_error_word() == L.LPQ_SELFTEST_WAIT_CODE
    L.lpq_clear_error_word()
    # the same context still runs the path
    X = torch.ones((4, 256), dtype=torch.bfloat16, device="cuda")
    q, s = L.quantize_act_fp8(X, L.GRAN_ROW)
    torch.cuda.synchronize()
    assert torch.all(s == s[0]) and L.lpq_read_error_word() == 0
