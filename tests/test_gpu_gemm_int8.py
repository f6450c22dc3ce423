"""INT8 W8A8 (SmoothQuant) GEMM vs the oracle: the int32 accumulation is
exact, so the output must equal bf16((fp32(acc) * s_x[t]) * s_w[n]) computed
from the exact integer product, bit for bit.  Both kernels are covered: with
a workspace the product runs on the tcgen05 tensor cores through E4M3 digit
planes (q = 16 h + l), without one on the warp-level int8 MMA."""
import numpy as np
import pytest
import torch

import synth
from oracle import quant as Q
from oracle import smooth as S
from oracle import gemm as G
from gpu_util import lpq, dev_bf16, dev, host

pytestmark = pytest.mark.gpu


def _bits_f32(y_bits):
    return (np.asarray(y_bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("M,N,K", [(256, 4096, 4096), (1, 128, 64), (130, 200, 4096), (300, 520, 1040),
                                   (1024, 1024, 4096)])
@pytest.mark.parametrize("workspace", [False, True])
def test_int8_gemm_bit_exact(M, N, K, workspace):
    L = lpq()
    xb = synth.activations(M, K, 8000 + M, n_outlier=max(1, K // 1000), lo=50, hi=500)
    wb = synth.weights(N, K, 8001 + N)
    sm = np.exp(np.random.Generator(np.random.PCG64(K)).uniform(-2, 2, K)).astype(np.float32)
    qx, sx = Q.int8_per_row(synth.f32_from_bf16_bits(xb), sm)
    qw, sw = Q.int8_per_row(synth.f32_from_bf16_bits(wb), sm, weight=True)
    ws = L.workspace_for(L.FMT_INT8, L.GRAN_ROW, L.GRAN_ROW, M, N, K) if workspace else None
    Y = L.gemm_scaled(L.FMT_INT8, L.GRAN_ROW, L.GRAN_ROW, dev(qx), dev(qw), dev(sx), dev(sw), M=M, N=N, K=K,
                      workspace=ws)
    torch.cuda.synchronize()
    want = G.int8_epilogue_fp32(G.int8_exact(qx, qw), sx, sw)
    got = _bits_f32(host(Y))
    bad = got != want
    assert not bad.any(), f"{bad.sum()} of {bad.size} differ"
    assert L.lpq_read_error_word() == 0


@pytest.mark.parametrize("K", [8192, 65536])
@pytest.mark.parametrize("workspace", [False, True])
def test_int8_gemm_extreme_codes(K, workspace):
    """Codes at the ends of the int8 range (and around the digit boundary 16)
    over long K: the largest partial sums the digit planes produce (225 K for
    the low digits) must stay exact."""
    L = lpq()
    M, N = 64, 256
    g = np.random.Generator(np.random.PCG64(K + 5))
    vals = np.array([-128, -127, 127, 126, 0, 1, -1, 15, 16, -16, -17], np.int8)
    qx = g.choice(vals, size=(M, K)).astype(np.int8)
    qw = g.choice(vals, size=(N, K)).astype(np.int8)
    qx[0, :] = 127
    qw[0, :] = 127
    qx[1, :] = -128
    qw[1, :] = -128
    sx = g.uniform(1e-4, 1e-2, M).astype(np.float32)
    sw = g.uniform(1e-4, 1e-2, N).astype(np.float32)
    ws = L.workspace_for(L.FMT_INT8, L.GRAN_ROW, L.GRAN_ROW, M, N, K) if workspace else None
    Y = L.gemm_scaled(L.FMT_INT8, L.GRAN_ROW, L.GRAN_ROW, dev(qx), dev(qw), dev(sx), dev(sw), M=M, N=N, K=K,
                      workspace=ws)
    torch.cuda.synchronize()
    want = G.int8_epilogue_fp32(G.int8_exact(qx, qw), sx, sw)
    got = _bits_f32(host(Y))
    bad = got != want
    assert not bad.any(), f"{bad.sum()} of {bad.size} differ"
    assert L.lpq_read_error_word() == 0


def test_int8_smoothquant_end_to_end():
    """Calibrate, smooth, quantize and multiply on the GPU; compare with the
    oracle doing the same from the same bf16 inputs (bit-exact)."""
    L = lpq()
    w = synth.configs.INT8_SMOOTHQUANT
    M, (K, N) = 256, (4096, 4096)
    cal = synth.configs.make_calib(w, K)
    xb = synth.configs.make_x(w, M, K)
    wb = synth.configs.make_w(w, N, K)
    amax = torch.zeros(K, dtype=torch.float32, device="cuda")
    L.lpq_act_absmax_update(dev_bf16(cal), amax)
    s = L.smooth_calibrate(amax, dev_bf16(wb), 0.5)
    qx, sx = L.quantize_act_int8(dev_bf16(xb), s)
    qw, sw = L.quantize_weight_int8(dev_bf16(wb), s)
    Y = L.gemm_scaled(L.FMT_INT8, L.GRAN_ROW, L.GRAN_ROW, qx, qw, sx, sw, M=M, N=N, K=K)
    torch.cuda.synchronize()
    so = S.smooth_factors(S.channel_absmax(synth.f32_from_bf16_bits(cal)), synth.f32_from_bf16_bits(wb), 0.5)
    assert np.array_equal(host(s), so)
    qxo, sxo = Q.int8_per_row(synth.f32_from_bf16_bits(xb), so)
    qwo, swo = Q.int8_per_row(synth.f32_from_bf16_bits(wb), so, weight=True)
    want = G.int8_epilogue_fp32(G.int8_exact(qxo, qwo), sxo, swo)
    assert np.array_equal(_bits_f32(host(Y)), want)


def test_int8_weight_planes_and_planes_gemm():
    """lpq_int8_weight_planes: plane h holds the E4M3 code of floor(q / 16),
    plane l that of q - 16 floor(q / 16) (oracle codec); the GEMM on those
    planes (LPQ_GEMM_B_INT8_PLANES) gives the exact int32 result."""
    from oracle import codecs as C
    L = lpq()
    M, N, K = 300, 520, 1040
    g = np.random.Generator(np.random.PCG64(77))
    qx = g.integers(-128, 128, size=(M, K), dtype=np.int16).astype(np.int8)
    qw = g.integers(-128, 128, size=(N, K), dtype=np.int16).astype(np.int8)
    sx = g.uniform(1e-4, 1e-2, M).astype(np.float32)
    sw = g.uniform(1e-4, 1e-2, N).astype(np.float32)
    planes = L.int8_weight_planes(dev(qw))
    torch.cuda.synchronize()
    h = np.floor_divide(qw.astype(np.int64), 16)
    lo = qw.astype(np.int64) - 16 * h
    got = host(planes)
    assert np.array_equal(got[0], C.e4m3fn_encode(h.astype(np.float64)))
    assert np.array_equal(got[1], C.e4m3fn_encode(lo.astype(np.float64)))
    flags = L.GEMM_B_INT8_PLANES
    ws = L.workspace_for(L.FMT_INT8, L.GRAN_ROW, L.GRAN_ROW, M, N, K, flags=flags)
    Y = L.gemm_scaled(L.FMT_INT8, L.GRAN_ROW, L.GRAN_ROW, dev(qx), planes, dev(sx), dev(sw), M=M, N=N, K=K,
                      workspace=ws, flags=flags)
    torch.cuda.synchronize()
    want = G.int8_epilogue_fp32(G.int8_exact(qx, qw), sx, sw)
    assert np.array_equal(_bits_f32(host(Y)), want)
    assert L.lpq_read_error_word() == 0
    # planes without a workspace cannot fall back to the int8 MMA
    with pytest.raises(L.LpqError) as e:
        L.gemm_scaled(L.FMT_INT8, L.GRAN_ROW, L.GRAN_ROW, dev(qx), planes, dev(sx), dev(sw), M=M, N=N, K=K,
                      flags=flags)
    assert e.value.status == L.LPQ_ERR_WORKSPACE
