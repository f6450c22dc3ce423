"""FP8 GEMM with 1x128 activation and 128x128 weight block scales (promotion
of every 128-wide K group in fp32) vs the oracle's fp64 dequantized product.
Tolerance: |y - y_ref| <= 1e-3 * sum_k |x^_k w^_k| + 1 bf16 ulp."""
import numpy as np
import pytest
import torch

import synth
from oracle import codecs as C
from oracle import quant as Q
from oracle import gemm as G
from gpu_util import lpq, dev_bf16, dev, host, bf16_to_f64

pytestmark = pytest.mark.gpu


def _dequant_block(qx, sx, qw, sw):
    M, K = qx.shape
    N = qw.shape[0]
    xh = (C.e4m3fn_decode(qx).reshape(M, K // 128, 128) * sx[..., None]).reshape(M, K)
    wv = C.e4m3fn_decode(qw)
    wh = np.empty_like(wv)
    for i in range((N + 127) // 128):
        for j in range(K // 128):
            wh[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128] = wv[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128] * sw[i, j]
    return xh, wh


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (1, 128, 256), (200, 296, 1024), (2048, 1024, 4096),
                                   (130, 4096, 14336), (513, 640, 512)])
def test_fp8_block_gemm(M, N, K):
    L = lpq()
    xb = synth.activations(M, K, 7000 + M, n_outlier=max(1, K // 1000), lo=50, hi=500)
    wb = synth.weights(N, K, 7001 + N)
    qx, sx = Q.fp8_per_group_1x128(synth.f32_from_bf16_bits(xb))
    qw, sw = Q.fp8_per_block_128x128_ragged(synth.f32_from_bf16_bits(wb))
    Y = L.gemm_scaled(L.FMT_FP8, L.GRAN_BLOCK_1x128, L.GRAN_BLOCK_128x128, dev(qx), dev(qw),
                      dev(np.ascontiguousarray(sx.T)), dev(sw), M=M, N=N, K=K)
    torch.cuda.synchronize()
    assert L.lpq_read_error_word() == 0
    yr, b = G.matmul_ref(*_dequant_block(qx, sx, qw, sw))
    ok, worst = G.check(bf16_to_f64(host(Y)), yr, b)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} out of tolerance, worst {worst:.3g}"


def test_fp8_block_end_to_end():
    L = lpq()
    w = synth.configs.PREFILL_FP8_BLOCK
    M, (K, N) = 256, (4096, 4096)
    xb = synth.configs.make_x(w, M, K)
    wb = synth.configs.make_w(w, N, K)
    qx, sx = L.quantize_act_fp8(dev_bf16(xb), L.GRAN_BLOCK_1x128)
    qw, sw = L.quantize_weight_fp8(dev_bf16(wb), L.GRAN_BLOCK_128x128)
    Y = L.gemm_scaled(L.FMT_FP8, L.GRAN_BLOCK_1x128, L.GRAN_BLOCK_128x128, qx, qw, sx, sw, M=M, N=N, K=K)
    torch.cuda.synchronize()
    assert L.lpq_read_error_word() == 0
    qxo, sxo = Q.fp8_per_group_1x128(synth.f32_from_bf16_bits(xb))
    qwo, swo = Q.fp8_per_block_128x128_ragged(synth.f32_from_bf16_bits(wb))
    yr, b = G.matmul_ref(*_dequant_block(qxo, sxo, qwo, swo))
    ok, worst = G.check(bf16_to_f64(host(Y)), yr, b)
    assert ok.all(), worst


def test_fp8_block_gemm_activations_larger_than_l2():
    """69 MB of activation codes (more than half the L2) and 4 MB of weights:
    tiles are visited weight-column fastest so each activation row block is
    read once.  Checked on a sample of rows against the oracle."""
    L = lpq()
    M, N, K = 8448, 512, 8192
    xb = synth.activations(M, K, 7100, n_outlier=8, lo=50, hi=500)
    wb = synth.weights(N, K, 7101)
    qx, sx = Q.fp8_per_group_1x128(synth.f32_from_bf16_bits(xb))
    qw, sw = Q.fp8_per_block_128x128_ragged(synth.f32_from_bf16_bits(wb))
    Y = L.gemm_scaled(L.FMT_FP8, L.GRAN_BLOCK_1x128, L.GRAN_BLOCK_128x128, dev(qx), dev(qw),
                      dev(np.ascontiguousarray(sx.T)), dev(sw), M=M, N=N, K=K)
    torch.cuda.synchronize()
    assert L.lpq_read_error_word() == 0
    rows = np.arange(0, M, 97)
    xh, wh = _dequant_block(qx[rows], sx[rows], qw, sw)
    yr, b = G.matmul_ref(xh, wh)
    ok, worst = G.check(bf16_to_f64(host(Y)[rows]), yr, b)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} out of tolerance, worst {worst:.3g}"
