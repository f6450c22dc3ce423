"""NVFP4 and MXFP4 W4A4 GEMMs on the block-scaled FP4 tensor cores vs the
oracle's fp64 dequantized product (through the C ABI).

Inputs of the GEMM are the oracle's codes and scales, packed into the
library's layouts (nibbles; 128x4 scale tiles); one case quantizes on the GPU
first.  Tolerance: |y - y_ref| <= 1e-3 * sum_k |x^_k w^_k| + 1 bf16 ulp.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import codecs as C
from oracle import quant as Q
from oracle import gemm as G
from gpu_util import lpq, dev_bf16, dev, host, bf16_to_f64, pack_nibbles, logical_to_sf

pytestmark = pytest.mark.gpu


def _operands(fmt, M, N, K, seed):
    xb = synth.activations(M, K, seed, n_outlier=max(1, K // 1000), lo=10, hi=2000, log_uniform=True)
    wb = synth.weights(N, K, seed + 1, sigma=0.015)
    x = synth.f32_from_bf16_bits(xb)
    w = synth.f32_from_bf16_bits(wb)
    if fmt == "nvfp4":
        qx, sfx, _, gx = Q.nvfp4(x)
        qw, sfw, _, gw = Q.nvfp4(w)
        xh, wh = Q.nvfp4_dequant(qx, sfx, gx), Q.nvfp4_dequant(qw, sfw, gw)
        return xb, wb, (qx, sfx, gx), (qw, sfw, gw), xh, wh
    qx, sfx = Q.mxfp4(x)
    qw, sfw = Q.mxfp4(w)
    return xb, wb, (qx, sfx, None), (qw, sfw, None), Q.mxfp4_dequant(qx, sfx), Q.mxfp4_dequant(qw, sfw)


def _gpu_gemm(L, fmt, ox, ow, M, N, K, workspace=False):
    F = L.FMT_NVFP4 if fmt == "nvfp4" else L.FMT_MXFP4
    blk = 16 if fmt == "nvfp4" else 32
    qx, sfx, gx = ox
    qw, sfw, gw = ow
    A = dev(pack_nibbles(qx))
    B = dev(pack_nibbles(qw))
    sa = dev(logical_to_sf(L, F, sfx, M, K, blk))
    sb = dev(logical_to_sf(L, F, sfw, N, K, blk))
    ga = dev(np.array([gx], np.float32)) if gx is not None else None
    gb = dev(np.array([gw], np.float32)) if gw is not None else None
    ws = L.workspace_for(F, L.GRAN_ROW, L.GRAN_ROW, M, N, K) if workspace else None
    Y = L.gemm_scaled(F, L.GRAN_ROW, L.GRAN_ROW, A, B, sa, sb, M=M, N=N, K=K, ga=ga, gb=gb, workspace=ws)
    torch.cuda.synchronize()
    return bf16_to_f64(host(Y))


SHAPES = [(128, 128, 256), (1, 128, 64), (130, 200, 96), (512, 1024, 8192), (300, 640, 1056), (64, 8192, 2048),
          (96, 104, 256), (64, 24, 128)]   # a clipped last 32-column block; Y narrower than 32 columns


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("workspace", [False, True])
def test_fp4_gemm(fmt, M, N, K, workspace):
    L = lpq()
    _, _, ox, ow, xh, wh = _operands(fmt, M, N, K, 3000 + M + N + K)
    y = _gpu_gemm(L, fmt, ox, ow, M, N, K, workspace)
    yr, b = G.matmul_ref(xh, wh)
    ok, worst = G.check(y, yr, b)
    assert ok.all(), f"{fmt}: {(~ok).sum()} of {ok.size} out of tolerance, worst {worst:.3g}"
    assert L.lpq_read_error_word() == 0


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_fp4_hand_built_codes(fmt):
    """One-hot E2M1 codes with distinct scales per block: each output is a
    single product of two elements and two block scales."""
    L = lpq()
    M, N, K = 128, 128, 512
    blk = 16 if fmt == "nvfp4" else 32
    qx = np.zeros((M, K), np.uint8)
    qw = np.zeros((N, K), np.uint8)
    for m in range(M):
        qx[m, (5 * m) % K] = 7 if m % 3 else 15          # +-6
    for n in range(N):
        qw[n, (5 * n) % K] = 4                             # +2
    r = np.random.Generator(np.random.PCG64(9))
    if fmt == "nvfp4":
        sfx = r.integers(0x20, 0x50, (M, K // blk)).astype(np.uint8)
        sfw = r.integers(0x20, 0x50, (N, K // blk)).astype(np.uint8)
        gx, gw = np.float32(0.75), np.float32(1.5)
        xh = (C.e2m1_decode(qx).reshape(M, -1, blk) * C.e4m3fn_decode(sfx)[..., None]).reshape(M, K) * float(gx)
        wh = (C.e2m1_decode(qw).reshape(N, -1, blk) * C.e4m3fn_decode(sfw)[..., None]).reshape(N, K) * float(gw)
    else:
        sfx = r.integers(120, 135, (M, K // blk)).astype(np.uint8)
        sfw = r.integers(120, 135, (N, K // blk)).astype(np.uint8)
        gx = gw = None
        xh = Q.mxfp4_dequant(qx, sfx)
        wh = Q.mxfp4_dequant(qw, sfw)
    y = _gpu_gemm(L, fmt, (qx, sfx, gx), (qw, sfw, gw), M, N, K)
    yr, b = G.matmul_ref(xh, wh)
    ok, worst = G.check(y, yr, b)
    assert ok.all(), f"{(~ok).sum()} bad, worst {worst:.3g}"
    assert np.count_nonzero(yr) > 0


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_fp4_end_to_end(fmt):
    L = lpq()
    M, N, K = 512, 256, 8192
    xb, wb, ox, ow, xh, wh = _operands(fmt, M, N, K, 4242)
    if fmt == "nvfp4":
        qx, sfx, gsx = L.quantize_nvfp4(dev_bf16(xb))
        qw, sfw, gsw = L.quantize_nvfp4(dev_bf16(wb))
        Y = L.gemm_scaled(L.FMT_NVFP4, L.GRAN_ROW, L.GRAN_ROW, qx, qw, sfx, sfw, M=M, N=N, K=K,
                          ga=gsx[1:], gb=gsw[1:])
    else:
        qx, sfx = L.quantize_mxfp4(dev_bf16(xb))
        qw, sfw = L.quantize_mxfp4(dev_bf16(wb))
        Y = L.gemm_scaled(L.FMT_MXFP4, L.GRAN_ROW, L.GRAN_ROW, qx, qw, sfx, sfw, M=M, N=N, K=K)
    torch.cuda.synchronize()
    yr, b = G.matmul_ref(xh, wh)
    ok, worst = G.check(bf16_to_f64(host(Y)), yr, b)
    assert ok.all(), worst
