"""FP8 per-token x per-channel GEMM on the tensor cores vs the oracle's fp64
dequantized product (through the C ABI).

The GEMM's inputs are the oracle's own codes and scales (uploaded), so the
comparison isolates the GEMM; one end-to-end case runs the GPU quantizers
first (their codes are bit-exact with the oracle's, tested elsewhere).
Tolerance: |y - y_ref| <= 1e-3 * sum_k |x^_k w^_k| + 1 bf16 ulp of y_ref.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import codecs as C
from oracle import quant as Q
from oracle import gemm as G
from gpu_util import lpq, dev_bf16, dev, host, bf16_to_f64

pytestmark = pytest.mark.gpu


def _oracle_operands(M, N, K, seed):
    xb = synth.activations(M, K, seed, n_outlier=max(1, K // 1000), lo=50, hi=500)
    wb = synth.weights(N, K, seed + 1)
    qx, sx = Q.fp8_per_row(synth.f32_from_bf16_bits(xb))
    qw, sw = Q.fp8_per_row(synth.f32_from_bf16_bits(wb))
    return xb, wb, qx, sx, qw, sw


def _ref(qx, sx, qw, sw):
    y, b = G.matmul_ref(Q.fp8_dequant(qx, sx[:, None]), Q.fp8_dequant(qw, sw[:, None]))
    return y, b


def _run(L, qx, sx, qw, sw, M, N, K, workspace=False, static=False):
    A, B = dev(qx), dev(qw)
    sa, sb = dev(sx), dev(sw)
    ws = L.workspace_for(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, M, N, K) if workspace else None
    gran = L.GRAN_TENSOR_STATIC if static else L.GRAN_ROW
    Y = L.gemm_scaled(L.FMT_FP8, gran, L.GRAN_ROW, A, B, sa, sb, M=M, N=N, K=K, workspace=ws)
    torch.cuda.synchronize()
    return host(Y), ws


SHAPES = [
    (16, 256, 256),        # the tiny W8A8 configuration
    (1, 128, 128), (1, 4096, 4096), (5, 200, 336), (16, 6144, 4096), (64, 4096, 14336),
    (200, 1000, 1024), (256, 4096, 4096), (300, 520, 4096), (1000, 4096, 2048), (517, 384, 144),
    (130, 12288, 512), (256, 19968, 1024),   # 96 tiles (one partial wave) / one wave + 4 tiles: K-split tail
    (1152, 4352, 256),                       # 153 tiles: one wave, then fewer leftover K iterations than CTAs
]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("workspace", [False, True])
def test_fp8_rowscale_gemm(M, N, K, workspace):
    L = lpq()
    _, _, qx, sx, qw, sw = _oracle_operands(M, N, K, 1000 + M + N + K)
    y, ws = _run(L, qx, sx, qw, sw, M, N, K, workspace=workspace)
    yr, b = _ref(qx, sx, qw, sw)
    ok, worst = G.check(bf16_to_f64(y), yr, b)
    assert ok.all(), f"{(~ok).sum()} outputs out of tolerance, worst ratio {worst:.3g}"


def test_fp8_tail_split_is_deterministic():
    """153 output tiles (one wave of 152 CTAs and one tile more): with a
    workspace the leftover tile is split along K and its slices are added by a
    second kernel in a fixed order, so repeated calls give identical bits."""
    L = lpq()
    M, N, K = 1152, 4352, 256
    _, _, qx, sx, qw, sw = _oracle_operands(M, N, K, 77)
    ws = L.workspace_for(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, M, N, K)
    assert ws.numel() > 16, "expected a split tail for 153 tiles"
    yr, b = _ref(qx, sx, qw, sw)
    outs = []
    for _ in range(3):
        A, B = dev(qx), dev(qw)
        Y = L.gemm_scaled(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, A, B, dev(sx), dev(sw), M=M, N=N, K=K, workspace=ws)
        torch.cuda.synchronize()
        outs.append(host(Y))
        ok, worst = G.check(bf16_to_f64(outs[-1]), yr, b)
        assert ok.all(), worst
    assert all(np.array_equal(outs[0], o) for o in outs[1:])
    assert L.lpq_read_error_word() == 0


def test_fp8_static_activation_scale():
    L = lpq()
    M, N, K = 64, 256, 512
    xb = synth.activations(M, K, 5, n_outlier=1, lo=5, hi=6)
    wb = synth.weights(N, K, 6)
    s_static = np.float32(0.05)
    qx = Q.fp8_static(synth.f32_from_bf16_bits(xb), s_static)
    qw, sw = Q.fp8_per_row(synth.f32_from_bf16_bits(wb))
    sx = np.array([s_static], np.float32)
    y, _ = _run(L, qx, sx, qw, sw, M, N, K, static=True)
    yr, b = G.matmul_ref(C.e4m3fn_decode(qx) * float(s_static), Q.fp8_dequant(qw, sw[:, None]))
    ok, worst = G.check(bf16_to_f64(y), yr, b)
    assert ok.all(), worst


def test_fp8_gemm_hand_built_codes():
    """One-hot and max codes: each output is a single product 448 * 448 * s_x * s_w,
    or a K-long sum of max codes; negative codes and zero rows included."""
    L = lpq()
    M, N, K = 130, 144, 256
    qx = np.zeros((M, K), np.uint8)
    qw = np.zeros((N, K), np.uint8)
    for m in range(M):
        qx[m, (7 * m) % K] = 0x7E if m % 2 else 0xFE
    for n in range(N):
        qw[n, (7 * n) % K] = 0x7E
    qw[5, :] = 0x7E                       # a row of max codes
    qx[129, :] = 0x01                     # smallest subnormal codes
    sx = np.linspace(0.5, 2.0, M).astype(np.float32)
    sw = np.linspace(1.0, 3.0, N).astype(np.float32) / 448
    y, _ = _run(L, qx, sx, qw, sw, M, N, K)
    yr, b = _ref(qx, sx, qw, sw)
    ok, worst = G.check(bf16_to_f64(y), yr, b)
    assert ok.all(), worst
    # a one-hot pair that meets gives exactly +-448*448*sx*sw (up to the bf16 rounding)
    m = 3
    n = 3
    assert abs(bf16_to_f64(y)[m, n] - 448.0 * 448.0 * sx[m] * sw[n]) <= C.bf16_ulp(yr[m, n])


def test_fp8_end_to_end_quantize_then_gemm():
    L = lpq()
    w = synth.configs.TINY_FP8
    M, (K, N) = 16, (256, 256)
    xb = synth.configs.make_x(w, M, K)
    wb = synth.configs.make_w(w, N, K)
    qx, sx = L.quantize_act_fp8(dev_bf16(xb), L.GRAN_ROW)
    qw, sw = L.quantize_weight_fp8(dev_bf16(wb), L.GRAN_ROW)
    Y = L.gemm_scaled(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, qx, qw, sx, sw, M=M, N=N, K=K)
    torch.cuda.synchronize()
    qxo, sxo = Q.fp8_per_row(synth.f32_from_bf16_bits(xb))
    qwo, swo = Q.fp8_per_row(synth.f32_from_bf16_bits(wb))
    yr, b = _ref(qxo, sxo, qwo, swo)
    ok, worst = G.check(bf16_to_f64(host(Y)), yr, b)
    assert ok.all(), worst


@pytest.mark.parametrize("M,N,K", [(1, 28672, 4096), (16, 4096, 14336), (256, 6144, 4096)])
def test_fp8_static_weights_flag(M, N, K):
    """LPQ_GEMM_B_STATIC lets the GEMM stream its weights while the activation
    quantizer launched just before it is still running; results must be
    identical to the unflagged call and within tolerance of the oracle."""
    L = lpq()
    xb = synth.activations(M, K, 900 + M, n_outlier=max(1, K // 1000), lo=50, hi=500)
    wb = synth.weights(N, K, 901)
    Wq, sw = L.quantize_weight_fp8(dev_bf16(wb), L.GRAN_ROW)
    X = dev_bf16(xb)
    ws = L.workspace_for(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, M, N, K)
    outs = []
    for flags in (0, L.GEMM_B_STATIC, L.GEMM_B_STATIC):
        qx, sx = L.quantize_act_fp8(X, L.GRAN_ROW)
        outs.append(L.gemm_scaled(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, qx, Wq, sx, sw, M=M, N=N, K=K,
                                  workspace=ws, flags=flags))
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    qxo, sxo = Q.fp8_per_row(synth.f32_from_bf16_bits(xb))
    qwo, swo = Q.fp8_per_row(synth.f32_from_bf16_bits(wb))
    yr, b = _ref(qxo, sxo, qwo, swo)
    ok, worst = G.check(bf16_to_f64(host(outs[1])), yr, b)
    assert ok.all(), worst


def test_fp8_activations_larger_than_l2():
    """69 MB of activation codes and 4 MB of weights: weight-column-fastest
    tile order.  A sample of rows against the oracle."""
    L = lpq()
    M, N, K = 8448, 512, 8192
    xb = synth.activations(M, K, 7200, n_outlier=8, lo=50, hi=500)
    wb = synth.weights(N, K, 7201)
    qx, sx = Q.fp8_per_row(synth.f32_from_bf16_bits(xb))
    qw, sw = Q.fp8_per_row(synth.f32_from_bf16_bits(wb))
    ws = L.workspace_for(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, M, N, K)
    Y = L.gemm_scaled(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, dev(qx), dev(qw), dev(sx), dev(sw), M=M, N=N, K=K,
                      workspace=ws)
    torch.cuda.synchronize()
    assert L.lpq_read_error_word() == 0
    rows = np.arange(0, M, 97)
    yr, b = _ref(qx[rows], sx[rows], qw, sw)
    ok, worst = G.check(bf16_to_f64(host(Y)[rows]), yr, b)
    assert ok.all(), worst
