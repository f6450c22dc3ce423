"""Full-size parity: every workload's largest shapes, quantized and multiplied
on the GPU in the launch configuration the benchmark times (same flags, same
workspace), checked on sampled outputs that the oracle computes row by row.

Per sampled activation row and weight row the oracle quantizes only that row
(per-token, 1x128, per-channel and MX scales are row-local; a 128x128 weight
block is quantized whole; the NVFP4 tensor scale comes from one extra row that
carries the full tensor's largest magnitude, which gives the oracle the same
max|x|).  Codes and scales of the sampled rows must match bit for bit, Y at the
sampled (row, column) pairs within the GEMM tolerance (INT8: bit for bit)."""
import numpy as np
import pytest
import torch

import synth
from synth import configs as CFG
from oracle import quant as Q
from oracle import gemm as G
from oracle import smooth as SM
from gpu_util import lpq, dev_bf16, host, bf16_to_f64, unpack_nibbles, sf_to_logical

pytestmark = pytest.mark.gpu


def _pick(n, k, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    idx = set([0, n - 1]) | set(g.choice(n, size=min(n, k), replace=False).tolist())
    return np.array(sorted(idx))


def _with_max_row(x_full, rows):
    """x_full[rows] plus one row holding the element of largest magnitude."""
    flat = np.argmax(np.abs(x_full))
    extra = np.zeros((1, x_full.shape[1]), np.float32)
    extra[0, 0] = x_full.reshape(-1)[flat]
    return np.concatenate([x_full[rows], extra], axis=0)


def _check_y(Y, rows, cols, yr, b):
    y = bf16_to_f64(host(Y[torch.as_tensor(rows, device="cuda")][:, torch.as_tensor(cols, device="cuda")]))
    ok, worst = G.check(y, yr, b)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} sampled outputs out of tolerance, worst {worst:.3g}"


@pytest.mark.parametrize("M", CFG.DECODE_FP8.Ms)
def test_decode_fp8_full_size(M):
    L = lpq()
    wl = CFG.DECODE_FP8
    for si, (K, N) in enumerate(wl.KNs):
        xb, wb = CFG.make_x(wl, M, K, salt=si), CFG.make_w(wl, N, K, salt=si)
        Wq, sw = L.quantize_weight_fp8(dev_bf16(wb), L.GRAN_ROW)
        Xq, sx = L.quantize_act_fp8(dev_bf16(xb), L.GRAN_ROW)
        ws = L.workspace_for(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, M, N, K)
        Y = L.gemm_scaled(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, Xq, Wq, sx, sw, M=M, N=N, K=K, workspace=ws,
                          flags=L.GEMM_B_STATIC)
        torch.cuda.synchronize()
        rows, cols = _pick(M, 6, 1 + si), _pick(N, 12, 2 + si)
        qx, sxo = Q.fp8_per_row(synth.f32_from_bf16_bits(xb[rows]))
        qw, swo = Q.fp8_per_row(synth.f32_from_bf16_bits(wb[cols]))
        assert np.array_equal(host(Xq)[rows], qx) and np.array_equal(host(sx)[rows], sxo)
        assert np.array_equal(host(Wq)[cols], qw) and np.array_equal(host(sw)[cols], swo)
        yr, b = G.matmul_ref(Q.fp8_dequant(qx, sxo[:, None]), Q.fp8_dequant(qw, swo[:, None]))
        _check_y(Y, rows, cols, yr, b)
    assert L.lpq_read_error_word() == 0


@pytest.mark.parametrize("K,N", [(4096, 28672), (14336, 4096)])
def test_prefill_fp8_block_full_size(K, N):
    from oracle import codecs as C
    L = lpq()
    wl = CFG.PREFILL_FP8_BLOCK
    M = max(wl.Ms)
    xb, wb = CFG.make_x(wl, M, K), CFG.make_w(wl, N, K)
    Xq, sx = L.quantize_act_fp8(dev_bf16(xb), L.GRAN_BLOCK_1x128)
    Wq, sw = L.quantize_weight_fp8(dev_bf16(wb), L.GRAN_BLOCK_128x128)
    Y = L.gemm_scaled(L.FMT_FP8, L.GRAN_BLOCK_1x128, L.GRAN_BLOCK_128x128, Xq, Wq, sx, sw, M=M, N=N, K=K)
    torch.cuda.synchronize()
    rows, cols = _pick(M, 6, 11), _pick(N, 12, 12)
    qx, sxo = Q.fp8_per_group_1x128(synth.f32_from_bf16_bits(xb[rows]))
    assert np.array_equal(host(Xq)[rows], qx) and np.array_equal(host(sx)[:, rows].T, sxo)
    # weight rows: quantize each sampled row's whole 128-row block
    wf = synth.f32_from_bf16_bits(wb)
    qw = np.empty((len(cols), K), np.uint8)
    swo = np.empty((len(cols), K // 128), np.float32)
    for r, j in enumerate(cols):
        blk = j // 128
        q_b, s_b = Q.fp8_per_block_128x128_ragged(wf[blk * 128:min(N, blk * 128 + 128)])
        qw[r], swo[r] = q_b[j - blk * 128], s_b[0]
        assert np.array_equal(host(sw)[blk], s_b[0])
    assert np.array_equal(host(Wq)[cols], qw)
    xh = (C.e4m3fn_decode(qx).reshape(len(rows), K // 128, 128) * sxo[..., None]).reshape(len(rows), K)
    wh = (C.e4m3fn_decode(qw).reshape(len(cols), K // 128, 128) * swo[..., None]).reshape(len(cols), K)
    yr, b = G.matmul_ref(xh, wh)
    _check_y(Y, rows, cols, yr, b)
    assert L.lpq_read_error_word() == 0


def test_int8_smoothquant_full_size():
    L = lpq()
    wl = CFG.INT8_SMOOTHQUANT
    M, (K, N) = max(wl.Ms), wl.KNs[-1]
    cal, xb, wb = CFG.make_calib(wl, K), CFG.make_x(wl, M, K), CFG.make_w(wl, N, K)
    amax = torch.zeros(K, dtype=torch.float32, device="cuda")
    L.lpq_act_absmax_update(dev_bf16(cal), amax)
    Wd = dev_bf16(wb)
    s = L.smooth_calibrate(amax, Wd, CFG.SMOOTH_ALPHA)
    Wq, sw = L.quantize_weight_int8(Wd, s)
    planes = L.int8_weight_planes(Wq)
    Xq, sx = L.quantize_act_int8(dev_bf16(xb), s)
    flags = L.GEMM_B_INT8_PLANES
    ws = L.workspace_for(L.FMT_INT8, L.GRAN_ROW, L.GRAN_ROW, M, N, K, flags=flags)
    Y = L.gemm_scaled(L.FMT_INT8, L.GRAN_ROW, L.GRAN_ROW, Xq, planes, sx, sw, M=M, N=N, K=K, workspace=ws,
                      flags=flags)
    torch.cuda.synchronize()
    so = SM.smooth_factors(SM.channel_absmax(synth.f32_from_bf16_bits(cal)), synth.f32_from_bf16_bits(wb),
                           CFG.SMOOTH_ALPHA)
    assert np.array_equal(host(s), so)
    rows, cols = _pick(M, 8, 21), _pick(N, 16, 22)
    qx, sxo = Q.int8_per_row(synth.f32_from_bf16_bits(xb[rows]), so)
    qw, swo = Q.int8_per_row(synth.f32_from_bf16_bits(wb[cols]), so, weight=True)
    assert np.array_equal(host(Xq)[rows], qx) and np.array_equal(host(sx)[rows], sxo)
    assert np.array_equal(host(Wq)[cols], qw) and np.array_equal(host(sw)[cols], swo)
    want = G.int8_epilogue_fp32(G.int8_exact(qx, qw), sxo, swo)
    got = host(Y[torch.as_tensor(rows, device="cuda")][:, torch.as_tensor(cols, device="cuda")])
    got = (np.asarray(got, np.uint16).astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(got, want)
    assert L.lpq_read_error_word() == 0


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_fp4_full_size(fmt):
    L = lpq()
    wl = CFG.NVFP4_W4A4 if fmt == "nvfp4" else CFG.MXFP4_W4A4
    M, (K, N) = max(wl.Ms), wl.KNs[-1]
    xb, wb = CFG.make_x(wl, M, K), CFG.make_w(wl, N, K)
    F = L.FMT_NVFP4 if fmt == "nvfp4" else L.FMT_MXFP4
    if fmt == "nvfp4":
        Xq, sfx, gx = L.quantize_nvfp4(dev_bf16(xb))
        Wq, sfw, gw = L.quantize_nvfp4(dev_bf16(wb))
        ga, gb = gx[1:], gw[1:]
    else:
        (Xq, sfx), (Wq, sfw) = L.quantize_mxfp4(dev_bf16(xb)), L.quantize_mxfp4(dev_bf16(wb))
        ga = gb = None
    ws = L.workspace_for(F, 0, 0, M, N, K)
    Y = L.gemm_scaled(F, 0, 0, Xq, Wq, sfx, sfw, M=M, N=N, K=K, ga=ga, gb=gb, workspace=ws)
    torch.cuda.synchronize()
    rows, cols = _pick(M, 6, 31), _pick(N, 12, 32)
    xf, wf = synth.f32_from_bf16_bits(xb), synth.f32_from_bf16_bits(wb)
    blk = 16 if fmt == "nvfp4" else 32
    if fmt == "nvfp4":
        qx, cx, _, gxo = Q.nvfp4(_with_max_row(xf, rows))
        qw, cw, _, gwo = Q.nvfp4(_with_max_row(wf, cols))
        qx, cx, qw, cw = qx[:-1], cx[:-1], qw[:-1], cw[:-1]
        assert host(gx)[1] == gxo and host(gw)[1] == gwo
        xh, wh = Q.nvfp4_dequant(qx, cx, gxo), Q.nvfp4_dequant(qw, cw, gwo)
    else:
        qx, cx = Q.mxfp4(xf[rows])
        qw, cw = Q.mxfp4(wf[cols])
        xh, wh = Q.mxfp4_dequant(qx, cx), Q.mxfp4_dequant(qw, cw)
    assert np.array_equal(unpack_nibbles(host(Xq)[rows]), qx)
    assert np.array_equal(unpack_nibbles(host(Wq)[cols]), qw)
    assert np.array_equal(sf_to_logical(L, F, host(sfx), M, K, blk)[rows], cx)
    assert np.array_equal(sf_to_logical(L, F, host(sfw), N, K, blk)[cols], cw)
    yr, b = G.matmul_ref(xh, wh)
    _check_y(Y, rows, cols, yr, b)
    assert L.lpq_read_error_word() == 0
