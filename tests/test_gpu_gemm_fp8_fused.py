"""FP8 GEMM with the per-token activation quantization fused into the call
(LPQ_GEMM_A_BF16): A is the bf16 activation matrix, the scales come back in
sa.  Checked through the C ABI against the oracle (scales bit-exact, Y within
the GEMM tolerance) and against the two-call path (lpq_quantize_act_fp8 then
lpq_gemm_scaled), whose output it must reproduce bit for bit: same codes,
same scales, same tiling.

"FP8 and INT8 Inference", sections 6-9 (quantization inside the GEMM so the
8-bit activations make no extra round trip through memory); "FP8 and FP4
inference, SmoothQuant and activation quantization", section "Implementation
sketch" (the per-token rule)."""
import numpy as np
import pytest
import torch

import synth
from oracle import quant as Q
from oracle import gemm as G
from gpu_util import lpq, dev, dev_bf16, host, bf16_to_f64

pytestmark = pytest.mark.gpu

# (M, N, K): cluster K split (S = 8 / 4), whole tiles, K not a multiple of
# 128, a single K block, more tiles than CTA slots (CTAs with two tiles), and
# token counts above the fused limit (quantized through the workspace)
SHAPES = [(1, 4096, 4096), (16, 6144, 4096), (7, 4096, 14336), (5, 200, 336), (1, 128, 64), (3, 2048, 1024),
          (16, 40960, 256), (16, 28672, 512), (17, 1024, 512), (64, 4096, 4096), (300, 520, 4096)]


def _operands(M, N, K, seed):
    xb = synth.activations(M, K, seed, n_outlier=max(1, K // 1000), lo=50, hi=500)
    wb = synth.weights(N, K, seed + 1)
    qw, sw = Q.fp8_per_row(synth.f32_from_bf16_bits(wb))
    return xb, qw, sw


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("static_w", [False, True])
def test_fused_matches_two_calls_and_oracle(M, N, K, static_w):
    L = lpq()
    xb, qw, sw = _operands(M, N, K, 9100 + M + N + K)
    X, Wq, swd = dev_bf16(xb), dev(qw), dev(sw)
    flags = L.GEMM_A_BF16 | (L.GEMM_B_STATIC if static_w else 0)
    ws = L.workspace_for(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, M, N, K, flags=flags)
    sx_f = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    Y_f = L.gemm_scaled(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, X, Wq, sx_f, swd, M=M, N=N, K=K,
                        workspace=ws if M > 16 else None, flags=flags)
    # two calls: the standalone quantizer, then the GEMM on its codes
    Xq, sx_u = L.quantize_act_fp8(X, L.GRAN_ROW)
    ws_u = L.workspace_for(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, M, N, K)
    Y_u = L.gemm_scaled(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, Xq, Wq, sx_u, swd, M=M, N=N, K=K,
                        workspace=ws_u if M > 16 else None)
    torch.cuda.synchronize()
    assert L.lpq_read_error_word() == 0
    qx_o, sx_o = Q.fp8_per_row(synth.f32_from_bf16_bits(xb))
    assert np.array_equal(host(sx_f).view(np.uint32), sx_o.astype(np.float32).view(np.uint32))
    assert np.array_equal(host(Y_f), host(Y_u))
    yr, b = G.matmul_ref(Q.fp8_dequant(qx_o, sx_o[:, None]), Q.fp8_dequant(qw, sw[:, None]))
    ok, worst = G.check(bf16_to_f64(host(Y_f)), yr, b)
    assert ok.all(), f"{(~ok).sum()} outputs out of tolerance, worst ratio {worst:.3g}"


def test_fused_needs_workspace_above_the_fused_limit():
    L = lpq()
    M, N, K = 32, 256, 256
    xb, qw, sw = _operands(M, N, K, 9200)
    sx = torch.empty((M,), dtype=torch.float32, device="cuda")
    with pytest.raises(L.LpqError) as e:
        L.gemm_scaled(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, dev_bf16(xb), dev(qw), sx, dev(sw), M=M, N=N, K=K,
                      flags=L.GEMM_A_BF16)
    assert e.value.status == L.LPQ_ERR_WORKSPACE
    d = L.GemmDesc()
    d.fmt, d.a_gran, d.b_gran, d.M, d.N, d.K, d.flags = L.FMT_FP8, 0, 0, M, N, K, L.GEMM_A_BF16
    assert L.lpq_gemm_workspace_bytes(d) >= M * K
    d.M = 16
    assert L.lpq_gemm_workspace_bytes(d) == 0


def test_fused_rejected_by_noalloc_and_other_formats():
    import ctypes
    L = lpq()
    f = L._lib().lpq_gemm_scaled_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(L.GemmDesc), ctypes.c_void_p]
    M, N, K = 4, 256, 256
    xb, qw, sw = _operands(M, N, K, 9300)
    sx = torch.empty((M,), dtype=torch.float32, device="cuda")
    Y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    d = L.make_desc(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, dev_bf16(xb), dev(qw), sx, dev(sw), Y, M=M, N=N, K=K,
                    flags=L.GEMM_A_BF16)
    assert f(ctypes.byref(d), L._stream(None)) == L.LPQ_ERR_UNSUPPORTED
    d2 = L.make_desc(L.FMT_FP8, L.GRAN_TENSOR_STATIC, L.GRAN_ROW, dev_bf16(xb), dev(qw), sx, dev(sw), Y, M=M, N=N,
                     K=K, flags=L.GEMM_A_BF16)
    with pytest.raises(L.LpqError):
        L.lpq_gemm_scaled(d2)
    torch.cuda.synchronize()
    assert not host(Y).any()
