"""lpq_gemm_scaled_noalloc, the GEMM entry point that allocates nothing.

It serves callers that cannot allocate device memory (a plugin whose host
runtime owns all device memory, or a path where cudaMalloc's implicit
synchronisation is not acceptable): its split-K scratch is an array inside the
library.  Checked here through the C ABI against lpq_gemm_scaled (given a
workspace of lpq_gemm_workspace_bytes) on two calls in a row, within the GEMM
tolerance of the other tests.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from oracle import quant as Q
from oracle import gemm as G
from gpu_util import lpq, dev, host, bf16_to_f64

pytestmark = pytest.mark.gpu


def _noalloc(L):
    f = L._lib().lpq_gemm_scaled_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(L.GemmDesc), ctypes.c_void_p]
    return f


def _problem(M, N, K, seed):
    xb = synth.activations(M, K, seed, n_outlier=max(1, K // 1000), lo=50, hi=500)
    wb = synth.weights(N, K, seed + 1)
    qx, sx = Q.fp8_per_row(synth.f32_from_bf16_bits(xb))
    qw, sw = Q.fp8_per_row(synth.f32_from_bf16_bits(wb))
    _, absum = G.matmul_ref(Q.fp8_dequant(qx, sx[:, None]), Q.fp8_dequant(qw, sw[:, None]))
    return dev(qx), dev(sx), dev(qw), dev(sw), absum


def test_noalloc_matches_gemm_scaled_on_two_calls():
    L = lpq()
    f = _noalloc(L)
    # different problems back to back: the first two need the built-in
    # scratch (153 and 156 output tiles, just over one wave of CTAs: the
    # leftover tiles are split along K and their partial sums go through the
    # shared array), the others use a cluster split or whole tiles
    for (M, N, K, seed) in ((1152, 4352, 256, 13), (256, 19968, 1024, 14), (300, 512, 1024, 15),
                            (16, 4096, 4096, 11), (1, 6144, 4096, 12)):
        A, sa, B, sb, absum = _problem(M, N, K, seed)
        Y_ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        ws = L.workspace_for(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, M, N, K)
        L.lpq_gemm_scaled(L.make_desc(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, A, B, sa, sb, Y_ref, M=M, N=N, K=K,
                                      workspace=ws))
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        d = L.make_desc(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, A, B, sa, sb, Y, M=M, N=N, K=K)
        st = f(ctypes.byref(d), L._stream(None))
        assert st == L.LPQ_OK, L._lib().lpq_status_string(st)
        torch.cuda.synchronize()
        y_ref = bf16_to_f64(host(Y_ref))
        y = bf16_to_f64(host(Y))
        tol = G.tolerance(y_ref, absum)
        assert np.all(np.abs(y - y_ref) <= tol), float(np.max(np.abs(y - y_ref) / tol))
    assert L.lpq_read_error_word() == 0


def test_noalloc_rejects_what_does_not_fit():
    L = lpq()
    f = _noalloc(L)
    lib = L._lib()
    limit = 16 << 20
    # a format it does not cover
    d = L.GemmDesc()
    d.fmt = L.FMT_INT8
    assert f(ctypes.byref(d), L._stream(None)) == L.LPQ_ERR_UNSUPPORTED
    for (M, N, K) in ((256, 28672, 4096), (64, 4096, 14336), (256, 4096, 14336)):
        probe = L.GemmDesc()
        probe.fmt, probe.a_gran, probe.b_gran, probe.M, probe.N, probe.K = L.FMT_FP8, 0, 0, M, N, K
        need = L.lpq_gemm_workspace_bytes(probe)
        if need <= limit:
            continue
        A = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
        B = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
        s1 = torch.ones(M, dtype=torch.float32, device="cuda")
        s2 = torch.ones(N, dtype=torch.float32, device="cuda")
        Y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
        d = L.make_desc(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, A, B, s1, s2, Y, M=M, N=N, K=K)
        assert f(ctypes.byref(d), L._stream(None)) == L.LPQ_ERR_WORKSPACE
        torch.cuda.synchronize()
        assert not host(Y).any()          # nothing was enqueued
