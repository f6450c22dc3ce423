"""Thin ctypes binding of liblpq.so (the C ABI in include/lpq.h).

Functions named `lpq_*` mirror the C entry points one to one: they take torch
tensors (device memory allocated by PyTorch), pass their data pointers, sizes
and the current CUDA stream, and raise `LpqError` on a non-OK status.  Every
step of the computation runs in the library's CUDA kernels; nothing here
computes.  The unprefixed helpers (`quantize_act_fp8`, `gemm_scaled`, ...)
only allocate the output tensors with torch and call the `lpq_*` function.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import c_int, c_int64, c_size_t, c_void_p, c_float, c_uint32, c_uint64, c_char_p, POINTER

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblpq.so")

# enums (include/lpq.h)
LPQ_OK, LPQ_ERR_NULL, LPQ_ERR_SHAPE, LPQ_ERR_ALIGN, LPQ_ERR_UNSUPPORTED, LPQ_ERR_CUDA, LPQ_ERR_WORKSPACE = range(7)
GRAN_ROW, GRAN_BLOCK_1x128, GRAN_BLOCK_128x128, GRAN_TENSOR_STATIC = range(4)
FMT_FP8, FMT_INT8, FMT_NVFP4, FMT_MXFP4 = range(4)
GEMM_B_STATIC = 1
GEMM_A_BF16 = 2
GEMM_B_INT8_PLANES = 4

EXPORTS = (
    "lpq_status_string", "lpq_last_cuda_error", "lpq_read_error_word", "lpq_clear_error_word",
    "lpq_version", "lpq_launch_count", "lpq_reset_launch_count",
    "lpq_act_absmax_update", "lpq_smooth_calibrate",
    "lpq_quantize_act_fp8", "lpq_quantize_weight_fp8", "lpq_quantize_act_int8", "lpq_quantize_weight_int8",
    "lpq_quantize_act_nvfp4", "lpq_quantize_weight_nvfp4", "lpq_quantize_act_mxfp4", "lpq_quantize_weight_mxfp4",
    "lpq_sf_bytes", "lpq_sf_offset", "lpq_gemm_workspace_bytes", "lpq_gemm_scaled", "lpq_int8_weight_planes",
    "lpq_selftest_bounded_wait",
)


class LpqError(RuntimeError):
    def __init__(self, status: int, fn: str):
        msg = _lib().lpq_status_string(status).decode() if _LIB is not None else str(status)
        if status == LPQ_ERR_CUDA:
            msg += f" (cudaError {_lib().lpq_last_cuda_error()})"
        super().__init__(f"{fn}: {msg}")
        self.status = status


class GemmDesc(ctypes.Structure):
    _fields_ = [
        ("fmt", c_int), ("a_gran", c_int), ("b_gran", c_int),
        ("M", c_int64), ("N", c_int64), ("K", c_int64),
        ("A", c_void_p), ("lda", c_int64),
        ("B", c_void_p), ("ldb", c_int64),
        ("sa", c_void_p), ("sb", c_void_p),
        ("ga", c_void_p), ("gb", c_void_p),
        ("Y", c_void_p), ("ldy", c_int64),
        ("workspace", c_void_p), ("workspace_bytes", c_size_t),
        ("flags", c_uint32),
    ]


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first (python -m w4a4_precision_gemm_gb300.build); "
                "there is no fallback implementation")
        L = ctypes.CDLL(LIB_PATH)
        S, P, I64 = c_int, c_void_p, c_int64
        sigs = {
            "lpq_status_string": (c_char_p, [c_int]),
            "lpq_last_cuda_error": (c_int, []),
            "lpq_read_error_word": (S, [POINTER(c_uint32)]),
            "lpq_clear_error_word": (S, []),
            "lpq_version": (c_char_p, []),
            "lpq_launch_count": (c_uint64, []),
            "lpq_reset_launch_count": (None, []),
            "lpq_act_absmax_update": (S, [P, I64, I64, I64, P, P]),
            "lpq_smooth_calibrate": (S, [P, P, I64, I64, I64, c_float, P, P]),
            "lpq_quantize_act_fp8": (S, [P, I64, I64, I64, c_int, P, P, P]),
            "lpq_quantize_weight_fp8": (S, [P, I64, I64, I64, c_int, P, P, P]),
            "lpq_quantize_act_int8": (S, [P, I64, I64, I64, P, P, P, P]),
            "lpq_quantize_weight_int8": (S, [P, I64, I64, I64, P, P, P, P]),
            "lpq_int8_weight_planes": (S, [P, I64, I64, I64, P, P]),
            "lpq_selftest_bounded_wait": (S, [ctypes.c_uint64, P]),
            "lpq_quantize_act_nvfp4": (S, [P, I64, I64, I64, P, P, P, P]),
            "lpq_quantize_weight_nvfp4": (S, [P, I64, I64, I64, P, P, P, P]),
            "lpq_quantize_act_mxfp4": (S, [P, I64, I64, I64, P, P, P]),
            "lpq_quantize_weight_mxfp4": (S, [P, I64, I64, I64, P, P, P]),
            "lpq_sf_bytes": (c_size_t, [c_int, I64, I64]),
            "lpq_sf_offset": (c_size_t, [c_int, I64, I64, I64, I64]),
            "lpq_gemm_workspace_bytes": (c_size_t, [POINTER(GemmDesc)]),
            "lpq_gemm_scaled": (S, [POINTER(GemmDesc), P]),
        }
        for name, (res, args) in sigs.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def library_path() -> str:
    return LIB_PATH


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, fn):
    if status != LPQ_OK:
        raise LpqError(status, fn)


def _bf16_2d(X, name):
    if X.dtype != torch.bfloat16 or X.dim() != 2 or X.stride(1) != 1 or not X.is_cuda:
        raise ValueError(f"{name}: expected a CUDA bf16 matrix with unit column stride")
    return X.shape[0], X.shape[1], X.stride(0)


# ---------------------------------------------------------------- C names --
def lpq_act_absmax_update(X, chan_amax, stream=None):
    M, K, ld = _bf16_2d(X, "X")
    _check(_lib().lpq_act_absmax_update(_ptr(X), M, K, ld, _ptr(chan_amax), _stream(stream)), "lpq_act_absmax_update")


def lpq_smooth_calibrate(chan_amax, W, alpha, s, stream=None):
    N, K, ld = _bf16_2d(W, "W")
    _check(_lib().lpq_smooth_calibrate(_ptr(chan_amax), _ptr(W), N, K, ld, float(alpha), _ptr(s), _stream(stream)),
           "lpq_smooth_calibrate")


def lpq_quantize_act_fp8(X, gran, Xq, sx, stream=None):
    M, K, ld = _bf16_2d(X, "X")
    _check(_lib().lpq_quantize_act_fp8(_ptr(X), M, K, ld, int(gran), _ptr(Xq), _ptr(sx), _stream(stream)),
           "lpq_quantize_act_fp8")


def lpq_quantize_weight_fp8(W, gran, Wq, sw, stream=None):
    N, K, ld = _bf16_2d(W, "W")
    _check(_lib().lpq_quantize_weight_fp8(_ptr(W), N, K, ld, int(gran), _ptr(Wq), _ptr(sw), _stream(stream)),
           "lpq_quantize_weight_fp8")


def lpq_quantize_act_int8(X, smooth, Xq, sx, stream=None):
    M, K, ld = _bf16_2d(X, "X")
    _check(_lib().lpq_quantize_act_int8(_ptr(X), M, K, ld, _ptr(smooth), _ptr(Xq), _ptr(sx), _stream(stream)),
           "lpq_quantize_act_int8")


def lpq_quantize_weight_int8(W, smooth, Wq, sw, stream=None):
    N, K, ld = _bf16_2d(W, "W")
    _check(_lib().lpq_quantize_weight_int8(_ptr(W), N, K, ld, _ptr(smooth), _ptr(Wq), _ptr(sw), _stream(stream)),
           "lpq_quantize_weight_int8")


def lpq_int8_weight_planes(Wq, planes, stream=None):
    N, K = Wq.shape
    _check(_lib().lpq_int8_weight_planes(_ptr(Wq), N, K, int(Wq.stride(0)), _ptr(planes), _stream(stream)),
           "lpq_int8_weight_planes")


def lpq_quantize_act_nvfp4(X, Xq, sf, gs, stream=None):
    M, K, ld = _bf16_2d(X, "X")
    _check(_lib().lpq_quantize_act_nvfp4(_ptr(X), M, K, ld, _ptr(Xq), _ptr(sf), _ptr(gs), _stream(stream)),
           "lpq_quantize_act_nvfp4")


def lpq_quantize_weight_nvfp4(W, Wq, sf, gs, stream=None):
    N, K, ld = _bf16_2d(W, "W")
    _check(_lib().lpq_quantize_weight_nvfp4(_ptr(W), N, K, ld, _ptr(Wq), _ptr(sf), _ptr(gs), _stream(stream)),
           "lpq_quantize_weight_nvfp4")


def lpq_quantize_act_mxfp4(X, Xq, sf, stream=None):
    M, K, ld = _bf16_2d(X, "X")
    _check(_lib().lpq_quantize_act_mxfp4(_ptr(X), M, K, ld, _ptr(Xq), _ptr(sf), _stream(stream)),
           "lpq_quantize_act_mxfp4")


def lpq_quantize_weight_mxfp4(W, Wq, sf, stream=None):
    N, K, ld = _bf16_2d(W, "W")
    _check(_lib().lpq_quantize_weight_mxfp4(_ptr(W), N, K, ld, _ptr(Wq), _ptr(sf), _stream(stream)),
           "lpq_quantize_weight_mxfp4")


def lpq_sf_bytes(fmt, rows, K):
    return int(_lib().lpq_sf_bytes(int(fmt), int(rows), int(K)))


def lpq_sf_offset(fmt, rows, K, r, kb):
    return int(_lib().lpq_sf_offset(int(fmt), int(rows), int(K), int(r), int(kb)))


def make_desc(fmt, a_gran, b_gran, A, B, sa, sb, Y, *, M, N, K, lda=None, ldb=None, ga=None, gb=None,
              workspace=None, flags=0):
    d = GemmDesc()
    d.fmt, d.a_gran, d.b_gran = int(fmt), int(a_gran), int(b_gran)
    d.M, d.N, d.K = int(M), int(N), int(K)
    d.A, d.B = A.data_ptr(), B.data_ptr()
    d.lda = int(lda if lda is not None else K)
    d.ldb = int(ldb if ldb is not None else K)
    d.sa = None if sa is None else sa.data_ptr()
    d.sb = None if sb is None else sb.data_ptr()
    d.ga = None if ga is None else ga.data_ptr()
    d.gb = None if gb is None else gb.data_ptr()
    d.Y, d.ldy = Y.data_ptr(), int(Y.stride(0))
    if workspace is not None:
        d.workspace, d.workspace_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    d.flags = int(flags)
    # the descriptor holds raw device pointers: keep the tensors alive with it
    d._tensors = (A, B, sa, sb, ga, gb, Y, workspace)
    return d


def lpq_gemm_workspace_bytes(desc):
    return int(_lib().lpq_gemm_workspace_bytes(ctypes.byref(desc)))


def lpq_gemm_scaled(desc, stream=None):
    _check(_lib().lpq_gemm_scaled(ctypes.byref(desc), _stream(stream)), "lpq_gemm_scaled")


LPQ_SELFTEST_WAIT_CODE = 0x0F0F


def lpq_selftest_bounded_wait(limit_ns, stream=None):
    _check(_lib().lpq_selftest_bounded_wait(int(limit_ns), _stream(stream)), "lpq_selftest_bounded_wait")


def lpq_read_error_word():
    v = c_uint32(0)
    _check(_lib().lpq_read_error_word(ctypes.byref(v)), "lpq_read_error_word")
    return int(v.value)


def lpq_clear_error_word():
    _check(_lib().lpq_clear_error_word(), "lpq_clear_error_word")


def lpq_launch_count():
    return int(_lib().lpq_launch_count())


def lpq_reset_launch_count():
    _lib().lpq_reset_launch_count()


# ------------------------------------------------- allocating conveniences --
def _empty(shape, dtype, like):
    return torch.empty(shape, dtype=dtype, device=like.device)


def quantize_act_fp8(X, gran=GRAN_ROW, static_scale=None, stream=None):
    M, K = X.shape
    Xq = _empty((M, K), torch.uint8, X)
    if gran == GRAN_ROW:
        sx = _empty((M,), torch.float32, X)
    elif gran == GRAN_BLOCK_1x128:
        sx = _empty((K // 128, M), torch.float32, X)
    else:
        sx = static_scale
    lpq_quantize_act_fp8(X, gran, Xq, sx, stream)
    return Xq, sx


def quantize_weight_fp8(W, gran=GRAN_ROW, stream=None):
    N, K = W.shape
    Wq = _empty((N, K), torch.uint8, W)
    sw = _empty((N,), torch.float32, W) if gran == GRAN_ROW else _empty(((N + 127) // 128, K // 128), torch.float32, W)
    lpq_quantize_weight_fp8(W, gran, Wq, sw, stream)
    return Wq, sw


def quantize_act_int8(X, smooth=None, stream=None):
    M, K = X.shape
    Xq = _empty((M, K), torch.int8, X)
    sx = _empty((M,), torch.float32, X)
    lpq_quantize_act_int8(X, smooth, Xq, sx, stream)
    return Xq, sx


def quantize_weight_int8(W, smooth=None, stream=None):
    N, K = W.shape
    Wq = _empty((N, K), torch.int8, W)
    sw = _empty((N,), torch.float32, W)
    lpq_quantize_weight_int8(W, smooth, Wq, sw, stream)
    return Wq, sw


def int8_weight_planes(Wq, stream=None):
    """[2, N, K] uint8: the E4M3 digit planes (high, low) of INT8 weight codes."""
    N, K = Wq.shape
    planes = _empty((2, N, K), torch.uint8, Wq)
    lpq_int8_weight_planes(Wq, planes, stream)
    return planes


def quantize_nvfp4(X, stream=None):
    R, K = X.shape
    q = _empty((R, K // 2), torch.uint8, X)
    sf = _empty((lpq_sf_bytes(FMT_NVFP4, R, K),), torch.uint8, X)
    gs = _empty((2,), torch.float32, X)
    lpq_quantize_act_nvfp4(X, q, sf, gs, stream)
    return q, sf, gs


def quantize_mxfp4(X, stream=None):
    R, K = X.shape
    q = _empty((R, K // 2), torch.uint8, X)
    sf = _empty((lpq_sf_bytes(FMT_MXFP4, R, K),), torch.uint8, X)
    lpq_quantize_act_mxfp4(X, q, sf, stream)
    return q, sf


def smooth_calibrate(chan_amax, W, alpha=0.5, stream=None):
    s = _empty((W.shape[1],), torch.float32, W)
    lpq_smooth_calibrate(chan_amax, W, alpha, s, stream)
    return s


def gemm_scaled(fmt, a_gran, b_gran, A, B, sa, sb, *, M, N, K, ga=None, gb=None, workspace=None, Y=None,
                stream=None, flags=0):
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    d = make_desc(fmt, a_gran, b_gran, A, B, sa, sb, Y, M=M, N=N, K=K, ga=ga, gb=gb, workspace=workspace,
                  flags=flags)
    lpq_gemm_scaled(d, stream)
    return Y


def workspace_for(fmt, a_gran, b_gran, M, N, K, device="cuda", flags=0):
    """A zero-filled workspace tensor of the size lpq_gemm_workspace_bytes reports."""
    d = GemmDesc()
    d.fmt, d.a_gran, d.b_gran, d.M, d.N, d.K = int(fmt), int(a_gran), int(b_gran), int(M), int(N), int(K)
    d.flags = int(flags)
    n = lpq_gemm_workspace_bytes(d)
    return torch.zeros((max(n, 16),), dtype=torch.uint8, device=device)
