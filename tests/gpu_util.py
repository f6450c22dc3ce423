"""Helpers for the GPU parity tests: building/loading the library and moving
seeded inputs and oracle results between numpy and torch.  No arithmetic of
the method lives here."""
import numpy as np
import pytest
import torch


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def lpq():
    """The binding, with the library built in-tree for this machine."""
    need_gpu()
    from w4a4_precision_gemm_gb300 import build
    build.build()
    from w4a4_precision_gemm_gb300 import lpq as L
    return L


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> CUDA bf16 tensor (same bits)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """[R, K/2] bytes -> [R, K] codes, element 2i in the low nibble of byte i."""
    lo = packed & 0xF
    hi = packed >> 4
    return np.stack([lo, hi], axis=-1).reshape(packed.shape[0], -1).astype(np.uint8)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, np.uint8).reshape(codes.shape[0], -1, 2)
    return (c[..., 0] | (c[..., 1] << 4)).astype(np.uint8)


def sf_to_logical(L, fmt, sf_bytes: np.ndarray, rows: int, K: int, block: int) -> np.ndarray:
    """Scale-factor buffer in the library's layout -> [rows, K/block] via lpq_sf_offset."""
    kb = K // block
    r = np.arange(rows)[:, None]
    k = np.arange(kb)[None, :]
    kb4 = (kb + 3) // 4
    off = ((r // 128) * kb4 + k // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + k % 4
    # the closed form above must agree with the library's own index function
    for (rr, kk) in ((0, 0), (rows - 1, kb - 1), (rows // 2, kb // 2)):
        assert L.lpq_sf_offset(fmt, rows, K, rr, kk) == off[rr, kk]
    return sf_bytes[off]


def logical_to_sf(L, fmt, sf: np.ndarray, rows: int, K: int, block: int) -> np.ndarray:
    """[rows, K/block] scale codes -> a zero-padded buffer in the library's layout."""
    out = np.zeros(L.lpq_sf_bytes(fmt, rows, K), np.uint8)
    kb = K // block
    r = np.arange(rows)[:, None]
    k = np.arange(kb)[None, :]
    kb4 = (kb + 3) // 4
    off = ((r // 128) * kb4 + k // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + k % 4
    out[off] = sf
    return out
