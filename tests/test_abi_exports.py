"""The C-ABI library builds, loads without a GPU and exports every entry
point include/lpq.h declares; host-only functions behave."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


def _declared():
    src = open(os.path.join(ROOT, "include", "lpq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = set(re.findall(r"\b(lpq_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from w4a4_precision_gemm_gb300 import build
    build.build()
    from w4a4_precision_gemm_gb300 import lpq
    return lpq


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 20
    so = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in names if not hasattr(so, n)]
    assert not missing, missing
    assert set(lib.EXPORTS) <= set(names)


def test_host_only_functions(lib):
    L = lib
    assert L._lib().lpq_version().startswith(b"lpq")
    assert L._lib().lpq_status_string(L.LPQ_ERR_SHAPE)
    # scale layout: 128-row x 4-block tiles of 512 bytes
    assert L.lpq_sf_bytes(L.FMT_NVFP4, 1, 64) == 128 * 4
    assert L.lpq_sf_bytes(L.FMT_NVFP4, 130, 8192) == 256 * 512
    assert L.lpq_sf_bytes(L.FMT_MXFP4, 128, 8192) == 128 * 256
    assert L.lpq_sf_offset(L.FMT_NVFP4, 256, 128, 0, 0) == 0
    assert L.lpq_sf_offset(L.FMT_NVFP4, 256, 128, 1, 0) == 16
    assert L.lpq_sf_offset(L.FMT_NVFP4, 256, 128, 32, 0) == 4
    assert L.lpq_sf_offset(L.FMT_NVFP4, 256, 128, 0, 3) == 3
    assert L.lpq_sf_offset(L.FMT_NVFP4, 256, 128, 0, 4) == 512
    assert L.lpq_sf_offset(L.FMT_NVFP4, 256, 128, 128, 0) == 2 * 512
    assert L.lpq_sf_bytes(L.FMT_FP8, 128, 128) == 0
    # the offsets of one tile are a permutation of 0..511
    offs = sorted(L.lpq_sf_offset(L.FMT_MXFP4, 128, 128, r, k) for r in range(128) for k in range(4))
    assert offs == list(range(512))


def test_null_desc_rejected(lib):
    L = lib
    assert L._lib().lpq_gemm_scaled(None, None) == L.LPQ_ERR_NULL
    d = L.GemmDesc()
    assert L._lib().lpq_gemm_workspace_bytes(ctypes.byref(d)) == 0
    d.fmt, d.M, d.N, d.K = L.FMT_FP8, 16, 256, 256
    assert L._lib().lpq_gemm_scaled(ctypes.byref(d), None) == L.LPQ_ERR_NULL
