"""GB300 (sm_103a) quantized-linear library: FP8 / INT8-SmoothQuant / NVFP4 /
MXFP4 activation and weight quantizers and tensor-core GEMMs with the scale
epilogue, behind the C ABI of include/lpq.h.

`lpq` is the ctypes binding (loads liblpq.so, built by `build`); importing
this package does not load the library.
"""
__all__ = ["lpq", "build"]
