"""Benchmark of the quantized-linear hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one pass of the hot path over one batch of synthetic input:
for every token count M and projection (K, N) of the workload, the dynamic
activation quantizer and the scaled GEMM (weights are quantized once, at load
time, before timing).  The default workload is Llama-8B-shaped FP8 W8A8
decode: M in {1, 16, 64, 256} x (K, N) in {(4096, 6144), (4096, 4096),
(4096, 28672), (14336, 4096)}; every weight copy streamed in a step is
distinct (no weight byte is read twice per step, 872 MB per step > L2).

Prints one JSON line (rank 0).  `value` is the whole step's GEMM TFLOP/s with
inputs resident in HBM; `e2e` is the same metric through the C ABI with the
activations copied from pinned host memory and Y copied back inside the timed
region; `roofline` is the dominant kernel's achieved HBM GB/s (or tensor
TFLOP/s) against the measured peak; `cpu_baseline` is the CPU oracle timed on
a bounded sample of the same workload.  `--impl reference` times that oracle
as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import configs as CFG  # noqa: E402


# -------------------------------------------------------- graph timing --
class GraphEvents:
    """Timing events that can live inside a CUDA graph: recorded with
    cudaEventRecordWithFlags(..., cudaEventRecordExternal), so that stream
    capture turns them into event-record nodes (torch's Event.record inside a
    capture only orders streams).  Uses the process's CUDA runtime."""

    def __init__(self):
        import ctypes
        self.ct = ctypes
        self.rt = None
        for name in ("libcudart.so.13", "libcudart.so"):
            try:
                self.rt = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if self.rt is None:
            raise RuntimeError("CUDA runtime library not found for graph timing events")
        self.rt.cudaEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
        self.rt.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        self.rt.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p, ctypes.c_void_p]
        self.rt.cudaEventDestroy.argtypes = [ctypes.c_void_p]
        self.events = []

    def new(self):
        e = self.ct.c_void_p()
        if self.rt.cudaEventCreate(self.ct.byref(e)) != 0:
            raise RuntimeError("cudaEventCreate failed")
        self.events.append(e)
        return e

    def record(self, ev, stream, external=True):
        # cudaEventRecordExternal (1) only inside a capture; a plain record otherwise
        r = self.rt.cudaEventRecordWithFlags(ev, self.ct.c_void_p(stream.cuda_stream), 1 if external else 0)
        if r != 0:
            raise RuntimeError(f"cudaEventRecordWithFlags failed ({r})")

    def elapsed_ms(self, a, b):
        f = self.ct.c_float()
        r = self.rt.cudaEventElapsedTime(self.ct.byref(f), a, b)
        if r != 0:
            raise RuntimeError(f"cudaEventElapsedTime failed ({r})")
        return f.value

    def close(self):
        for e in self.events:
            self.rt.cudaEventDestroy(e)
        self.events = []


# ------------------------------------------------------------------ peaks --
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


# nominal dense ratios to bf16 (2.25 PF): FP8 4.5 -> 2x, FP4 13.5 -> 6x
NOMINAL_RATIO = {"fp8": 2.0, "fp4": 6.0, "bf16": 1.0, "int8": 2.0}


def measure_int8_library_peak(torch, n=8192, reps=10):
    """TOPS of the vendor INT8 GEMM (torch._int_mm -> cuBLASLt) at n^3, best of reps."""
    a = torch.randint(-127, 128, (n, n), dtype=torch.int8, device="cuda")
    b = torch.randint(-127, 128, (n, n), dtype=torch.int8, device="cuda").t()
    for _ in range(3):
        torch._int_mm(a, b)
    torch.cuda.synchronize()
    best = 1e9
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(reps):
        e0.record()
        torch._int_mm(a, b)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    return 2.0 * n ** 3 / (best * 1e-3) / 1e12


# --------------------------------------------------------------- traffic --
TRAFFIC_FILES = {"gemm_fp8": "gemm_fp8_decode_traffic.txt", "gemm_fp4": "gemm_fp4_nvfp4_traffic.txt",
                 "gemm_fp8_block": "gemm_fp8_block_prefill_traffic.txt", "gemm_int8": "gemm_int8_traffic.txt"}
KERNEL_SOURCES = {"gemm_fp8": ["gemm_fp8.cu", "gemm_common.cuh", "ptx.cuh"],
                  "gemm_fp4": ["gemm_fp4.cu", "gemm_common.cuh", "ptx.cuh"],
                  "gemm_fp8_block": ["gemm_fp8_block.cu", "gemm_common.cuh", "ptx.cuh"],
                  "gemm_int8": ["gemm_int8_tc.cu", "gemm_common.cuh", "ptx.cuh"]}


def kernel_source_hash(kind: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kind, []):
        with open(os.path.join(ROOT, "w4a4_precision_gemm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kind: str):
    """DRAM bytes per launch of `kind` from the committed ncu summary, or
    None when there is none or the kernel's sources changed since it was taken."""
    name = TRAFFIC_FILES.get(kind)
    path = os.path.join(ROOT, "profiles", name) if name else None
    if not path or not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("source_sha256") != kernel_source_hash(kind):
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------- multi-process --
def max_over_ranks(x: float, dist, device) -> float:
    """The largest value of `x` over all ranks (the job is as slow as its
    slowest replica); `x` itself without a process group."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Work of all replicas per second (weak scaling: every rank runs the
    same step on its own GPU)."""
    return work_per_rank_step * world / (ms_per_step * 1e-3)


# ----------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# -------------------------------------------------------------- workloads --
class Workload:
    """Holds device buffers and the list of launches of one step."""

    def __init__(self, name, L, torch, rank=0):
        self.name = name
        self.L = L
        self.torch = torch
        self.rank = rank
        self.calls = []       # list of dicts: kind, fn (launch), flops, bytes

    def dev_bf16(self, bits):
        t = self.torch
        return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(t.bfloat16).cuda()

    def arena(self, wl):
        """One device buffer (and its pinned host mirror) for all of a step's
        activations and one for all its outputs: the end-to-end step moves
        each with a single copy.  `input` / `output` hand out [rows, cols]
        views in call order (offsets stay 16-byte aligned: K, N % 8 == 0)."""
        t = self.torch
        n_in = sum(M * K for M in wl.Ms for K, _ in wl.KNs)
        n_out = sum(M * N for M in wl.Ms for _, N in wl.KNs)
        self.din = t.empty(n_in, dtype=t.bfloat16, device="cuda")
        self.dout = t.empty(n_out, dtype=t.bfloat16, device="cuda")
        self.hin = t.empty(n_in, dtype=t.bfloat16).pin_memory()
        self.hout = t.empty(n_out, dtype=t.bfloat16).pin_memory()
        self._oi = self._oo = 0
        self.dev_in, self.dev_out, self.host_in, self.host_out = [], [], [], []
        self.subset = False

    def input(self, bits):
        t = self.torch
        M, K = bits.shape
        h = self.hin[self._oi:self._oi + M * K].view(M, K)
        h.copy_(t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(t.bfloat16))
        d = self.din[self._oi:self._oi + M * K].view(M, K)
        d.copy_(h)
        self._oi += M * K
        self.host_in.append(h)
        self.dev_in.append(d)
        return d

    def output(self, M, N):
        h = self.hout[self._oo:self._oo + M * N].view(M, N)
        d = self.dout[self._oo:self._oo + M * N].view(M, N)
        self._oo += M * N
        self.host_out.append(h)
        self.dev_out.append(d)
        return d


def workload_config(name: str) -> dict:
    """The `config` object of a workload's JSON line (no device needed: the
    reference arm prints the same one)."""
    if name == "decode_fp8":
        wl = CFG.DECODE_FP8
        return {"workload": wl.name, "Ms": list(wl.Ms), "KNs": [list(x) for x in wl.KNs],
                "act": "fp8 e4m3 per-token dynamic", "weight": "fp8 e4m3 per-channel static",
                "l2": "inputs larger than L2: 872 MB of distinct FP8 weights streamed per step"}
    if name in ("nvfp4", "mxfp4"):
        wl = CFG.NVFP4_W4A4 if name == "nvfp4" else CFG.MXFP4_W4A4
        return {"workload": wl.name, "Ms": list(wl.Ms), "KNs": [list(x) for x in wl.KNs],
                "format": wl.fmt, "l2": "inputs larger than L2 for M=8192; M=512 weights 37-117 MB"}
    if name == "prefill_fp8_block":
        wl = CFG.PREFILL_FP8_BLOCK
        return {"workload": wl.name, "Ms": list(wl.Ms), "KNs": [list(x) for x in wl.KNs],
                "act": "fp8 e4m3 per 1x128 group, dynamic", "weight": "fp8 e4m3 per 128x128 block",
                "l2": "inputs larger than L2 (M=8192 activations 64-235 MB bf16; weights 17-117 MB fp8)"}
    if name == "int8_smoothquant":
        wl = CFG.INT8_SMOOTHQUANT
        return {"workload": wl.name, "Ms": list(wl.Ms), "KNs": [list(x) for x in wl.KNs],
                "alpha": CFG.SMOOTH_ALPHA, "calibration_tokens": CFG.INT8_CALIB_TOKENS,
                "l2": "inputs larger than L2 for M=4096 (W 16-117 MB int8, X 32 MB bf16)"}
    raise KeyError(name)


def build_decode_fp8(L, torch, wl=CFG.DECODE_FP8):
    """FP8 W8A8 decode: per-token act quant + the FP8 GEMM (swap-AB up to 64 tokens, cluster K split for few tiles)."""
    W = Workload(wl.name, L, torch)
    W.config = workload_config("decode_fp8")
    W.dominant = "gemm_fp8"
    W.dominant_bound = "hbm"
    W.arena(wl)
    for mi, M in enumerate(wl.Ms):
        for si, (K, N) in enumerate(wl.KNs):
            wb = CFG.make_w(wl, N, K, salt=si)              # same weights, one fp8 copy per M
            Wd = W.dev_bf16(wb)
            Wq, sw = L.quantize_weight_fp8(Wd, L.GRAN_ROW)
            del Wd
            xb = CFG.make_x(wl, M, K, salt=mi * 10 + si)
            Xd = W.input(xb)
            Xq = torch.empty((M, K), dtype=torch.uint8, device="cuda")
            sx = torch.empty((M,), dtype=torch.float32, device="cuda")
            Y = W.output(M, N)
            ws = L.workspace_for(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, M, N, K)
            desc = L.make_desc(L.FMT_FP8, L.GRAN_ROW, L.GRAN_ROW, Xq, Wq, sx, sw, Y, M=M, N=N, K=K, workspace=ws,
                               flags=L.GEMM_B_STATIC)   # weights quantized at load time
            W.keep = getattr(W, "keep", []) + [Wq, sw, ws]
            W.calls.append(dict(kind="quant_fp8_row", M=M, K=K, N=N,
                                fn=(lambda Xd=Xd, Xq=Xq, sx=sx: L.lpq_quantize_act_fp8(Xd, L.GRAN_ROW, Xq, sx)),
                                bytes=M * K * 2 + M * K + 4 * M, flops=0))
            W.calls.append(dict(kind="gemm_fp8", M=M, K=K, N=N, fn=(lambda d=desc: L.lpq_gemm_scaled(d)),
                                bytes=N * K + 4 * N + M * K + 4 * M + 2 * M * N, flops=2 * M * N * K))
    return W


def build_fp4(L, torch, wl):
    nv = wl.fmt == "nvfp4"
    W = Workload(wl.name, L, torch)
    W.config = workload_config(wl.fmt)
    W.dominant = "gemm_fp4"
    W.dominant_bound = "tensor"
    W.dominant_dtype = "fp4"
    W.arena(wl)
    F = L.FMT_NVFP4 if nv else L.FMT_MXFP4
    for mi, M in enumerate(wl.Ms):
        for si, (K, N) in enumerate(wl.KNs):
            Wd = W.dev_bf16(CFG.make_w(wl, N, K, salt=si))
            if nv:
                Wq, sfw, gsw = L.quantize_nvfp4(Wd)
            else:
                (Wq, sfw), gsw = L.quantize_mxfp4(Wd), None
            del Wd
            xb = CFG.make_x(wl, M, K, salt=mi * 10 + si)
            Xd = W.input(xb)
            Xq = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
            sfx = torch.empty((L.lpq_sf_bytes(F, M, K),), dtype=torch.uint8, device="cuda")
            gsx = torch.empty((2,), dtype=torch.float32, device="cuda")
            Y = W.output(M, N)
            ws = L.workspace_for(F, L.GRAN_ROW, L.GRAN_ROW, M, N, K)
            desc = L.make_desc(F, L.GRAN_ROW, L.GRAN_ROW, Xq, Wq, sfx, sfw, Y, M=M, N=N, K=K,
                               ga=gsx[1:] if nv else None, gb=gsw[1:] if nv else None, workspace=ws)
            W.keep = getattr(W, "keep", []) + [Wq, sfw, gsw, ws, gsx]
            if nv:
                qfn = (lambda Xd=Xd, Xq=Xq, sfx=sfx, gsx=gsx: L.lpq_quantize_act_nvfp4(Xd, Xq, sfx, gsx))
            else:
                qfn = (lambda Xd=Xd, Xq=Xq, sfx=sfx: L.lpq_quantize_act_mxfp4(Xd, Xq, sfx))
            blk = 16 if nv else 32
            W.calls.append(dict(kind="quant_" + wl.fmt, M=M, K=K, N=N, fn=qfn,
                                bytes=M * K * 2 + M * K // 2 + M * K // blk, flops=0))
            W.calls.append(dict(kind="gemm_fp4", M=M, K=K, N=N, fn=(lambda d=desc: L.lpq_gemm_scaled(d)),
                                bytes=(M + N) * K // 2 + (M + N) * K // blk + 2 * M * N, flops=2 * M * N * K))
    return W


def build_prefill_block(L, torch, wl=CFG.PREFILL_FP8_BLOCK):
    """FP8 prefill with 1x128 activation / 128x128 weight block scales."""
    W = Workload(wl.name, L, torch)
    W.config = workload_config("prefill_fp8_block")
    W.dominant = "gemm_fp8_block"
    W.dominant_bound = "tensor"
    W.dominant_dtype = "fp8"
    W.arena(wl)
    wq = {}
    for si, (K, N) in enumerate(wl.KNs):
        Wd = W.dev_bf16(CFG.make_w(wl, N, K, salt=si))
        wq[si] = L.quantize_weight_fp8(Wd, L.GRAN_BLOCK_128x128)
        del Wd
    for mi, M in enumerate(wl.Ms):
        for si, (K, N) in enumerate(wl.KNs):
            Wq, sw = wq[si]
            xb = CFG.make_x(wl, M, K, salt=mi * 10 + si)
            Xd = W.input(xb)
            Xq = torch.empty((M, K), dtype=torch.uint8, device="cuda")
            sx = torch.empty((K // 128, M), dtype=torch.float32, device="cuda")
            Y = W.output(M, N)
            desc = L.make_desc(L.FMT_FP8, L.GRAN_BLOCK_1x128, L.GRAN_BLOCK_128x128, Xq, Wq, sx, sw, Y, M=M, N=N, K=K)
            W.keep = getattr(W, "keep", []) + [desc, Wq, sw, Xq, sx, Y]
            W.calls.append(dict(kind="quant_fp8_1x128", M=M, K=K, N=N,
                                fn=(lambda Xd=Xd, Xq=Xq, sx=sx: L.lpq_quantize_act_fp8(Xd, L.GRAN_BLOCK_1x128, Xq, sx)),
                                bytes=M * K * 3 + 4 * M * K // 128, flops=0))
            W.calls.append(dict(kind="gemm_fp8_block", M=M, K=K, N=N, fn=(lambda d=desc: L.lpq_gemm_scaled(d)),
                                bytes=(M + N) * K + 2 * M * N, flops=2 * M * N * K))
    return W


def _int8_probe_desc(L, M, N, K, flags):
    d = L.GemmDesc()
    d.fmt, d.a_gran, d.b_gran, d.M, d.N, d.K, d.flags = L.FMT_INT8, L.GRAN_ROW, L.GRAN_ROW, M, N, K, flags
    return d


def build_int8(L, torch, wl=CFG.INT8_SMOOTHQUANT):
    """INT8 W8A8 with SmoothQuant: calibration, smoothed weight quantization
    and the weights' digit planes at load; per step the smoothed per-token
    quantizer and the INT8 GEMM (tensor cores, exact int32 result)."""
    W = Workload(wl.name, L, torch)
    W.config = workload_config("int8_smoothquant")
    W.dominant = "gemm_int8"
    W.dominant_bound = "tensor"
    W.dominant_dtype = "int8"
    W.arena(wl)
    K = wl.KNs[0][0]
    amax = torch.zeros(K, dtype=torch.float32, device="cuda")
    L.lpq_act_absmax_update(W.dev_bf16(CFG.make_calib(wl, K)), amax)
    wq = {}
    for si, (K, N) in enumerate(wl.KNs):
        Wd = W.dev_bf16(CFG.make_w(wl, N, K, salt=si))
        sm = L.smooth_calibrate(amax, Wd, CFG.SMOOTH_ALPHA)
        Wq, sw = L.quantize_weight_int8(Wd, sm)
        planes = L.int8_weight_planes(Wq)        # the tensor-core GEMM's digit planes, at load time too
        wq[si] = (planes, sw, sm)
        del Wd, Wq
    flags = L.GEMM_B_INT8_PLANES
    ws_bytes = max(L.lpq_gemm_workspace_bytes(_int8_probe_desc(L, M, N, K, flags))
                   for M in wl.Ms for (K, N) in wl.KNs)
    ws = torch.zeros((ws_bytes,), dtype=torch.uint8, device="cuda")   # shared: the calls run in order
    W.keep = [ws]
    for mi, M in enumerate(wl.Ms):
        for si, (K, N) in enumerate(wl.KNs):
            Wq, sw, sm = wq[si]
            xb = CFG.make_x(wl, M, K, salt=mi * 10 + si)
            Xd = W.input(xb)
            Xq = torch.empty((M, K), dtype=torch.int8, device="cuda")
            sx = torch.empty((M,), dtype=torch.float32, device="cuda")
            Y = W.output(M, N)
            desc = L.make_desc(L.FMT_INT8, L.GRAN_ROW, L.GRAN_ROW, Xq, Wq, sx, sw, Y, M=M, N=N, K=K, workspace=ws,
                               flags=flags)
            W.keep = getattr(W, "keep", []) + [desc, Wq, sw, sm, Xq, sx, Y]
            W.calls.append(dict(kind="quant_int8_smooth", M=M, K=K, N=N,
                                fn=(lambda Xd=Xd, Xq=Xq, sx=sx, sm=sm: L.lpq_quantize_act_int8(Xd, sm, Xq, sx)),
                                bytes=M * K * 3 + 4 * M, flops=0))
            W.calls.append(dict(kind="gemm_int8", M=M, K=K, N=N, fn=(lambda d=desc: L.lpq_gemm_scaled(d)),
                                bytes=(M + N) * K + 4 * (M + N) + 2 * M * N, flops=2 * M * N * K))
    return W


BUILDERS = {
    "decode_fp8": lambda L, t: build_decode_fp8(L, t),
    "prefill_fp8_block": lambda L, t: build_prefill_block(L, t),
    "int8_smoothquant": lambda L, t: build_int8(L, t),
    "nvfp4": lambda L, t: build_fp4(L, t, CFG.NVFP4_W4A4),
    "mxfp4": lambda L, t: build_fp4(L, t, CFG.MXFP4_W4A4),
}


# ------------------------------------------------------------ CPU oracle --
def oracle_sample(workload: str, budget_s: float = 15.0):
    """Time the CPU oracle on a bounded sample of the workload: every (M, K, N)
    GEMM of the step, restricted to its first `n_rows` output channels, with
    the activation quantizer on the full X.  Returns (TFLOP/s, description,
    threads)."""
    from oracle import quant as Q
    from oracle import gemm as G
    wl = {"decode_fp8": CFG.DECODE_FP8, "nvfp4": CFG.NVFP4_W4A4, "mxfp4": CFG.MXFP4_W4A4,
          "prefill_fp8_block": CFG.PREFILL_FP8_BLOCK, "int8_smoothquant": CFG.INT8_SMOOTHQUANT}[workload]
    n_rows = 64
    Ms = [m for m in wl.Ms if m <= 512] or [min(wl.Ms)]
    flops, t_total, done = 0, 0.0, 0
    for mi, M in enumerate(Ms):
        for si, (K, N) in enumerate(wl.KNs):
            xb = CFG.make_x(wl, M, K, salt=mi * 10 + si)
            wb = CFG.make_w(wl, n_rows, K, salt=si)
            x = synth.f32_from_bf16_bits(xb)
            w = synth.f32_from_bf16_bits(wb)
            if wl.fmt == "fp8_block":
                qw, sw = Q.fp8_per_block_128x128_ragged(w)      # load time, untimed
                t0 = time.perf_counter()
                qx, sx = Q.fp8_per_group_1x128(x)
                from oracle import codecs as Cd
                xh = (Cd.e4m3fn_decode(qx).reshape(M, K // 128, 128) * sx[..., None]).reshape(M, K)
                wh = (Cd.e4m3fn_decode(qw).reshape(n_rows, K // 128, 128) * sw[0][None, :, None]).reshape(n_rows, K)
                G.matmul_ref(xh, wh)
            elif wl.fmt == "int8":
                qw, sw = Q.int8_per_row(w, None, weight=True)
                t0 = time.perf_counter()
                qx, sx = Q.int8_per_row(x)
                G.int8_epilogue_fp32(G.int8_exact(qx, qw), sx, sw)
            elif wl.fmt == "fp8":
                qw, sw = Q.fp8_per_row(w)                       # load time, untimed
                t0 = time.perf_counter()
                qx, sx = Q.fp8_per_row(x)
                G.matmul_ref(Q.fp8_dequant(qx, sx[:, None]), Q.fp8_dequant(qw, sw[:, None]))
            elif wl.fmt == "nvfp4":
                qw, sfw, _, gw = Q.nvfp4(w)
                t0 = time.perf_counter()
                qx, sfx, _, gx = Q.nvfp4(x)
                G.matmul_ref(Q.nvfp4_dequant(qx, sfx, gx), Q.nvfp4_dequant(qw, sfw, gw))
            else:
                qw, sfw = Q.mxfp4(w)
                t0 = time.perf_counter()
                qx, sfx = Q.mxfp4(x)
                G.matmul_ref(Q.mxfp4_dequant(qx, sfx), Q.mxfp4_dequant(qw, sfw))
            t_total += time.perf_counter() - t0
            flops += 2 * M * n_rows * K
            done += 1
            if t_total > budget_s:
                break
        if t_total > budget_s:
            break
    desc = (f"{done} GEMMs of the step (M<=512) restricted to their first {n_rows} output channels, "
            f"activation quantizer on the full X; weights quantized untimed")
    threads = os.cpu_count()
    return flops / t_total / 1e12, desc, threads


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    vals = []
    desc, threads = "", os.cpu_count()
    for _ in range(args.warmup):
        oracle_sample(args.workload, budget_s=2.0)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, desc, threads = oracle_sample(args.workload, budget_s=max(2.0, 60.0 / max(1, args.steps)))
        vals.append(v)
    el = time.perf_counter() - t0
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": dict(workload_config(args.workload), parallelism=f"replicas x{max(1, args.gpus)}"),
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


METRIC = "scaled-GEMM TFLOP/s & % of GB300 FP8/FP4 peak; quantizer GB/s & % of HBM"


# ------------------------------------------------------------------- main --
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode_fp8", choices=sorted(BUILDERS))
    ap.add_argument("--impl", default="lpq", choices=["lpq", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="launch every call from Python instead of a CUDA graph")
    ap.add_argument("--only", default="", help="keep only these M:N pairs, e.g. 1:28672,16:4096 (profiling)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        return run_reference(args)

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from w4a4_precision_gemm_gb300 import build as B
    B.build()
    from w4a4_precision_gemm_gb300 import lpq as L

    W = BUILDERS[args.workload](L, torch)
    if args.only:
        keep = {tuple(int(v) for v in p.split(":")) for p in args.only.split(",")}
        idx = [i for i in range(0, len(W.calls), 2) if (W.calls[i]["M"], W.calls[i]["N"]) in keep]
        W.calls = [W.calls[j] for i in idx for j in (i, i + 1)]
        W.dev_in = [W.dev_in[i // 2] for i in idx]
        W.dev_out = [W.dev_out[i // 2] for i in idx]
        W.host_in = [W.host_in[i // 2] for i in idx]
        W.host_out = [W.host_out[i // 2] for i in idx]
        W.subset = True
        W.config["only"] = args.only
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step():
        for c in W.calls:
            c["fn"]()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- CUDA graphs (the library's calls are plain stream work, so stream
    # capture records them as kernel nodes; consecutive kernels overlap their
    # launch through programmatic dependent launch):
    #   g_run  the K steps exactly as timed (no extra nodes),
    #   g_dom  the K steps' launches of the dominant kernel only (its average
    #          launch duration for the roofline),
    #   g_ins  the K steps with a timing-event node around every launch (the
    #          per-kernel table; the events themselves serialise the kernels).
    GE = GraphEvents()
    evs = [[(GE.new(), GE.new()) for _ in W.calls] for _ in range(args.steps)]
    cap = torch.cuda.Stream()

    def run_steps():
        for _ in range(args.steps):
            step()

    def dom_steps():
        for _ in range(args.steps):
            for c in W.calls:
                if c["kind"] == W.dominant:
                    c["fn"]()

    def ins_steps(on, external=True):
        for s_ in range(args.steps):
            for i, c in enumerate(W.calls):
                GE.record(evs[s_][i][0], on, external)
                c["fn"]()
                GE.record(evs[s_][i][1], on, external)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                fn()
        stream.wait_stream(cap)
        g.replay()                      # one untimed replay of each graph
        torch.cuda.synchronize()
        return g

    g_run = g_dom = g_ins = None
    if not args.eager:
        try:
            L.lpq_reset_launch_count()
            g_run = capture(run_steps)
            launches = L.lpq_launch_count()   # library kernels in the timed graph
            g_dom = capture(dom_steps)
            g_ins = capture(lambda: ins_steps(cap))
        except Exception as e:  # capture unavailable: time the same calls eagerly
            print(f"bench: graph capture failed ({e}); timing eagerly", file=sys.stderr)
            g_run = g_dom = g_ins = None
            torch.cuda.synchronize()

    def timed(fn_graph, fn_eager):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        if fn_graph is not None:
            fn_graph.replay()
        else:
            fn_eager()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if g_run is None:
        L.lpq_reset_launch_count()
    ms_total = timed(g_run, run_steps)           # <- the timed region: K steps
    if g_run is None:
        launches = L.lpq_launch_count()
    if dist:
        dist.barrier()
    ms_dom = timed(g_dom, dom_steps)
    timed(g_ins, lambda: ins_steps(stream, external=False))
    clocks = clk.stop()
    ms_total = max_over_ranks(ms_total, dist, "cuda")
    ms_step = ms_total / args.steps

    flops_step = sum(c["flops"] for c in W.calls)
    value = whole_job_rate(flops_step, world, ms_step) / 1e12

    # per-kernel statistics from the instrumented replay
    kinds = {}
    for s in range(args.steps):
        for i, c in enumerate(W.calls):
            ms = GE.elapsed_ms(evs[s][i][0], evs[s][i][1])
            for key in (c["kind"], f'{c["kind"]}[M={c["M"]},K={c["K"]},N={c["N"]}]'):
                k = kinds.setdefault(key, {"launch_ms": 0.0, "launches": 0, "bytes": 0, "flops": 0})
                k["launch_ms"] += ms
                k["launches"] += 1
                k["bytes"] += c["bytes"]
                k["flops"] += c["flops"]
    peaks = load_peaks()
    kern = {}
    for name, k in kinds.items():
        kern[name] = {"launches_per_step": k["launches"] // args.steps,
                      "avg_us": 1000 * k["launch_ms"] / k["launches"],
                      "GB/s": k["bytes"] / (k["launch_ms"] * 1e-3) / 1e9,
                      "TFLOP/s": k["flops"] / (k["launch_ms"] * 1e-3) / 1e12 if k["flops"] else 0.0,
                      "share": k["launch_ms"] / sum(v["launch_ms"] for n, v in kinds.items() if "[" not in n)}
    dom = dict(kinds[W.dominant])
    dom["launch_ms"] = ms_dom          # all dominant launches of K steps, back to back, no inner events
    if W.dominant_bound == "hbm":
        achieved = dom["bytes"] / (dom["launch_ms"] * 1e-3) / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
    else:
        achieved = dom["flops"] / (dom["launch_ms"] * 1e-3) / 1e12
        ratio = NOMINAL_RATIO[getattr(W, "dominant_dtype", "fp8")]
        peak, unit = peaks["bf16_tflops"] * ratio, "TFLOP/s"
    peak_src = f"{peaks['src']} ({'hbm_gbs' if unit == 'GB/s' else 'bf16_tflops x nominal ratio'})"
    extra = {}
    if getattr(W, "dominant_dtype", "") == "int8":
        # no tcgen05 INT8 MMA on this part: the GEMM runs four E4M3 MMAs per
        # int8 product (digit planes), so its tensor roofline in int8
        # operations is the FP8 rate / 4; the vendor library's INT8 GEMM
        # (legacy int8 MMA) is measured live for context
        peak = peaks["bf16_tflops"] * NOMINAL_RATIO["fp8"] / 4
        peak_src = f"{peaks['src']} (bf16_tflops x 2 for FP8, / 4 E4M3 MMAs per int8 product)"
        extra["library_int8_tops"] = measure_int8_library_peak(torch)
        extra["library_int8_src"] = "measured live: torch._int_mm 8192^3 (cuBLASLt INT8)"
    roofline = {"bound": W.dominant_bound, "kernel": W.dominant, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak,
                "peak_src": peak_src, **extra,
                "traffic": recorded_traffic(W.dominant),
                "algorithmic_bytes_per_launch": dom["bytes"] / dom["launches"],
                "algorithmic_flops_per_launch": dom["flops"] / dom["launches"],
                "avg_launch_us": 1000 * ms_dom / dom["launches"],
                "timing": "CUDA events around a graph replay of the K steps' launches of this kernel only"}

    # ---- end to end through the C ABI with host buffers (pinned): every step
    # copies its activations in and its Y out; the calls are captured in a
    # graph the way a serving loop replays them
    h2d = sum(t.numel() * t.element_size() for t in W.host_in)
    d2h = sum(t.numel() * t.element_size() for t in W.host_out)
    n_e2e = max(3, args.steps // 2)

    # the whole step's activations / outputs as one copy each (per call for a subset)
    pairs_in = list(zip(W.host_in, W.dev_in)) if W.subset else [(W.hin, W.din)]
    pairs_out = list(zip(W.host_out, W.dev_out)) if W.subset else [(W.hout, W.dout)]

    def e2e_steps():
        for _ in range(n_e2e):
            for h, d in pairs_in:
                d.copy_(h, non_blocking=True)
            step()
            for h, d in pairs_out:
                h.copy_(d, non_blocking=True)

    g2 = capture(e2e_steps) if g_run is not None else None
    if g2 is None:
        e2e_steps()
        torch.cuda.synchronize()
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_s.record(stream)
    if g2 is not None:
        g2.replay()
    else:
        e2e_steps()
    e_e.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e_s.elapsed_time(e_e) / n_e2e, dist, "cuda")
    e2e_val = whole_job_rate(flops_step, world, e2e_ms) / 1e12
    GE.close()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, desc, threads = oracle_sample(args.workload)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": {"decode_fp8": "fp8-e4m3 (fp32 accum)",
                                               "prefill_fp8_block": "fp8-e4m3 block-scaled (fp32 accum)",
                                               "int8_smoothquant": "int8 (int32 accum)",
                                               "nvfp4": "nvfp4-e2m1 (fp32 accum)",
                                               "mxfp4": "mxfp4-e2m1 (fp32 accum)"}[args.workload],
                "data": "synthetic (seeded, pages' shapes and outlier mix)",
                "config": dict(W.config, parallelism=f"replicas x{world}"),
                "roofline": roofline, "kernels": kern, "cpu_baseline": cpu,
                "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                        "ms_per_step": e2e_ms},
                "gpu_launches": launches, "clocks": clocks,
                "launch_mode": "cuda-graph replay" if g_run is not None else "eager",
                "kernel_table_timing": "per-launch event nodes in a replay after the timed region (adds a few us per launch)"}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
