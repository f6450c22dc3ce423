// gemm_noalloc.cu - lpq_gemm_scaled_noalloc: the FP8 row-scaled GEMM with
// its split-K scratch taken from a fixed array inside the library instead of
// a caller-provided workspace.
//
// Who needs this: a caller that cannot allocate device memory for a
// workspace - for example a plugin running inside a serving runtime that owns
// every byte of device memory through its own pool and hands the plugin only
// the tensors of the operation, or a latency-critical path where cudaMalloc's
// implicit device-wide synchronisation is not acceptable and no workspace was
// reserved ahead of time.  Such a caller still passes its inputs and outputs;
// only the partial sums of split tail tiles live here.
//
// The scratch is a file-scope __device__ array of LPQ_NOALLOC_SCRATCH_BYTES
// (16 MiB).  Every GPU that loads the library holds it until the process
// exits.  All calls on a device share it (no call reads what an earlier one
// left), so calls that may run at the same time on the GPU (different
// streams without ordering between them) race on it and give wrong results -
// order them on one stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/lpq.h"
#include "gemm_fp8.h"
#include "internal.h"

namespace lpq {
namespace {

constexpr size_t kNoallocScratchBytes = LPQ_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDev] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
lpq_status scratch_ptr(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_cuda(e);
  if (dev < 0 || dev >= kMaxDev) return LPQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return record_cuda(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return LPQ_OK;
}

}  // namespace
}  // namespace lpq

using namespace lpq;

extern "C" {

lpq_status lpq_gemm_scaled_noalloc(const lpq_gemm_desc* d, void* stream) {
  LPQ_CHECK_NULL(d);
  const bool fp8_row = d->fmt == LPQ_FMT_FP8 &&
                       (d->a_gran == LPQ_GRAN_ROW || d->a_gran == LPQ_GRAN_TENSOR_STATIC) && d->b_gran == LPQ_GRAN_ROW;
  if (!fp8_row || (d->flags & LPQ_GEMM_A_BF16)) return LPQ_ERR_UNSUPPORTED;   // codes only, no bf16 activations
  // the same argument rules as lpq_gemm_scaled for this format
  LPQ_CHECK_NULL(d->A);
  LPQ_CHECK_NULL(d->B);
  LPQ_CHECK_NULL(d->Y);
  LPQ_CHECK_NULL(d->sa);
  LPQ_CHECK_NULL(d->sb);
  if (d->M <= 0 || d->N <= 0 || d->K <= 0 || d->K % 16 != 0) return LPQ_ERR_SHAPE;
  if (d->M > 0x7FFFFFFFLL || d->N > 0x7FFFFFFFLL || d->K > 0x7FFFFFFFLL) return LPQ_ERR_SHAPE;
  if (d->lda < d->K || d->ldb < d->K || d->ldy < d->N) return LPQ_ERR_SHAPE;
  if (d->lda % 16 != 0 || d->ldb % 16 != 0 || d->ldy % 8 != 0) return LPQ_ERR_ALIGN;
  LPQ_CHECK_ALIGN(d->A);
  LPQ_CHECK_ALIGN(d->B);
  LPQ_CHECK_ALIGN(d->Y);

  // the tiling lpq_gemm_scaled would use with a large enough workspace
  const Fp8Plan pl = plan_fp8_rowscale(d->M, d->N, d->K, true, SIZE_MAX);
  const size_t need = plan_ws_bytes(pl);
  if (need > kNoallocScratchBytes) return LPQ_ERR_WORKSPACE;   // problem needs more than the built-in scratch

  void* scratch = nullptr;
  lpq_status s = scratch_ptr(&scratch);
  if (s != LPQ_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  const void* opA = pl.transposed ? d->B : d->A;
  const void* opB = pl.transposed ? d->A : d->B;
  const int64_t ldA = pl.transposed ? d->ldb : d->lda;
  const int64_t ldB = pl.transposed ? d->lda : d->ldb;
  CUtensorMap tmA, tmB;
  if ((s = make_tmap_u8(&tmA, opA, pl.I, d->K, ldA, 128, 128, true)) != LPQ_OK) return s;
  if ((s = make_tmap_u8(&tmB, opB, pl.J, d->K, ldB, 128, pl.bn, true)) != LPQ_OK) return s;
  GemmParams p{};
  p.K = static_cast<int>(d->K);
  p.sx = static_cast<const float*>(d->sa);
  p.sx_stride = (d->a_gran == LPQ_GRAN_TENSOR_STATIC) ? 0 : 1;
  p.sw = static_cast<const float*>(d->sb);
  p.sw_stride = 1;
  p.Y = d->Y;
  p.ldy = d->ldy;
  p.err = error_word_ptr();
  return launch_fp8_rowscale(pl, tmA, tmB, p, pl.tail_s > 1 ? scratch : nullptr, st);
}

}  // extern "C"
