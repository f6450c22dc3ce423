// abi.cu - the C ABI's shared host code: status strings, error and launch
// accounting, device queries, tensor-map encoding, the scale-factor layout
// and the GEMM dispatcher (lpq_gemm_scaled).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/lpq.h"
#include "gemm_fp8.h"
#include "internal.h"
#include "ptx.cuh"

namespace lpq {

namespace {
thread_local int t_last_cuda_error = 0;
thread_local uint64_t t_launches = 0;

__device__ uint32_t g_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

int current_device() {
  int d = 0;
  cudaGetDevice(&d);
  return (d >= 0 && d < kMaxDevices) ? d : 0;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}
}  // namespace

lpq_status record_cuda(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return LPQ_ERR_CUDA;
}

void count_launch(uint64_t n) { t_launches += n; }

uint32_t* error_word_ptr() {
  const int d = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) == cudaSuccess) g_err_ptr[d] = static_cast<uint32_t*>(p);
  }
  return g_err_ptr[d];
}

int sm_count() {
  const int d = current_device();
  if (g_sms[d] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = v > 0 ? v : 1;
  }
  return g_sms[d];
}

lpq_status ensure_smem_attr(const void* func, int bytes, uint64_t* done_mask) {
  const int d = current_device();
  const uint64_t bit = 1ull << d;
  if (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit) return LPQ_OK;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return record_cuda(e);
  __atomic_fetch_or(done_mask, bit, __ATOMIC_RELEASE);
  return LPQ_OK;
}

lpq_status make_tmap_u8(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes, int64_t ld_bytes,
                        int box_bytes, int box_rows, bool swizzle128) {
  auto enc = encode_fn();
  if (!enc) return record_cuda(cudaErrorNotSupported);
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return record_cuda(cudaErrorInvalidValue);
  return LPQ_OK;
}

}  // namespace lpq

using namespace lpq;

namespace lpq_diag {

// One barrier wait that nothing ends, bounded the way every wait in the
// library's kernels is: after limit_ns the thread records `where` in the
// device error word and the kernel returns (no trap; the context stays usable).
__global__ void bounded_wait_kernel(uint64_t limit_ns, uint32_t* err, uint32_t where) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    lpq::mbar_init(lpq::smem_u32(&bar), 1);
    lpq::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = lpq::globaltimer_ns();
    while (!lpq::mbar_try_wait(lpq::smem_u32(&bar), 0)) {
      if (lpq::globaltimer_ns() - t0 > limit_ns) {
        atomicCAS(err, 0u, where);
        break;
      }
    }
  }
}

}  // namespace lpq_diag

extern "C" {

lpq_status lpq_selftest_bounded_wait(uint64_t limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 2000000000ull) return LPQ_ERR_SHAPE;
  uint32_t* err = error_word_ptr();
  if (!err) return record_cuda(cudaErrorInvalidSymbol);
  lpq_diag::bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, err, LPQ_SELFTEST_WAIT_CODE);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? LPQ_OK : record_cuda(e);
}


const char* lpq_status_string(lpq_status s) {
  switch (s) {
    case LPQ_OK: return "ok";
    case LPQ_ERR_NULL: return "a required pointer is NULL";
    case LPQ_ERR_SHAPE: return "invalid size or stride (K must be a multiple of the block; ld >= K)";
    case LPQ_ERR_ALIGN: return "pointer not 16-byte aligned or row stride not a multiple of 8";
    case LPQ_ERR_UNSUPPORTED: return "format / granularity combination not supported";
    case LPQ_ERR_CUDA: return "CUDA launch error (see lpq_last_cuda_error)";
    case LPQ_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

int lpq_last_cuda_error(void) { return t_last_cuda_error; }

lpq_status lpq_read_error_word(uint32_t* out) {
  LPQ_CHECK_NULL(out);
  uint32_t* p = error_word_ptr();
  if (!p) return record_cuda(cudaErrorInvalidSymbol);
  cudaError_t e = cudaMemcpy(out, p, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? LPQ_OK : record_cuda(e);
}

lpq_status lpq_clear_error_word(void) {
  uint32_t* p = error_word_ptr();
  if (!p) return record_cuda(cudaErrorInvalidSymbol);
  cudaError_t e = cudaMemset(p, 0, sizeof(uint32_t));
  return e == cudaSuccess ? LPQ_OK : record_cuda(e);
}

const char* lpq_version(void) { return "lpq 0.1 (sm_103a)"; }
uint64_t lpq_launch_count(void) { return t_launches; }
void lpq_reset_launch_count(void) { t_launches = 0; }

size_t lpq_sf_bytes(lpq_format fmt, int64_t rows, int64_t K) {
  const int64_t blk = (fmt == LPQ_FMT_NVFP4) ? 16 : (fmt == LPQ_FMT_MXFP4 ? 32 : 0);
  if (blk == 0 || rows <= 0 || K <= 0) return 0;
  const int64_t kb4 = (K / blk + 3) / 4;
  return static_cast<size_t>((rows + 127) / 128 * 128 * kb4 * 4);
}

size_t lpq_sf_offset(lpq_format fmt, int64_t rows, int64_t K, int64_t r, int64_t kb) {
  const int64_t blk = (fmt == LPQ_FMT_NVFP4) ? 16 : (fmt == LPQ_FMT_MXFP4 ? 32 : 0);
  (void)rows;
  if (blk == 0) return 0;
  const int64_t kb4 = (K / blk + 3) / 4;
  return static_cast<size_t>(((r / 128) * kb4 + kb / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 4);
}

}  // extern "C"
