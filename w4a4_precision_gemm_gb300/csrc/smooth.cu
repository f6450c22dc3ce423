// smooth.cu - SmoothQuant calibration: per-input-channel activation maxima
// over a calibration batch and the smoothing factors
//   s_j = max(ax_j, 1e-5)^alpha / max(aw_j, 1e-5)^(1 - alpha)
// ("Low-bit LLM Weights and Activations", sections 4.2 and 4.3; the 1e-5
// clamps follow the emulation in "FP8 and FP4 inference, SmoothQuant and
// activation quantization", section "Implementation sketch").
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace lpq {
namespace {

// Column max of |X| for a [rows, K] bf16 matrix, folded into out[K] with an
// atomicMax on the (non-negative) fp32 bit pattern.  Thread (x) owns 8
// consecutive columns; blockIdx.y strides over row slices.
__global__ void __launch_bounds__(256) col_absmax_kernel(const uint16_t* __restrict__ X, int64_t rows, int64_t K,
                                                         int64_t ld, int64_t rows_per_slice,
                                                         unsigned int* __restrict__ out) {
  pdl_launch();
  pdl_wait();
  const int64_t c8 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c8 * 8 >= K) return;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_slice;
  const int64_t r1 = (r0 + rows_per_slice < rows) ? r0 + rows_per_slice : rows;
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int64_t r = r0; r < r1; ++r) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(X + r * ld + c8 * 8));
    a[0] = fmaxf(a[0], fabsf(bf16lo(u.x))); a[1] = fmaxf(a[1], fabsf(bf16hi(u.x)));
    a[2] = fmaxf(a[2], fabsf(bf16lo(u.y))); a[3] = fmaxf(a[3], fabsf(bf16hi(u.y)));
    a[4] = fmaxf(a[4], fabsf(bf16lo(u.z))); a[5] = fmaxf(a[5], fabsf(bf16hi(u.z)));
    a[6] = fmaxf(a[6], fabsf(bf16lo(u.w))); a[7] = fmaxf(a[7], fabsf(bf16hi(u.w)));
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) atomicMax(out + c8 * 8 + i, __float_as_uint(a[i]));
}

// s_j from ax_j and aw_j (aw held in s on entry), fp64 power, one rounding.
__global__ void smooth_finalize_kernel(const float* __restrict__ ax, float* __restrict__ s, int64_t K, float alpha) {
  pdl_launch();
  pdl_wait();
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= K) return;
  const double a = static_cast<double>(alpha);
  const double x = static_cast<double>(fmaxf(ax[j], 1e-5f));
  const double w = static_cast<double>(fmaxf(s[j], 1e-5f));
  s[j] = static_cast<float>(pow(x, a) / pow(w, 1.0 - a));
}

lpq_status launch_colmax(const uint16_t* X, int64_t rows, int64_t K, int64_t ld, float* out, cudaStream_t st) {
  const int64_t cols8 = K / 8;
  const unsigned gx = static_cast<unsigned>((cols8 + 255) / 256);
  // enough row slices to put ~4 CTAs on every SM
  int64_t slices = std::max<int64_t>(1, std::min<int64_t>(rows, (static_cast<int64_t>(sm_count()) * 4 + gx - 1) / gx));
  slices = std::min<int64_t>(slices, 65535);
  const int64_t per = (rows + slices - 1) / slices;
  slices = (rows + per - 1) / per;
  return launch_pdl(col_absmax_kernel, dim3(gx, static_cast<unsigned>(slices)), dim3(256), 0, st, 1, X, rows, K, ld, per,
                    reinterpret_cast<unsigned int*>(out));
}

}  // namespace
}  // namespace lpq

using namespace lpq;

extern "C" {

lpq_status lpq_act_absmax_update(const uint16_t* X, int64_t M, int64_t K, int64_t ldx, float* chan_amax,
                                 void* stream) {
  LPQ_CHECK_NULL(X);
  LPQ_CHECK_NULL(chan_amax);
  if (M <= 0 || K <= 0 || ldx < K || K % 16 != 0) return LPQ_ERR_SHAPE;
  LPQ_CHECK_ALIGN(X);
  LPQ_CHECK_ALIGN(chan_amax);
  if (ldx % 8 != 0) return LPQ_ERR_ALIGN;
  return launch_colmax(X, M, K, ldx, chan_amax, static_cast<cudaStream_t>(stream));
}

lpq_status lpq_smooth_calibrate(const float* chan_amax, const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                                float alpha, float* s, void* stream) {
  LPQ_CHECK_NULL(chan_amax);
  LPQ_CHECK_NULL(W);
  LPQ_CHECK_NULL(s);
  if (N <= 0 || K <= 0 || ldw < K || K % 16 != 0) return LPQ_ERR_SHAPE;
  if (!(alpha >= 0.0f && alpha <= 1.0f)) return LPQ_ERR_SHAPE;
  LPQ_CHECK_ALIGN(W);
  LPQ_CHECK_ALIGN(s);
  if (ldw % 8 != 0) return LPQ_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(s, 0, static_cast<size_t>(K) * sizeof(float), st);
  if (e != cudaSuccess) return record_cuda(e);
  lpq_status r = launch_colmax(W, N, K, ldw, s, st);
  if (r != LPQ_OK) return r;
  return launch_pdl(smooth_finalize_kernel, dim3(static_cast<unsigned>((K + 255) / 256)), dim3(256), 0, st, 1, chan_amax, s,
                    K, alpha);
}

}  // extern "C"
