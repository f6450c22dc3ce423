// quant.cu - dynamic quantizers (HBM-bound elementwise + reductions).
//
// Every kernel reads bf16 with 128-bit loads (8 elements per thread per
// load), reduces max|x| with warp shuffles, divides with IEEE round-to-nearest
// (__fdiv_rn, never a reciprocal multiply) and converts with the hardware's
// round-to-nearest-even, saturating conversions (cvt.rn.satfinite), so that
// codes and scales are the exact functions of the inputs stated in lpq.h.
//
// Formulas: "FP8 and FP4 inference, SmoothQuant and activation quantization",
// sections "Scale granularity" and "Implementation sketch"; "FP8 and INT8
// Inference", section 5; "Low-bit LLM Weights and Activations", sections 2.1,
// 2.4 and 4.2-4.3.
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace lpq {
namespace {

constexpr float kScaleFloor = 1e-8f;   // clamp(min=1e-8) of the per-token scale
constexpr int kRowThreads = 256;       // threads per row in the per-row kernels

struct Chunk8 {
  float v[8];
};

__device__ __forceinline__ Chunk8 load_bf16x8(const uint16_t* p) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  Chunk8 c;
  c.v[0] = bf16lo(u.x); c.v[1] = bf16hi(u.x);
  c.v[2] = bf16lo(u.y); c.v[3] = bf16hi(u.y);
  c.v[4] = bf16lo(u.z); c.v[5] = bf16hi(u.z);
  c.v[6] = bf16lo(u.w); c.v[7] = bf16hi(u.w);
  return c;
}

// Streaming variant for tensors read exactly once (keeps them out of L1).
__device__ __forceinline__ Chunk8 load_bf16x8_stream(const uint16_t* p) {
  uint4 u;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
               : "l"(p));
  Chunk8 c;
  c.v[0] = bf16lo(u.x); c.v[1] = bf16hi(u.x);
  c.v[2] = bf16lo(u.y); c.v[3] = bf16hi(u.y);
  c.v[4] = bf16lo(u.z); c.v[5] = bf16hi(u.z);
  c.v[6] = bf16lo(u.w); c.v[7] = bf16hi(u.w);
  return c;
}

__device__ __forceinline__ float amax8(const Chunk8& c) {
  float a = fabsf(c.v[0]);
#pragma unroll
  for (int i = 1; i < 8; ++i) a = fmaxf(a, fabsf(c.v[i]));
  return a;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide max over kRowThreads threads; every thread gets the result.
__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int i = 1; i < kRowThreads / 32; ++i) r = fmaxf(r, red[i]);
  __syncthreads();
  return r;
}

// Eight fp32 values -> eight E4M3FN codes (8 bytes), element 0 in the low byte.
__device__ __forceinline__ uint2 e4m3x8(const float (&q)[8]) {
  uint2 o;
  o.x = cvt_e4m3x2(q[0], q[1]) | (cvt_e4m3x2(q[2], q[3]) << 16);
  o.y = cvt_e4m3x2(q[4], q[5]) | (cvt_e4m3x2(q[6], q[7]) << 16);
  return o;
}

__device__ __forceinline__ uint32_t int8_code(float v) {
  int i = __float2int_rn(v);          // round half to even
  i = max(-127, min(127, i));
  return static_cast<uint32_t>(i) & 0xFFu;
}

// ------------------------------------------------------------------------
// Memory-level parallelism.  Each thread issues kCPT independent 16-byte
// loads before it uses any of them, so a resident thread keeps 64 bytes in
// flight; register use stays low enough for full occupancy.
// ------------------------------------------------------------------------
constexpr int kCPT = 4;

__device__ __forceinline__ void zero8(Chunk8& c) {
#pragma unroll
  for (int i = 0; i < 8; ++i) c.v[i] = 0.0f;
}

// Block-wide max for any blockDim that is a multiple of 32 (<= 1024).
__device__ __forceinline__ float block_max_any(float v, float* red) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  if (l == 0) red[w] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < nw; ++i) r = fmaxf(r, red[i]);
  __syncthreads();
  return r;
}

// ------------------------------------------------------------------------
// Per-row quantizers: one CTA per row, blockDim chosen on the host so that
// the row fits in kCPT chunks per thread (registers) up to 1024 threads;
// longer rows are read a second time (from L2).
// MODE 0: FP8 (x / s), MODE 1: INT8 activation (x / smooth_j), MODE 2: INT8
// weight (w * smooth_j), MODE 3: INT8 without smoothing.
// ------------------------------------------------------------------------
template <int MODE>
__device__ __forceinline__ void pre_transform(Chunk8& c, const float* smooth, int64_t k0) {
  if constexpr (MODE == 1 || MODE == 2) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(smooth + k0));
    const float4 b = __ldg(reinterpret_cast<const float4*>(smooth + k0 + 4));
    const float sm[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) c.v[i] = (MODE == 1) ? __fdiv_rn(c.v[i], sm[i]) : __fmul_rn(c.v[i], sm[i]);
  }
}

template <int MODE>
__device__ __forceinline__ void emit_codes(const Chunk8& c, float s, uint8_t* out) {
  float q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(c.v[i], s);
  if constexpr (MODE == 0) {
    *reinterpret_cast<uint2*>(out) = e4m3x8(q);
  } else {
    uint2 o;
    o.x = int8_code(q[0]) | (int8_code(q[1]) << 8) | (int8_code(q[2]) << 16) | (int8_code(q[3]) << 24);
    o.y = int8_code(q[4]) | (int8_code(q[5]) << 8) | (int8_code(q[6]) << 16) | (int8_code(q[7]) << 24);
    *reinterpret_cast<uint2*>(out) = o;
  }
}

template <int MODE>
__global__ void __launch_bounds__(1024) quant_row_kernel(const uint16_t* __restrict__ X, int K, int64_t ldx,
                                                          const float* __restrict__ smooth, uint8_t* __restrict__ Q,
                                                          float* __restrict__ S) {
  pdl_launch();
  pdl_wait();
  __shared__ float red[32];
  const int64_t row = blockIdx.x;
  const uint16_t* xr = X + row * ldx;
  uint8_t* qr = Q + row * K;
  const int T = blockDim.x;
  const int nchunks = K / 8;
  const float qmax = (MODE == 0) ? 448.0f : 127.0f;
  if (nchunks <= T * kCPT) {
    Chunk8 c[kCPT];
#pragma unroll
    for (int j = 0; j < kCPT; ++j) {
      const int ci = j * T + threadIdx.x;
      if (ci < nchunks) c[j] = load_bf16x8_stream(xr + static_cast<int64_t>(ci) * 8);
      else zero8(c[j]);
    }
    float a = 0.0f;
#pragma unroll
    for (int j = 0; j < kCPT; ++j) {
      const int ci = j * T + threadIdx.x;
      if (ci < nchunks) {
        pre_transform<MODE>(c[j], smooth, static_cast<int64_t>(ci) * 8);
        a = fmaxf(a, amax8(c[j]));
      }
    }
    a = block_max_any(a, red);
    const float s = __fdiv_rn(fmaxf(a, kScaleFloor), qmax);
    if (threadIdx.x == 0) S[row] = s;
#pragma unroll
    for (int j = 0; j < kCPT; ++j) {
      const int ci = j * T + threadIdx.x;
      if (ci < nchunks) emit_codes<MODE>(c[j], s, qr + static_cast<int64_t>(ci) * 8);
    }
  } else {
    float a = 0.0f;
    for (int ci = threadIdx.x; ci < nchunks; ci += T) {
      Chunk8 c = load_bf16x8(xr + static_cast<int64_t>(ci) * 8);
      pre_transform<MODE>(c, smooth, static_cast<int64_t>(ci) * 8);
      a = fmaxf(a, amax8(c));
    }
    a = block_max_any(a, red);
    const float s = __fdiv_rn(fmaxf(a, kScaleFloor), qmax);
    if (threadIdx.x == 0) S[row] = s;
    for (int ci = threadIdx.x; ci < nchunks; ci += T) {
      Chunk8 c = load_bf16x8(xr + static_cast<int64_t>(ci) * 8);
      pre_transform<MODE>(c, smooth, static_cast<int64_t>(ci) * 8);
      emit_codes<MODE>(c, s, qr + static_cast<int64_t>(ci) * 8);
    }
  }
}

// ------------------------------------------------------------------------
// FP8 per 1x128 group, on the row-segment mapping (declared below with the
// other segment kernels): for each j the 16 lanes 16g..16g+15 of a warp hold
// the 16 chunks of one 128-element group, so a half-warp reduces a group and
// every CTA reads a contiguous stretch of one row.  The scale is stored
// K-group major, S[kg * M + row] (the layout the block-scaled GEMM reads).
// ------------------------------------------------------------------------
__device__ __forceinline__ int seg_chunk(int j);

__global__ void __launch_bounds__(256) quant_fp8_group128_kernel(const uint16_t* __restrict__ X, int64_t M,
                                                                 int64_t K, int64_t ldx, uint8_t* __restrict__ Q,
                                                                 float* __restrict__ S) {
  pdl_launch();
  pdl_wait();
  const int64_t row = blockIdx.x;
  const int cpr = static_cast<int>(K / 8);
  const int lane = threadIdx.x & 31;
  Chunk8 c[kCPT];
#pragma unroll
  for (int j = 0; j < kCPT; ++j) {
    const int c8 = seg_chunk(j);
    if (c8 < cpr) c[j] = load_bf16x8_stream(X + row * ldx + static_cast<int64_t>(c8) * 8);
    else zero8(c[j]);
  }
#pragma unroll
  for (int j = 0; j < kCPT; ++j) {
    const int c8 = seg_chunk(j);
    float a = amax8(c[j]);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float s = __fdiv_rn(fmaxf(a, kScaleFloor), 448.0f);
    if (c8 < cpr) {
      if ((lane & 15) == 0) S[static_cast<int64_t>(c8 >> 4) * M + row] = s;
      float q[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(c[j].v[i], s);
      *reinterpret_cast<uint2*>(Q + row * K + static_cast<int64_t>(c8) * 8) = e4m3x8(q);
    }
  }
}

// ------------------------------------------------------------------------
// FP8 per 128x128 weight block: one CTA per block; 16 threads across the 128
// columns (8 each), 16 row phases x 8 rows.  Rows past N are skipped.
// ------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_fp8_block128_kernel(const uint16_t* __restrict__ W, int64_t N,
                                                                 int64_t K, int64_t ldw, uint8_t* __restrict__ Q,
                                                                 float* __restrict__ S) {
  pdl_launch();
  pdl_wait();
  __shared__ float red[8];
  const int64_t nb = blockIdx.y, kb = blockIdx.x;
  const int col8 = threadIdx.x & 15;
  const int rph = threadIdx.x >> 4;
  Chunk8 c[8];
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t r = nb * 128 + rph + 16 * i;
    if (r < N) {
      c[i] = load_bf16x8_stream(W + r * ldw + kb * 128 + col8 * 8);
      a = fmaxf(a, amax8(c[i]));
    }
  }
  a = block_max(a, red);
  const float s = __fdiv_rn(fmaxf(a, kScaleFloor), 448.0f);
  if (threadIdx.x == 0) S[nb * (K / 128) + kb] = s;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t r = nb * 128 + rph + 16 * i;
    if (r < N) {
      float q[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) q[j] = __fdiv_rn(c[i].v[j], s);
      *reinterpret_cast<uint2*>(Q + r * K + kb * 128 + col8 * 8) = e4m3x8(q);
    }
  }
}

// ------------------------------------------------------------------------
// Row-segment mapping shared by the elementwise and block-16/32 kernels:
// grid (rows, segments), blockDim T (multiple of 32); thread t of segment y
// handles chunks y*T*kCPT + j*T + t, j < kCPT, of its row.  Lanes of a warp
// hold consecutive chunks for each j.
// ------------------------------------------------------------------------
__device__ __forceinline__ int seg_chunk(int j) {
  return static_cast<int>(blockIdx.y) * static_cast<int>(blockDim.x) * kCPT + j * static_cast<int>(blockDim.x) +
         static_cast<int>(threadIdx.x);
}

// FP8 with a given (static) per-tensor scale: q = E4M3(x / s).
__global__ void __launch_bounds__(256) quant_fp8_static_kernel(const uint16_t* __restrict__ X, int64_t K,
                                                               int64_t ldx, const float* __restrict__ S,
                                                               uint8_t* __restrict__ Q) {
  pdl_launch();
  pdl_wait();
  const int64_t row = blockIdx.x;
  const int cpr = static_cast<int>(K / 8);
  const float s = __ldg(S);
  Chunk8 c[kCPT];
#pragma unroll
  for (int j = 0; j < kCPT; ++j) {
    const int c8 = seg_chunk(j);
    if (c8 < cpr) c[j] = load_bf16x8_stream(X + row * ldx + static_cast<int64_t>(c8) * 8);
  }
#pragma unroll
  for (int j = 0; j < kCPT; ++j) {
    const int c8 = seg_chunk(j);
    if (c8 < cpr) {
      float q[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(c[j].v[i], s);
      *reinterpret_cast<uint2*>(Q + row * K + static_cast<int64_t>(c8) * 8) = e4m3x8(q);
    }
  }
}

// ------------------------------------------------------------------------
// Tensor max|x| (NVFP4 pass 1): CTAs stride over rows with the row-segment
// mapping, block reduce, one atomicMax of the fp32 bit pattern (non-negative
// floats order like their bits).
// ------------------------------------------------------------------------
__global__ void __launch_bounds__(256) tensor_amax_kernel(const uint16_t* __restrict__ X, int64_t M, int64_t K,
                                                          int64_t ldx, float* __restrict__ out) {
  pdl_launch();
  pdl_wait();
  __shared__ float red[32];
  const int cpr = static_cast<int>(K / 8);
  float a = 0.0f;
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    Chunk8 c[kCPT];
#pragma unroll
    for (int j = 0; j < kCPT; ++j) {
      const int c8 = seg_chunk(j);
      if (c8 < cpr) c[j] = load_bf16x8(X + row * ldx + static_cast<int64_t>(c8) * 8);
      else zero8(c[j]);
    }
#pragma unroll
    for (int j = 0; j < kCPT; ++j) a = fmaxf(a, amax8(c[j]));
  }
  a = block_max_any(a, red);
  if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned int*>(out), __float_as_uint(a));
}

// Offset of scale (r, kb) in the 128x4-tile layout of lpq_sf_offset.
__device__ __forceinline__ int64_t sf_off(int64_t r, int64_t kb, int64_t kb4) {
  return ((r >> 7) * kb4 + (kb >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (kb & 3);
}

// ------------------------------------------------------------------------
// NVFP4 pass 2 (row-segment mapping): two lanes per 16-element block; eight
// lanes = four consecutive blocks = one 32-bit word of scale codes.
// ------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_nvfp4_kernel(const uint16_t* __restrict__ X, int64_t K, int64_t ldx,
                                                          uint8_t* __restrict__ Q, uint8_t* __restrict__ SF,
                                                          float* __restrict__ gs) {
  pdl_launch();
  pdl_wait();
  const int64_t row = blockIdx.x;
  const int cpr = static_cast<int>(K / 8);
  const float amax = gs[0];
  const float g = amax > 0.0f ? __fdiv_rn(amax, 2688.0f) : 1.0f;   // 448 * 6
  if (row == 0 && blockIdx.y == 0 && threadIdx.x == 0) gs[1] = g;
  Chunk8 c[kCPT];
#pragma unroll
  for (int j = 0; j < kCPT; ++j) {
    const int c8 = seg_chunk(j);
    if (c8 < cpr) c[j] = load_bf16x8_stream(X + row * ldx + static_cast<int64_t>(c8) * 8);
    else zero8(c[j]);
  }
  const int lane = threadIdx.x & 31;
  const int64_t kb4 = ((K / 16) + 3) / 4;
#pragma unroll
  for (int j = 0; j < kCPT; ++j) {
    const int c8 = seg_chunk(j);
    float ab = amax8(c[j]);
    ab = fmaxf(ab, __shfl_xor_sync(0xffffffffu, ab, 1));
    const float tsc = __fdiv_rn(__fdiv_rn(ab, 6.0f), g);
    const uint32_t code = cvt_e4m3x2(tsc, 0.0f) & 0xFFu;
    uint32_t packed = 0;
    if (code != 0) {
      const float s = __fmul_rn(e4m3_to_f32(code), g);
      float q[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(c[j].v[i], s);
      packed = cvt_e2m1x8(q);
    }
    // scale codes of 4 consecutive blocks -> one 32-bit word (lanes 8i..8i+7)
    uint32_t word = code << (8 * ((lane >> 1) & 3));
    word |= __shfl_xor_sync(0xffffffffu, word, 2);
    word |= __shfl_xor_sync(0xffffffffu, word, 4);
    if (c8 < cpr) {
      *reinterpret_cast<uint32_t*>(Q + row * (K / 2) + static_cast<int64_t>(c8) * 4) = packed;
      const int64_t kb = c8 >> 1;
      if ((K & 63) == 0) {
        if ((lane & 7) == 0) *reinterpret_cast<uint32_t*>(SF + sf_off(row, kb, kb4)) = word;
      } else if ((c8 & 1) == 0) {
        SF[sf_off(row, kb, kb4)] = static_cast<uint8_t>(code);
      }
    }
  }
}

// ------------------------------------------------------------------------
// MXFP4 (row-segment mapping): four lanes per 32-element block; exponent
// from the fp32 exponent field of the block max (exact floor(log2)), scaling
// by an exact power of 2.
// ------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_mxfp4_kernel(const uint16_t* __restrict__ X, int64_t K, int64_t ldx,
                                                          uint8_t* __restrict__ Q, uint8_t* __restrict__ SF) {
  pdl_launch();
  pdl_wait();
  const int64_t row = blockIdx.x;
  const int cpr = static_cast<int>(K / 8);
  Chunk8 c[kCPT];
#pragma unroll
  for (int j = 0; j < kCPT; ++j) {
    const int c8 = seg_chunk(j);
    if (c8 < cpr) c[j] = load_bf16x8_stream(X + row * ldx + static_cast<int64_t>(c8) * 8);
    else zero8(c[j]);
  }
  const int lane = threadIdx.x & 31;
  const int64_t kb4 = ((K / 32) + 3) / 4;
#pragma unroll
  for (int j = 0; j < kCPT; ++j) {
    const int c8 = seg_chunk(j);
    float ab = amax8(c[j]);
    ab = fmaxf(ab, __shfl_xor_sync(0xffffffffu, ab, 1));
    ab = fmaxf(ab, __shfl_xor_sync(0xffffffffu, ab, 2));
    const int E = static_cast<int>((__float_as_uint(ab) >> 23) & 0xFFu);
    // floor(log2 ab) = E - 127 for normal ab; zero / subnormal -> clamp to -127
    const int e = (E == 0) ? -127 : max(E - 129, -127);
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);   // 2^-e, exact
    float q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = __fmul_rn(c[j].v[i], inv);
    const uint32_t packed = cvt_e2m1x8(q);
    const uint32_t code = static_cast<uint32_t>(e + 127);
    uint32_t word = code << (8 * ((lane >> 2) & 3));
    word |= __shfl_xor_sync(0xffffffffu, word, 4);
    word |= __shfl_xor_sync(0xffffffffu, word, 8);
    if (c8 < cpr) {
      *reinterpret_cast<uint32_t*>(Q + row * (K / 2) + static_cast<int64_t>(c8) * 4) = packed;
      const int64_t kb = c8 >> 2;
      if ((K & 127) == 0) {
        if ((lane & 15) == 0) *reinterpret_cast<uint32_t*>(SF + sf_off(row, kb, kb4)) = word;
      } else if ((c8 & 3) == 0) {
        SF[sf_off(row, kb, kb4)] = static_cast<uint8_t>(code);
      }
    }
  }
}

// Zero the padding of a scale-factor buffer: rows [rows, rows_pad) of every
// tile and blocks [kblocks, kb4*4) of every row.
__global__ void sf_pad_kernel(uint8_t* __restrict__ SF, int64_t rows, int64_t kblocks) {
  pdl_launch();
  pdl_wait();
  const int64_t kb4 = (kblocks + 3) / 4;
  const int64_t rows_pad = (rows + 127) / 128 * 128;
  const int64_t n = rows_pad * kb4 * 4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / (kb4 * 4), kb = i % (kb4 * 4);
    if (r >= rows || kb >= kblocks) SF[sf_off(r, kb, kb4)] = 0;
  }
}

int64_t grid_for(int64_t threads, int block = 256) { return (threads + block - 1) / block; }

// Largest row, in elements, that the 32-bit chunk indices of the kernels
// above cover (K / 8 chunks, times kCPT, in an int).
constexpr int64_t kMaxK = int64_t(1) << 30;

lpq_status check_x(const uint16_t* X, int64_t M, int64_t K, int64_t ldx, int64_t kmult) {
  LPQ_CHECK_NULL(X);
  if (M <= 0 || K <= 0 || ldx < K || K % kmult != 0 || K > kMaxK || M > 0x7FFFFFFFLL) return LPQ_ERR_SHAPE;
  LPQ_CHECK_ALIGN(X);
  if (ldx % 8 != 0) return LPQ_ERR_ALIGN;
  return LPQ_OK;
}

// Row-segment launch shape: T threads (multiple of 32, <= 256) and the number
// of segments per row.
struct SegShape {
  int threads;
  unsigned segs;
};
SegShape seg_shape(int64_t K) {
  const int64_t cpr = K / 8;
  int64_t t = (cpr + kCPT - 1) / kCPT;
  t = std::min<int64_t>(256, std::max<int64_t>(32, (t + 31) / 32 * 32));
  return {static_cast<int>(t), static_cast<unsigned>((cpr + t * kCPT - 1) / (t * kCPT))};
}

lpq_status launch_row(int mode, const uint16_t* X, int64_t M, int64_t K, int64_t ldx, const float* smooth,
                      uint8_t* Q, float* S, cudaStream_t st) {
  // Few rows: spread each row over more threads (one chunk each) for latency;
  // many rows: kCPT chunks per thread for bytes in flight.
  const int64_t nch = K / 8;
  const int64_t per = (M < 2 * static_cast<int64_t>(sm_count())) ? 1 : kCPT;
  int64_t t = (nch + per - 1) / per;
  t = std::min<int64_t>(1024, std::max<int64_t>(32, (t + 31) / 32 * 32));
  const dim3 grid(static_cast<unsigned>(M)), block(static_cast<unsigned>(t));
  const int k = static_cast<int>(K);
  switch (mode) {
    case 0: return launch_pdl(quant_row_kernel<0>, grid, block, 0, st, 1, X, k, ldx, smooth, Q, S);
    case 1: return launch_pdl(quant_row_kernel<1>, grid, block, 0, st, 1, X, k, ldx, smooth, Q, S);
    case 2: return launch_pdl(quant_row_kernel<2>, grid, block, 0, st, 1, X, k, ldx, smooth, Q, S);
    default: return launch_pdl(quant_row_kernel<3>, grid, block, 0, st, 1, X, k, ldx, smooth, Q, S);
  }
}

lpq_status fp4_common(bool nv, const uint16_t* X, int64_t M, int64_t K, int64_t ldx, uint8_t* Q, uint8_t* SF,
                      float* gs, cudaStream_t st) {
  lpq_status s = check_x(X, M, K, ldx, 32);
  if (s != LPQ_OK) return s;
  LPQ_CHECK_NULL(Q);
  LPQ_CHECK_NULL(SF);
  LPQ_CHECK_ALIGN(Q);
  LPQ_CHECK_ALIGN(SF);
  const SegShape sh = seg_shape(K);
  if (sh.segs > 65535u) return LPQ_ERR_SHAPE;
  const dim3 grid(static_cast<unsigned>(M), sh.segs), block(static_cast<unsigned>(sh.threads));
  if (nv) {
    LPQ_CHECK_NULL(gs);
    if ((reinterpret_cast<uintptr_t>(gs) & 3u) != 0) return LPQ_ERR_ALIGN;
    cudaError_t e = cudaMemsetAsync(gs, 0, sizeof(float), st);
    if (e != cudaSuccess) return record_cuda(e);
    const int64_t want = std::max<int64_t>(1, static_cast<int64_t>(sm_count()) * (2048 / sh.threads) / sh.segs);
    const dim3 agrid(static_cast<unsigned>(std::min<int64_t>(M, want)), sh.segs);
    if ((s = launch_pdl(tensor_amax_kernel, agrid, block, 0, st, 1, X, M, K, ldx, gs)) != LPQ_OK) return s;
    if ((s = launch_pdl(quant_nvfp4_kernel, grid, block, 0, st, 1, X, K, ldx, Q, SF, gs)) != LPQ_OK) return s;
  } else {
    if ((s = launch_pdl(quant_mxfp4_kernel, grid, block, 0, st, 1, X, K, ldx, Q, SF)) != LPQ_OK) return s;
  }
  const int64_t kblocks = K / (nv ? 16 : 32);
  if (M % 128 != 0 || kblocks % 4 != 0) {
    const unsigned pg = static_cast<unsigned>(std::min<int64_t>(grid_for((M + 127) / 128 * 128 * (kblocks + 3)), 4096));
    if ((s = launch_pdl(sf_pad_kernel, dim3(pg), dim3(256), 0, st, 1, SF, M, kblocks)) != LPQ_OK) return s;
  }
  return LPQ_OK;
}

}  // namespace
}  // namespace lpq

using namespace lpq;

extern "C" {

lpq_status lpq_quantize_act_fp8(const uint16_t* X, int64_t M, int64_t K, int64_t ldx, lpq_gran g, uint8_t* Xq,
                                float* sx, void* stream) {
  const int64_t kmult = (g == LPQ_GRAN_BLOCK_1x128) ? 128 : 16;
  lpq_status s = check_x(X, M, K, ldx, kmult);
  if (s != LPQ_OK) return s;
  LPQ_CHECK_NULL(Xq);
  LPQ_CHECK_NULL(sx);
  LPQ_CHECK_ALIGN(Xq);
  if ((reinterpret_cast<uintptr_t>(sx) & 3u) != 0) return LPQ_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (g) {
    case LPQ_GRAN_ROW:
      return launch_row(0, X, M, K, ldx, nullptr, Xq, sx, st);
    case LPQ_GRAN_BLOCK_1x128: {
      const SegShape sh = seg_shape(K);
      if (sh.segs > 65535u) return LPQ_ERR_SHAPE;
      const dim3 grid(static_cast<unsigned>(M), sh.segs);
      return launch_pdl(quant_fp8_group128_kernel, grid, dim3(static_cast<unsigned>(sh.threads)), 0, st, 1, X, M, K,
                        ldx, Xq, sx);
    }
    case LPQ_GRAN_TENSOR_STATIC: {
      const SegShape sh = seg_shape(K);
      if (sh.segs > 65535u) return LPQ_ERR_SHAPE;
      const dim3 grid(static_cast<unsigned>(M), sh.segs);
      return launch_pdl(quant_fp8_static_kernel, grid, dim3(static_cast<unsigned>(sh.threads)), 0, st, 1, X, K, ldx,
                        static_cast<const float*>(sx), Xq);
    }
    default:
      return LPQ_ERR_UNSUPPORTED;
  }
}

lpq_status lpq_quantize_weight_fp8(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, lpq_gran g, uint8_t* Wq,
                                   float* sw, void* stream) {
  const int64_t kmult = (g == LPQ_GRAN_BLOCK_128x128) ? 128 : 16;
  lpq_status s = check_x(W, N, K, ldw, kmult);
  if (s != LPQ_OK) return s;
  LPQ_CHECK_NULL(Wq);
  LPQ_CHECK_NULL(sw);
  LPQ_CHECK_ALIGN(Wq);
  if ((reinterpret_cast<uintptr_t>(sw) & 3u) != 0) return LPQ_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (g == LPQ_GRAN_ROW) return launch_row(0, W, N, K, ldw, nullptr, Wq, sw, st);
  if (g == LPQ_GRAN_BLOCK_128x128) {
    dim3 grid(static_cast<unsigned>(K / 128), static_cast<unsigned>((N + 127) / 128));
    return launch_pdl(quant_fp8_block128_kernel, grid, dim3(256), 0, st, 1, W, N, K, ldw, Wq, sw);
  }
  return LPQ_ERR_UNSUPPORTED;
}

lpq_status lpq_quantize_act_int8(const uint16_t* X, int64_t M, int64_t K, int64_t ldx, const float* smooth,
                                 int8_t* Xq, float* sx, void* stream) {
  lpq_status s = check_x(X, M, K, ldx, 16);
  if (s != LPQ_OK) return s;
  LPQ_CHECK_NULL(Xq);
  LPQ_CHECK_NULL(sx);
  LPQ_CHECK_ALIGN(Xq);
  if (smooth) LPQ_CHECK_ALIGN(smooth);
  if ((reinterpret_cast<uintptr_t>(sx) & 3u) != 0) return LPQ_ERR_ALIGN;
  return launch_row(smooth ? 1 : 3, X, M, K, ldx, smooth, reinterpret_cast<uint8_t*>(Xq), sx,
                    static_cast<cudaStream_t>(stream));
}

lpq_status lpq_quantize_weight_int8(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, const float* smooth,
                                    int8_t* Wq, float* sw, void* stream) {
  lpq_status s = check_x(W, N, K, ldw, 16);
  if (s != LPQ_OK) return s;
  LPQ_CHECK_NULL(Wq);
  LPQ_CHECK_NULL(sw);
  LPQ_CHECK_ALIGN(Wq);
  if (smooth) LPQ_CHECK_ALIGN(smooth);
  if ((reinterpret_cast<uintptr_t>(sw) & 3u) != 0) return LPQ_ERR_ALIGN;
  return launch_row(smooth ? 2 : 3, W, N, K, ldw, smooth, reinterpret_cast<uint8_t*>(Wq), sw,
                    static_cast<cudaStream_t>(stream));
}

lpq_status lpq_quantize_act_nvfp4(const uint16_t* X, int64_t M, int64_t K, int64_t ldx, uint8_t* Xq, uint8_t* sf,
                                  float* gs, void* stream) {
  return fp4_common(true, X, M, K, ldx, Xq, sf, gs, static_cast<cudaStream_t>(stream));
}

lpq_status lpq_quantize_weight_nvfp4(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, uint8_t* Wq, uint8_t* sf,
                                     float* gs, void* stream) {
  return fp4_common(true, W, N, K, ldw, Wq, sf, gs, static_cast<cudaStream_t>(stream));
}

lpq_status lpq_quantize_act_mxfp4(const uint16_t* X, int64_t M, int64_t K, int64_t ldx, uint8_t* Xq, uint8_t* sf,
                                  void* stream) {
  return fp4_common(false, X, M, K, ldx, Xq, sf, nullptr, static_cast<cudaStream_t>(stream));
}

lpq_status lpq_quantize_weight_mxfp4(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, uint8_t* Wq, uint8_t* sf,
                                     void* stream) {
  return fp4_common(false, W, N, K, ldw, Wq, sf, nullptr, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
