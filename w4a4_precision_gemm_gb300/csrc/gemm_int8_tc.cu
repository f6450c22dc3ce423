// gemm_int8_tc.cu - INT8 W8A8 GEMM on the 5th-generation tensor cores, exact.
//
// The operation is that of gemm_int8.cu: acc = sum_k q_x q_w exactly (int32),
// Y = bf16((float(acc) * s_x[t]) * s_w[n]) ("FP8 and INT8 Inference", section
// 5 "INT8 in practice"; "Low-bit LLM Weights and Activations", sections 3.4
// and 4.3).  sm_103a has no tcgen05 MMA kind for 8-bit integers, so each int8
// code is split into two base-16 digits that E4M3 represents exactly:
//   q = 16 h + l,   h = floor(q / 16) in [-8, 7],   l = q - 16 h in [0, 15],
// and the integer product is assembled from four FP8 products:
//   X W^T = 256 Xh Wh^T + 16 (Xh Wl^T + Xl Wh^T) + Xl Wl^T.
// Every partial sum is an integer of magnitude < 2^24 for K <= 65536 (at most
// 225 K), so the FP32 accumulation of the tensor core is exact; the epilogue
// converts the three accumulators to int32, combines them and applies the
// scales exactly as the int32 path does.
//
// Digit planes: int8_digit_split_kernel writes H and L ([rows][K] E4M3 codes)
// for both operands into the caller's workspace.  GEMM: 128 x 128 tiles,
// warp 0 TMA (four 16 KB operand tiles per stage: Ah, Al, Bh, Bl), warp 1
// tcgen05.mma into three tensor-memory accumulators (hh, hl + lh, ll),
// warps 2-5 epilogue.  All waits bounded.
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>

#include "gemm_common.cuh"
#include "gemm_fp8.h"
#include "internal.h"
#include "ptx.cuh"

namespace lpq {
namespace {

// Read-only load kept in program order (volatile asm): the epilogue loads a
// chunk's weight scales where it uses them instead of all 128 up front.
__device__ __forceinline__ float ld_nc_ordered(const float* ptr) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(ptr));
  return v;
}

constexpr int kThreads = 192;
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBKBytes = 128;                  // K elements per stage (one 128-byte swizzle row)
constexpr int kOpBytes = 128 * kBKBytes;       // one operand tile of one stage
constexpr int kStageBytes = 4 * kOpBytes;      // Ah, Al, Bh, Bl
constexpr int kStages = 3;
constexpr int kTmemCols = 512;                 // three 128-column accumulators
constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256;
// D fp32, A/B E4M3, both K-major, N = 128, M = 128
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(kBN >> 3) << 17) | (static_cast<uint32_t>(kBM >> 4) << 24);

// int8 codes [rows][ld] -> digit planes H, L [rows][K] (E4M3 codes of the
// integers h and l).  Grid (rows, ceil(K / 16 / 256)), 16 codes per thread.
__global__ void __launch_bounds__(256) int8_digit_split_kernel(const int8_t* __restrict__ Q, int64_t K, int64_t ld,
                                                               uint8_t* __restrict__ H, uint8_t* __restrict__ L) {
  pdl_launch();
  pdl_wait();
  const int64_t row = blockIdx.x;
  const int64_t c16 = static_cast<int64_t>(blockIdx.y) * blockDim.x + threadIdx.x;
  if (c16 * 16 >= K) return;
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(Q + row * ld + c16 * 16));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t hcodes = 0, lcodes = 0;
#pragma unroll
    for (int b = 0; b < 4; b += 2) {
      const int q0 = static_cast<int8_t>(w[i] >> (8 * b));
      const int q1 = static_cast<int8_t>(w[i] >> (8 * (b + 1)));
      const int h0 = q0 >> 4, h1 = q1 >> 4;          // floor division by 16
      const int l0 = q0 - 16 * h0, l1 = q1 - 16 * h1;
      // small integers are exact in E4M3, so the conversion only encodes them
      hcodes |= cvt_e4m3x2(static_cast<float>(h0), static_cast<float>(h1)) << (8 * b);
      lcodes |= cvt_e4m3x2(static_cast<float>(l0), static_cast<float>(l1)) << (8 * b);
    }
    hw[i] = hcodes;
    lw[i] = lcodes;
  }
  *reinterpret_cast<uint4*>(H + row * K + c16 * 16) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  *reinterpret_cast<uint4*>(L + row * K + c16 * 16) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_int8_tc_kernel(const __grid_constant__ CUtensorMap tmAh, const __grid_constant__ CUtensorMap tmAl,
                        const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmBl,
                        const GemmParams p) {
  constexpr int S = kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * kStageBytes);
  // bars: full[S], empty[S], tfull, tempty, drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + S + s); };
  const uint32_t tfull = smem_u32(bars + 2 * S);
  const uint32_t tempty = smem_u32(bars + 2 * S + 1);
  const uint32_t drain = smem_u32(bars + 2 * S + 2);
  auto op = [&](int s, int which) { return smem + s * kStageBytes + which * kOpBytes; };   // 0 Ah 1 Al 2 Bh 3 Bl

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmAh);
    tma_prefetch_desc(&tmAl);
    tma_prefetch_desc(&tmBh);
    tma_prefetch_desc(&tmBl);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_launch();
  pdl_wait();      // the digit planes come from the split kernels just before

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const uint64_t pol_a = policy_evict_last();
      const uint64_t pol_b = policy_evict_first();
      uint32_t stage = 0, phase = 0, issued = 0, issued_par = 0;
      bool ok = true;
      WorkIter wi(p, blockIdx.x, gridDim.x);
      Seg w;
      while (ok && wi.next(p, blockIdx.x, gridDim.x, w)) {
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait(empty(stage), phase ^ 1u, p.err, 0x401u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(full(stage), kStageBytes);
          const int x = kb * kBKBytes;
          tma_load_2d(smem_u32(op(stage, 0)), &tmAh, full(stage), x, w.i_tile * kBM, pol_a);
          tma_load_2d(smem_u32(op(stage, 1)), &tmAl, full(stage), x, w.i_tile * kBM, pol_a);
          tma_load_2d(smem_u32(op(stage, 2)), &tmBh, full(stage), x, w.j_tile * kBN, pol_b);
          tma_load_2d(smem_u32(op(stage, 3)), &tmBl, full(stage), x, w.j_tile * kBN, pol_b);
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        volatile int no_abort = 0;
        for (int s = 0; s < S; ++s)
          if (issued & (1u << s)) mbar_wait(full(s), (issued_par >> s) & 1u, nullptr, 0, &no_abort);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------------- MMA
      const uint32_t d_hh = tmem_base, d_mid = tmem_base + kBN, d_ll = tmem_base + 2 * kBN;
      uint32_t stage = 0, phase = 0, tphase = 0;
      bool ok = true;
      WorkIter wi(p, blockIdx.x, gridDim.x);
      Seg w;
      while (ok && wi.next(p, blockIdx.x, gridDim.x, w)) {
        if (!mbar_wait(tempty, tphase ^ 1u, p.err, 0x402u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait(full(stage), phase, p.err, 0x403u, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t ah = smem_u32(op(stage, 0)), al = smem_u32(op(stage, 1));
          const uint32_t bh = smem_u32(op(stage, 2)), bl = smem_u32(op(stage, 3));
#pragma unroll
          for (int k = 0; k < kBKBytes / 32; ++k) {
            const uint64_t dah = smem_desc(ah + k * 32, 16, 1024, 2), dal = smem_desc(al + k * 32, 16, 1024, 2);
            const uint64_t dbh = smem_desc(bh + k * 32, 16, 1024, 2), dbl = smem_desc(bl + k * 32, 16, 1024, 2);
            const uint32_t accum = (kb > w.kb0 || k > 0) ? 1u : 0u;
            mma_f8f6f4(d_hh, dah, dbh, kIdesc, accum);
            mma_f8f6f4(d_mid, dah, dbl, kIdesc, accum);
            mma_f8f6f4(d_mid, dal, dbh, kIdesc, 1u);
            mma_f8f6f4(d_ll, dal, dbl, kIdesc, accum);
          }
          tc_commit(empty(stage));
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(tfull);
        tphase ^= 1u;
      }
      tc_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, nullptr, 0, &no_abort);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // thread = one output row; acc = 256 hh + 16 (hl + lh) + ll, exact
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    uint32_t tphase = 0;
    WorkIter wi(p, blockIdx.x, gridDim.x);
    Seg w;
    while (wi.next(p, blockIdx.x, gridDim.x, w)) {
      if (!warp_wait(tfull, tphase, p.err, 0x404u, abort_flag)) break;
      tc_fence_after();
      const uint32_t lanes = static_cast<uint32_t>(quarter * 32) << 16;
      const int i = w.i_tile * kBM + row_in_tile;
      const int jt = w.j_tile * kBN;
      const float sxi = i < p.I ? __ldg(p.sx + i) : 0.0f;
      // the whole row into packed bf16 first, y = bf16((float(acc) s_x) s_w),
      // then release the accumulators and store: the next tile's MMAs run
      // under the stores (three accumulators leave no room for a second set)
      uint32_t y[kBN / 2];
#pragma unroll
      for (int c0 = 0; c0 < kBN; c0 += 16) {
        uint32_t hh[16], mid[16], ll[16];
        tmem_ld_32x32b_x16(tmem_base + lanes + c0, hh);
        tmem_ld_32x32b_x16(tmem_base + lanes + kBN + c0, mid);
        tmem_ld_32x32b_x16(tmem_base + lanes + 2 * kBN + c0, ll);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          float yv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int acc = 256 * __float2int_rn(__uint_as_float(hh[j + e])) +
                            16 * __float2int_rn(__uint_as_float(mid[j + e])) + __float2int_rn(__uint_as_float(ll[j + e]));
            const int jj = jt + c0 + j + e;
            const float swj = jj < p.J ? ld_nc_ordered(p.sw + jj) : 0.0f;
            yv[e] = __fmul_rn(__fmul_rn(static_cast<float>(acc), sxi), swj);
          }
          y[(c0 + j) / 2] = pack_bf16x2(yv[0], yv[1]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
      tphase ^= 1u;
      if (i < p.I) {
        uint16_t* yrow = p.Y + static_cast<int64_t>(i) * p.ldy + jt;
        const int n = p.J - jt;   // columns of this tile inside Y
        if (n >= kBN) {
#pragma unroll
          for (int c = 0; c < kBN; c += 8)
            *reinterpret_cast<uint4*>(yrow + c) = make_uint4(y[c / 2], y[c / 2 + 1], y[c / 2 + 2], y[c / 2 + 3]);
        } else {
#pragma unroll
          for (int c = 0; c < kBN; c += 2) {
            if (c + 1 < n) {
              *reinterpret_cast<uint32_t*>(yrow + c) = y[c / 2];
            } else if (c < n) {
              yrow[c] = static_cast<uint16_t>(y[c / 2]);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace

lpq_status split_planes(const int8_t* Q, int64_t rows, int64_t K, int64_t ld, uint8_t* H, uint8_t* L, cudaStream_t st) {
  const unsigned segs = static_cast<unsigned>((K / 16 + 255) / 256);
  return launch_pdl(int8_digit_split_kernel, dim3(static_cast<unsigned>(rows), segs), dim3(256), 0, st, 1, Q, K, ld, H, L);
}

size_t int8_tc_workspace_bytes(int64_t M, int64_t N, int64_t K, bool b_planes) {
  auto a256 = [](size_t b) { return (b + 255) / 256 * 256; };
  return 2 * a256(static_cast<size_t>(M) * K) + (b_planes ? 0 : 2 * a256(static_cast<size_t>(N) * K));
}

lpq_status launch_int8_tc(const int8_t* A, int64_t lda, const void* B, int64_t ldb, bool b_planes, int64_t M,
                          int64_t N, int64_t K, const float* sx, const float* sw, uint16_t* Y, int64_t ldy, void* ws,
                          cudaStream_t st) {
  if (K > kInt8TcMaxK || K % 16 != 0) return LPQ_ERR_UNSUPPORTED;
  auto a256 = [](size_t b) { return (b + 255) / 256 * 256; };
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint8_t* Ah = base;
  uint8_t* Al = Ah + a256(static_cast<size_t>(M) * K);
  const uint8_t* Bh;
  const uint8_t* Bl;
  lpq_status s;
  if ((s = split_planes(A, M, K, lda, Ah, Al, st)) != LPQ_OK) return s;
  if (b_planes) {
    Bh = static_cast<const uint8_t*>(B);
    Bl = Bh + static_cast<size_t>(N) * K;
  } else {
    uint8_t* bh = Al + a256(static_cast<size_t>(M) * K);
    uint8_t* bl = bh + a256(static_cast<size_t>(N) * K);
    if ((s = split_planes(static_cast<const int8_t*>(B), N, K, ldb, bh, bl, st)) != LPQ_OK) return s;
    Bh = bh;
    Bl = bl;
  }
  CUtensorMap tAh, tAl, tBh, tBl;
  if ((s = make_tmap_u8(&tAh, Ah, M, K, K, 128, kBM, true)) != LPQ_OK) return s;
  if ((s = make_tmap_u8(&tAl, Al, M, K, K, 128, kBM, true)) != LPQ_OK) return s;
  if ((s = make_tmap_u8(&tBh, Bh, N, K, K, 128, kBN, true)) != LPQ_OK) return s;
  if ((s = make_tmap_u8(&tBl, Bl, N, K, K, 128, kBN, true)) != LPQ_OK) return s;
  GemmParams p{};
  p.I = static_cast<int>(M);
  p.J = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.i_tiles = static_cast<int>((M + kBM - 1) / kBM);
  p.j_tiles = static_cast<int>((N + kBN - 1) / kBN);
  p.kblocks = static_cast<int>((K + kBKBytes - 1) / kBKBytes);
  p.dp_tiles = p.i_tiles * p.j_tiles;
  p.tail_s = 1;
  p.csplit = 1;
  p.kb_per_split = p.kblocks;
  p.j_fast = j_fastest(M, N, K, 2.0) ? 1 : 0;
  p.transposed = 0;
  p.sx = sx;
  p.sx_stride = 1;
  p.sw = sw;
  p.sw_stride = 1;
  p.Y = Y;
  p.ldy = ldy;
  p.err = error_word_ptr();
  static uint64_t done_mask = 0;
  if ((s = ensure_smem_attr(reinterpret_cast<const void*>(&gemm_int8_tc_kernel), kSmemBytes, &done_mask)) != LPQ_OK)
    return s;
  const int grid = static_cast<int>(std::min<int64_t>(static_cast<int64_t>(p.dp_tiles), sm_count()));
  return launch_pdl(gemm_int8_tc_kernel, dim3(grid), dim3(kThreads), kSmemBytes, st, 1, tAh, tAl, tBh, tBl, p);
}

}  // namespace lpq

using namespace lpq;

extern "C" lpq_status lpq_int8_weight_planes(const int8_t* Wq, int64_t N, int64_t K, int64_t ldw, uint8_t* planes,
                                             void* stream) {
  LPQ_CHECK_NULL(Wq);
  LPQ_CHECK_NULL(planes);
  if (N <= 0 || K <= 0 || K % 16 != 0 || ldw < K || N > 0x7FFFFFFFLL) return LPQ_ERR_SHAPE;
  LPQ_CHECK_ALIGN(Wq);
  LPQ_CHECK_ALIGN(planes);
  if (ldw % 16 != 0) return LPQ_ERR_ALIGN;
  return split_planes(Wq, N, K, ldw, planes, planes + static_cast<size_t>(N) * K, static_cast<cudaStream_t>(stream));
}
