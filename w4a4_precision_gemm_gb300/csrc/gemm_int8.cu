// gemm_int8.cu - INT8 W8A8 GEMM (SmoothQuant path): int8 x int8 -> exact
// int32 accumulation, epilogue Y = bf16((float(acc) * s_x[t]) * s_w[n])
// ("FP8 and INT8 Inference", section 5 "INT8 in practice"; "Low-bit LLM
// Weights and Activations", sections 3.4 and 4.3).
//
// sm_103a has no tcgen05 MMA kind for 8-bit integers (ptxas rejects
// tcgen05.mma.kind::i8 for this target), so the product runs on the warp-level
// integer tensor-core instruction mma.sync.m16n8k32.s8.s8.s32.  Operands still
// move by TMA (128-byte swizzled tiles, mbarrier ring) and are read into
// registers with ldmatrix from the swizzled layout.
//
// CTA: 128 x 128 output tile, warp 0 = TMA producer, warps 1-4 = consumers in
// a 2 x 2 grid of 64 x 64 warp tiles (4 x 8 m16n8 accumulators per thread).
// Persistent over tiles; all waits bounded.
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>

#include "gemm_common.cuh"
#include "gemm_fp8.h"
#include "internal.h"
#include "ptx.cuh"

namespace lpq {
namespace {

constexpr int kBM = 128, kBN = 128, kBK = 128;   // bytes of K per stage = int8 elements
constexpr int kConsumers = 4;
constexpr int kThreads = 32 * (1 + kConsumers);
constexpr int kStageBytes = (kBM + kBN) * kBK;
constexpr int kStages = 6;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256;

struct Int8Params {
  int M, N, K;
  int m_tiles, n_tiles, kblocks;
  const float* sx;
  const float* sw;
  uint16_t* Y;
  int64_t ldy;
  uint32_t* err;
};

// address of 16-byte chunk `chunk` of row `row` in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128(uint32_t base, int row, int chunk) {
  return base + row * 128 + ((chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_s8(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_int8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const Int8Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kBM * kBK;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * kBN * kBK);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kStages);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + kStages + s); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kConsumers);
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  __syncthreads();
  pdl_launch();
  pdl_wait();      // inputs of this call may come from the previous kernel
  const int tiles = p.m_tiles * p.n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      uint32_t stage = 0, phase = 0, issued = 0, issued_par = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int mt = t % p.m_tiles, nt = t / p.m_tiles;
        for (int kb = 0; kb < p.kblocks; ++kb) {
          if (!mbar_wait(empty(stage), phase ^ 1u, p.err, 0x401u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(full(stage), kStageBytes);
          tma_load_2d(smem_u32(sA + stage * kBM * kBK), &tmA, full(stage), kb * kBK, mt * kBM, pol);
          tma_load_2d(smem_u32(sB + stage * kBN * kBK), &tmB, full(stage), kb * kBK, nt * kBN, pol);
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        volatile int no_abort = 0;
        for (int s = 0; s < kStages; ++s)
          if (issued & (1u << s)) mbar_wait(full(s), (issued_par >> s) & 1u, nullptr, 0, &no_abort);
      }
    }
  } else {
    const int cw = warp - 1;               // consumer warp 0..3
    const int wm = cw & 1, wn = cw >> 1;   // 64 x 64 warp tile at (64 wm, 64 wn)
    const int gid = lane >> 2, tig = lane & 3;
    uint32_t stage = 0, phase = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
      const int mt = t % p.m_tiles, nt = t / p.m_tiles;
      int acc[4][8][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[i][j][q] = 0;
      bool ok = true;
      for (int kb = 0; kb < p.kblocks; ++kb) {
        if (!mbar_wait(full(stage), phase, p.err, 0x402u, abort_flag)) { ok = false; break; }
        const uint32_t a0 = smem_u32(sA + stage * kBM * kBK);
        const uint32_t b0 = smem_u32(sB + stage * kBN * kBK);
#pragma unroll
        for (int ks = 0; ks < kBK / 32; ++ks) {
          const int c0 = ks * 2;           // 16-byte chunk of this k32 step
          uint32_t af[4][4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            // matrices: [rows 0-7, c0], [rows 8-15, c0], [rows 0-7, c0+1], [rows 8-15, c0+1]
            const int r = wm * 64 + i * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            ldsm_x4(sw128(a0, r, c0 + (lane >> 4)), af[i][0], af[i][1], af[i][2], af[i][3]);
          }
          uint32_t bf[8][2];
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            // matrices: [n 0-7, c0], [n 0-7, c0+1], [n 8-15, c0], [n 8-15, c0+1]
            const int r = wn * 64 + j * 8 + (lane & 7) + (lane >> 4) * 8;
            ldsm_x4(sw128(b0, r, c0 + ((lane >> 3) & 1)), bf[j][0], bf[j][1], bf[j + 1][0], bf[j + 1][1]);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) mma_s8(acc[i][j], af[i], bf[j][0], bf[j][1]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(stage));
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      // epilogue: y = bf16((float(acc) * s_x[m]) * s_w[n])
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int m = mt * kBM + wm * 64 + i * 16 + gid + h * 8;
          if (m >= p.M) continue;
          const float sxm = __ldg(p.sx + m);
          uint16_t* yrow = p.Y + static_cast<int64_t>(m) * p.ldy;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int n = nt * kBN + wn * 64 + j * 8 + tig * 2;
            if (n + 1 < p.N) {
              const float y0 = __fmul_rn(__fmul_rn(static_cast<float>(acc[i][j][2 * h]), sxm), __ldg(p.sw + n));
              const float y1 = __fmul_rn(__fmul_rn(static_cast<float>(acc[i][j][2 * h + 1]), sxm), __ldg(p.sw + n + 1));
              *reinterpret_cast<uint32_t*>(yrow + n) = pack_bf16x2(y0, y1);
            } else if (n < p.N) {
              const float y0 = __fmul_rn(__fmul_rn(static_cast<float>(acc[i][j][2 * h]), sxm), __ldg(p.sw + n));
              yrow[n] = __bfloat16_as_ushort(__float2bfloat16_rn(y0));
            }
          }
        }
      }
    }
  }
  __syncthreads();
}

}  // namespace

lpq_status launch_int8(const CUtensorMap& tmA, const CUtensorMap& tmB, int64_t M, int64_t N, int64_t K,
                       const float* sx, const float* sw, uint16_t* Y, int64_t ldy, cudaStream_t st) {
  static uint64_t done_mask = 0;
  lpq_status s = ensure_smem_attr(reinterpret_cast<const void*>(&gemm_int8_kernel), kSmemBytes, &done_mask);
  if (s != LPQ_OK) return s;
  Int8Params p{};
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.m_tiles = static_cast<int>((M + kBM - 1) / kBM);
  p.n_tiles = static_cast<int>((N + kBN - 1) / kBN);
  p.kblocks = static_cast<int>((K + kBK - 1) / kBK);
  p.sx = sx;
  p.sw = sw;
  p.Y = Y;
  p.ldy = ldy;
  p.err = error_word_ptr();
  const int grid = std::min(p.m_tiles * p.n_tiles, sm_count());
  return launch_pdl(gemm_int8_kernel, dim3(grid), dim3(kThreads), kSmemBytes, st, 1, tmA, tmB, p);
}

}  // namespace lpq
