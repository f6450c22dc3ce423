// gemm_fp8_block.cu - FP8 GEMM with DeepSeek-V3-style block scales:
// activations scaled per 1x128 K group (s_x[kb][m]), weights per 128x128
// block (s_w[n/128][kb]).  Block scales sit inside the K reduction, so they
// cannot be applied once at the end; the partial product of every 128-wide K
// group is promoted into an fp32 accumulator with its two scales:
//   acc[m, n] += (sum_{k in group kb} q_x q_w) * s_x[kb][m] * s_w[n/128][kb]
// ("FP8 and INT8 Inference", section 5 "What DeepSeek did": fine-grained
// block scaling with FP32 accumulation at intervals; "FP8 and FP4 inference,
// SmoothQuant and activation quantization", section "Scale granularity").
//
// Warp roles as in the row-scaled kernel, except that the tensor-memory
// buffers hold per-group partial sums (NP of them, so the MMA of group kb+1..
// overlaps the promotion of group kb) and the running accumulator lives in
// the epilogue threads' registers (thread = output row, 128 of 256 columns).
// The promotion is bound by the latency of tensor-memory loads (a load-and-
// wait round trip costs ~140 cycles per warp); 128 x 128 tiles, which let a
// warp issue all its loads of a group before one wait, measured slower
// because they stage twice the operand bytes per MMA.
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>

#include "gemm_common.cuh"
#include "gemm_fp8.h"
#include "internal.h"
#include "ptx.cuh"

namespace lpq {
namespace {

constexpr int kEpiWarps = 8;                 // two per tensor-memory lane quarter, 128 columns each
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kBM = 128;
constexpr int kBN = kFp8BlockBN;
constexpr int kBK = 128;
constexpr int kNP = 2;                       // partial-sum buffers in tensor memory
constexpr int kStageBytes = (kBM + kBN) * kBK;
constexpr int kStages = 4;
constexpr int kTmemCols = 512;               // kNP x 256
constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256;
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(kBN >> 3) << 17) | (static_cast<uint32_t>(kBM >> 4) << 24);

struct BlockParams {
  int M, N, K;
  int m_tiles, n_tiles, kblocks;
  int n_fast;         // tile order: 1 = consecutive tiles share the activation rows
  const float* sx;    // [K/128][M]
  const float* sw;    // [ceil(N/128)][K/128]
  uint16_t* Y;
  int64_t ldy;
  uint32_t* err;
};

// 10 warps put three on some SM sub-partitions, whose register file holds
// 16K registers, so 168 per thread is the most this block can launch with.
__global__ void __maxnreg__(168)
    gemm_fp8_block_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const BlockParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kBM * kBK;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * kBN * kBK);
  // full[S], empty[S], pfull[NP], pempty[NP], drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 2 * kNP + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + kStages + s); };
  auto pfull = [&](int b) { return smem_u32(bars + 2 * kStages + b); };
  auto pempty = [&](int b) { return smem_u32(bars + 2 * kStages + kNP + b); };
  const uint32_t drain = smem_u32(bars + 2 * kStages + 2 * kNP);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < kNP; ++b) {
      mbar_init(pfull(b), 1);
      mbar_init(pempty(b), kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
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
  pdl_wait();      // inputs of this call may come from the previous kernel
  const int tiles = p.m_tiles * p.n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_a = policy_evict_last();
      const uint64_t pol_b = policy_evict_last();
      uint32_t stage = 0, phase = 0, issued = 0, issued_par = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int mt = p.n_fast ? t / p.n_tiles : t % p.m_tiles, nt = p.n_fast ? t % p.n_tiles : t / p.m_tiles;
        for (int kb = 0; kb < p.kblocks; ++kb) {
          if (!mbar_wait(empty(stage), phase ^ 1u, p.err, 0x301u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(full(stage), kStageBytes);
          tma_load_2d(smem_u32(sA + stage * kBM * kBK), &tmA, full(stage), kb * kBK, mt * kBM, pol_a);
          tma_load_2d(smem_u32(sB + stage * kBN * kBK), &tmB, full(stage), kb * kBK, nt * kBN, pol_b);
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
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, pb = 0, pphase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        for (int kb = 0; kb < p.kblocks; ++kb) {
          if (!mbar_wait(pempty(pb), pphase ^ 1u, p.err, 0x302u, abort_flag)) { ok = false; break; }
          if (!mbar_wait(full(stage), phase, p.err, 0x303u, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem_base + pb * kBN;
          const uint32_t a0 = smem_u32(sA + stage * kBM * kBK);
          const uint32_t b0 = smem_u32(sB + stage * kBN * kBK);
#pragma unroll
          for (int k = 0; k < kBK / 32; ++k)
            mma_f8f6f4(d, smem_desc(a0 + k * 32, 16, 1024, 2), smem_desc(b0 + k * 32, 16, 1024, 2), kIdesc,
                       k > 0 ? 1u : 0u);
          tc_commit(empty(stage));
          tc_commit(pfull(pb));
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
          if (++pb == kNP) { pb = 0; pphase ^= 1u; }
        }
      }
      tc_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, nullptr, 0, &no_abort);
    }
  } else {
    // epilogue / promotion: thread = one output row, 128 of the 256 columns
    // (one 128-column weight block, so one weight scale per K group)
    const int quarter = warp & 3;             // lane quarter this warp may read
    const int half = (warp - 2) / 4;          // column half of the tile
    const int row_in_tile = quarter * 32 + lane;
    const int nb_count = (p.N + 127) / 128;
    uint32_t pb = 0, pphase = 0;
    bool ok = true;
    GemmParams ep{};
    ep.I = p.M;
    ep.J = p.N;
    ep.Y = p.Y;
    ep.ldy = p.ldy;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
      const int mt = p.n_fast ? t / p.n_tiles : t % p.m_tiles, nt = p.n_fast ? t % p.n_tiles : t / p.m_tiles;
      const int m = mt * kBM + row_in_tile;
      const bool row_ok = m < p.M;
      const int nb = nt * 2 + half;
      const bool nb_ok = nb < nb_count;
      float acc[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
      // the group's two scales are loaded one group ahead, so their latency
      // overlaps the previous group's promotion instead of preceding it
      float sxv = row_ok ? __ldg(p.sx + m) : 0.0f;
      float swv = nb_ok ? __ldg(p.sw + static_cast<int64_t>(nb) * p.kblocks) : 0.0f;
      for (int kb = 0; kb < p.kblocks; ++kb) {
        const float c = __fmul_rn(sxv, swv);
        if (kb + 1 < p.kblocks) {
          sxv = row_ok ? __ldg(p.sx + static_cast<int64_t>(kb + 1) * p.M + m) : 0.0f;
          swv = nb_ok ? __ldg(p.sw + static_cast<int64_t>(nb) * p.kblocks + kb + 1) : 0.0f;
        }
        if (!warp_wait(pfull(pb), pphase, p.err, 0x304u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t taddr = tmem_base + pb * kBN + half * 128 + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[c0 + j] = __fmaf_rn(__uint_as_float(r[j]), c, acc[c0 + j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pempty(pb));
        if (++pb == kNP) { pb = 0; pphase ^= 1u; }
      }
      if (!ok) break;
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = acc[c0 + j];
        epilogue_store<32>(ep, m, nt * kBN + half * 128 + c0, v);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace

lpq_status launch_fp8_block(const CUtensorMap& tmA, const CUtensorMap& tmB, int64_t M, int64_t N, int64_t K,
                            const float* sx, const float* sw, uint16_t* Y, int64_t ldy, cudaStream_t st) {
  static uint64_t done_mask = 0;
  lpq_status s = ensure_smem_attr(reinterpret_cast<const void*>(&gemm_fp8_block_kernel), kSmemBytes, &done_mask);
  if (s != LPQ_OK) return s;
  static int max_threads = 0;
  if (max_threads == 0) {
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(&gemm_fp8_block_kernel));
    if (e != cudaSuccess) return record_cuda(e);
    max_threads = fa.maxThreadsPerBlock;
  }
  if (max_threads < kThreads) return record_cuda(cudaErrorLaunchOutOfResources);
  BlockParams p{};
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.m_tiles = static_cast<int>((M + kBM - 1) / kBM);
  p.n_tiles = static_cast<int>((N + kBN - 1) / kBN);
  p.kblocks = static_cast<int>(K / kBK);
  p.n_fast = j_fastest(M, N, K, 1.0) ? 1 : 0;
  p.sx = sx;
  p.sw = sw;
  p.Y = Y;
  p.ldy = ldy;
  p.err = error_word_ptr();
  const int grid = std::min(p.m_tiles * p.n_tiles, sm_count());
  return launch_pdl(gemm_fp8_block_kernel, dim3(grid), dim3(kThreads), kSmemBytes, st, 1, tmA, tmB, p);
}

}  // namespace lpq
