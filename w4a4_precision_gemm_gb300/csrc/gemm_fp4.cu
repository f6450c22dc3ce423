// gemm_fp4.cu - W4A4 GEMM on the block-scaled FP4 tensor-core path:
//   NVFP4: E2M1 x E2M1, one E4M3 scale per 16 elements (scale_vec::4X),
//          epilogue y = acc * g_x * g_w (the fp32 tensor scales);
//   MXFP4: E2M1 x E2M1, one E8M0 scale per 32 elements (scale_vec::2X).
// "FP8 and FP4 inference, SmoothQuant and activation quantization", sections
// "The bottleneck" (FP4 doubles the rate again over FP8), "Scale granularity"
// and "Implementation sketch" (nvfp4); "Low-bit LLM Weights and Activations",
// section 2.4.
//
// Same warp roles as the FP8 kernel.  Per pipeline stage the producer loads a
// 128 x 256 (A) and BN x 256 (B) tile of packed nibbles (one 128-byte
// swizzled row each) plus the matching scale-factor tiles (512-byte blocks of
// 128 rows x 4 scales, the layout the quantizers write) with bulk copies.
// The block-scaled MMA reads the scales of A row m from tensor-memory lane m,
// column (slot + m / 32), and the scales of B row n from every lane quarter
// (lane n % 32 of the quarter, column slot + 4 (n / 128) + (n % 128) / 32): in
// each quarter lane i, column 4 g + c holds row 128 g + 32 c + i, i.e. every
// 512-byte atom replicated into the four quarters.  Four scale-staging warps
// (one per lane quarter) write that layout with tcgen05.st from shared
// memory, so the MMA thread issues nothing but the four K=64 block-scaled
// MMAs of a stage: a tcgen05.cp of each atom, issued by the MMA thread, took
// about as long as the MMAs themselves.  (Staging them in the epilogue warps
// instead stalled the next tile's MMAs behind the previous tile's stores.)
// The staging warps arrive on the stage's full barrier (count 1 + 4), so the
// MMA thread waits once per stage: its per-stage bookkeeping sits on the
// critical path of the 4-stage ring.
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>

#include "gemm_common.cuh"
#include "gemm_fp8.h"
#include "internal.h"
#include "ptx.cuh"

namespace lpq {
namespace {

constexpr int kThreads = 320;      // TMA, MMA, 4 epilogue warps, 4 scale-staging warps
constexpr int kBM = 128;
constexpr int kBKBytes = 128;        // 256 packed E2M1 elements per row per stage
constexpr int kKPerStage = 256;
constexpr int kAtom = 512;           // 128 rows x 4 scale bytes

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

template <int BN, bool NV>
struct Fp4Cfg {
  static constexpr int kBlk = NV ? 16 : 32;                    // elements per scale
  static constexpr int kAtomsPerStage = kKPerStage / kBlk / 4;  // NV 4, MX 2 (per 128 rows)
  static constexpr int kBGroups = BN / 128;                     // 128-row groups of B (1 or 2)
  static constexpr int kSfaBytes = kAtomsPerStage * kAtom;
  static constexpr int kSfbBytes = kBGroups * kAtomsPerStage * kAtom;
  static constexpr int kStageBytes = (kBM + BN) * kBKBytes + kSfaBytes + kSfbBytes;
  static constexpr int kStages = cmin(8, (222 * 1024) / kStageBytes);
  // tensor-memory columns: accumulators (two when they fit next to the scale
  // slots, so the epilogue of one tile overlaps the next tile's K loop; one
  // for 256-wide tiles) + per-stage scale slots (4 columns per atom)
  static constexpr int kSfaCols = kAtomsPerStage * 4;
  static constexpr int kSfbCols = kBGroups * kAtomsPerStage * 4;
  static constexpr int kSfCols = kStages * (kSfaCols + kSfbCols);
  static constexpr int kAccBufs = (2 * BN + kSfCols <= 512) ? 2 : 1;
  static constexpr int kNeedCols = kAccBufs * BN + kSfCols;
  static constexpr int kTmemCols = kNeedCols <= 32 ? 32 : kNeedCols <= 64 ? 64 : kNeedCols <= 128 ? 128
                                   : kNeedCols <= 256 ? 256 : 512;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256;
  // block-scaled instruction descriptor: E2M1 x E2M1 (1), K-major, N, M = 128,
  // scale type UE4M3 (0, NVFP4) or UE8M0 (1, MXFP4); scale-data ids set per MMA
  static constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                                     ((NV ? 0u : 1u) << 23) | (static_cast<uint32_t>(kBM >> 4) << 24);
};
static_assert(Fp4Cfg<128, true>::kNeedCols <= 512, "tensor memory budget");
static_assert(Fp4Cfg<256, true>::kNeedCols <= 512 && Fp4Cfg<256, false>::kNeedCols <= 512, "tensor memory budget");
static_assert(Fp4Cfg<256, true>::kSmemBytes <= 227 * 1024, "shared memory budget");

// Epilogue of a whole tile that frees tensor memory before it writes Y: each
// lane converts its row of the 128 x BN accumulator, y = acc * (g_x g_w)
// (NVFP4) or acc (MXFP4), into BN / 2 registers of packed bf16, the warp
// releases the accumulator (arrives on `tempty`), and only then stores the
// row, so the next tile's MMAs run under the stores.  (With one accumulator
// per CTA the MMAs otherwise wait for the stores, and the CTAs, which finish
// tiles at about the same time, all store at once.)
template <int BN>
__device__ __forceinline__ void epilogue_tile_release_first(const GemmParams& p, const Seg& w, uint32_t tmem_acc,
                                                            int quarter, int lane, uint32_t tempty_bar) {
  const uint32_t taddr = tmem_acc + (static_cast<uint32_t>(quarter * 32) << 16);
  const int i = w.i_tile * 128 + quarter * 32 + lane;
  const bool scaled = p.gx != nullptr;
  const float g = scaled ? __fmul_rn(__ldg(p.gx), __ldg(p.gw)) : 1.0f;
  uint32_t y[BN / 2];
#pragma unroll
  for (int c = 0; c < BN; c += 32) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr + c, r);
    tmem_ld_wait();
#pragma unroll
    for (int t = 0; t < 32; t += 2) {
      const float a = __uint_as_float(r[t]), b = __uint_as_float(r[t + 1]);
      y[(c + t) / 2] = scaled ? pack_bf16x2(__fmul_rn(a, g), __fmul_rn(b, g)) : pack_bf16x2(a, b);
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(tempty_bar);
  if (i >= p.I) return;
  const int jt = w.j_tile * BN;
  uint16_t* yrow = p.Y + static_cast<int64_t>(i) * p.ldy + jt;
  const int n = p.J - jt;   // columns of this tile inside Y
  if (n >= BN) {
#pragma unroll
    for (int c = 0; c < BN; c += 8)
      *reinterpret_cast<uint4*>(yrow + c) = make_uint4(y[c / 2], y[c / 2 + 1], y[c / 2 + 2], y[c / 2 + 3]);
  } else {
#pragma unroll
    for (int c = 0; c < BN; c += 2) {
      if (c + 1 < n) {
        *reinterpret_cast<uint32_t*>(yrow + c) = y[c / 2];
      } else if (c < n) {
        yrow[c] = static_cast<uint16_t>(y[c / 2]);
      }
    }
  }
}

// 10 warps put three on two SM sub-partitions, whose register file holds 16K
// registers: 168 per thread is the most this block can launch with.
template <int BN, bool NV>
__global__ void __maxnreg__(168)
    gemm_fp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const uint8_t* __restrict__ sfa, const uint8_t* __restrict__ sfb, int64_t sf_kb4,
                    const GemmParams p) {
  using C = Fp4Cfg<BN, NV>;
  static_assert(BN == 256 && C::kAtomsPerStage % 2 == 0, "scale staging assumes two B groups, atom pairs");
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * kBM * kBKBytes;
  uint8_t* sSFA = sB + S * BN * kBKBytes;
  uint8_t* sSFB = sSFA + S * C::kSfaBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sSFB + S * C::kSfbBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + S + s); };
  auto tfull = [&](int a) { return smem_u32(bars + 2 * S + a); };
  auto tempty = [&](int a) { return smem_u32(bars + 2 * S + 2 + a); };
  const uint32_t drain = smem_u32(bars + 2 * S + 4);
  // full[s] completes when the operand tiles have landed (TMA bytes) and the
  // four staging warps have put the stage's scales into tensor memory
  auto sff = [&](int s) { return smem_u32(bars + 2 * S + 5 + s); };   // scales of stage s in shared memory

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1 + 4);
      mbar_init(empty(s), 1);
      mbar_init(sff(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull(a), 1);
      mbar_init(tempty(a), 4);
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
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_launch();
  pdl_wait();      // inputs of this call may come from the previous kernel
  // MMA k-steps (64 elements) in the last, possibly partial, stage
  const int ksteps_total = (p.K + 63) / 64;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_a = p.transposed ? policy_evict_first() : policy_evict_last();
      const uint64_t pol_b = p.transposed ? policy_evict_last() : policy_evict_first();
      uint32_t stage = 0, phase = 0, issued = 0, issued_par = 0;
      bool ok = true;
      WorkIter wi(p, blockIdx.x, gridDim.x);
      Seg w;
      while (ok && wi.next(p, blockIdx.x, gridDim.x, w)) {
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait(empty(stage), phase ^ 1u, p.err, 0x201u, abort_flag)) { ok = false; break; }
          // scale atoms of this stage that exist (a partial last stage has fewer)
          const int ksteps = min(4, ksteps_total - kb * 4);
          const int atoms = NV ? ksteps : (ksteps + 1) / 2;
          const uint32_t sf_bytes = atoms * kAtom;
          // 128-row groups of this B tile that exist in the scale buffer
          const int bgroups = min(C::kBGroups, (p.J + 127) / 128 - w.j_tile * C::kBGroups);
          // the scale tiles first, on their own barrier: the staging warps
          // move them into tensor memory while the operand tiles are in flight
          const int64_t atom0 = static_cast<int64_t>(kb) * C::kAtomsPerStage;
          mbar_arrive_expect_tx(sff(stage), sf_bytes * (1 + bgroups));
          bulk_g2s(smem_u32(sSFA + stage * C::kSfaBytes), sfa + (w.i_tile * sf_kb4 + atom0) * kAtom, sf_bytes,
                   sff(stage));
#pragma unroll
          for (int g = 0; g < C::kBGroups; ++g)
            if (g < bgroups)
              bulk_g2s(smem_u32(sSFB + stage * C::kSfbBytes + g * C::kSfaBytes),
                     sfb + ((w.j_tile * C::kBGroups + g) * sf_kb4 + atom0) * kAtom, sf_bytes, sff(stage));
          mbar_arrive_expect_tx(full(stage), (kBM + BN) * kBKBytes);
          tma_load_2d(smem_u32(sA + stage * kBM * kBKBytes), &tmA, full(stage), kb * kBKBytes, w.i_tile * kBM, pol_a);
          tma_load_2d(smem_u32(sB + stage * BN * kBKBytes), &tmB, full(stage), kb * kBKBytes, w.j_tile * BN, pol_b);
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        volatile int no_abort = 0;
        for (int s = 0; s < S; ++s)
          if (issued & (1u << s)) {
            mbar_wait(sff(s), (issued_par >> s) & 1u, nullptr, 0, &no_abort);
            mbar_wait(full(s), (issued_par >> s) & 1u, nullptr, 0, &no_abort);
          }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      const uint32_t sf_base = tmem_base + C::kAccBufs * BN;
      // operand descriptors of stage 0; a stage / a K step moves the start
      // address (bytes >> 4, 14 bits, shared memory stays below 256 KB)
      const uint64_t ad0 = smem_desc(smem_u32(sA), 16, 1024, 2);
      const uint64_t bd0 = smem_desc(smem_u32(sB), 16, 1024, 2);
      constexpr uint64_t kAStage = (kBM * kBKBytes) >> 4, kBStage = (BN * kBKBytes) >> 4, kKStep = 32 >> 4;
      auto mma = [&](uint32_t d, uint64_t ad, uint64_t bd, uint32_t tsfa, uint32_t tsfb, int k, uint32_t acc_in) {
        if constexpr (NV) {
          mma_nvf4(d, ad + k * kKStep, bd + k * kKStep, C::kIdesc, tsfa + k * 4, tsfb + k * 4 * C::kBGroups, acc_in);
        } else {
          const uint32_t id = static_cast<uint32_t>((k & 1) * 2);
          mma_mxf4(d, ad + k * kKStep, bd + k * kKStep, C::kIdesc | (id << 4) | (id << 29), tsfa + (k >> 1) * 4,
                   tsfb + (k >> 1) * 4 * C::kBGroups, acc_in);
        }
      };
      WorkIter wi(p, blockIdx.x, gridDim.x);
      Seg w;
      while (ok && wi.next(p, blockIdx.x, gridDim.x, w)) {
        if (!mbar_wait(tempty(acc), acc_phase ^ 1u, p.err, 0x202u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait(full(stage), phase, p.err, 0x203u, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t tsfa = sf_base + stage * (C::kSfaCols + C::kSfbCols);
          const uint32_t tsfb = tsfa + C::kSfaCols;
          const uint64_t ad = ad0 + stage * kAStage, bd = bd0 + stage * kBStage;
          const uint32_t first = kb > w.kb0 ? 1u : 0u;
          if (kb * 4 + 4 <= ksteps_total) {
#pragma unroll
            for (int k = 0; k < 4; ++k) mma(d, ad, bd, tsfa, tsfb, k, k > 0 ? 1u : first);
          } else {
            // last stage of a K not a multiple of 256: fewer K steps
            const int ksteps = ksteps_total - kb * 4;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (k < ksteps) mma(d, ad, bd, tsfa, tsfb, k, k > 0 ? 1u : first);
          }
          tc_commit(empty(stage));
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(tfull(acc));
        if (++acc == C::kAccBufs) { acc = 0; acc_phase ^= 1u; }
      }
      tc_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, nullptr, 0, &no_abort);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    uint32_t acc = 0, acc_phase = 0;
    WorkIter wi(p, blockIdx.x, gridDim.x);
    Seg w;
    while (wi.next(p, blockIdx.x, gridDim.x, w)) {
      if (!warp_wait(tfull(acc), acc_phase, p.err, 0x204u, abort_flag)) break;
      tc_fence_after();
      if (w.full) {
        epilogue_tile_release_first<BN>(p, w, tmem_base + acc * BN, quarter, lane, tempty(acc));
      } else {
        epilogue_tile<BN>(p, w, tmem_base + acc * BN, quarter, lane);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty(acc));
      }
      if (++acc == C::kAccBufs) { acc = 0; acc_phase ^= 1u; }
    }
  } else {
    // ------------------------------------------------------ scale staging
    // warps 6..9, one per lane quarter: every stage's scale tiles from shared
    // memory into this warp's quarter of the stage's tensor-memory slot
    const int quarter = warp & 3;
    const uint32_t sf_lanes = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + C::kAccBufs * BN;
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    WorkIter wi(p, blockIdx.x, gridDim.x);
    Seg w;
    while (ok && wi.next(p, blockIdx.x, gridDim.x, w)) {
      for (int kb = w.kb0; kb < w.kb1; ++kb) {
        if (!warp_wait(sff(stage), phase, p.err, 0x205u, abort_flag)) { ok = false; break; }
        // atom a of A -> columns 4a..4a+3; atom a of B group g -> columns 8a + 4g..+3
        // (lane i gets bytes 16 i..16 i + 15 of the atom); atoms past the end
        // of K were not loaded and are never read by an MMA
        const uint32_t tsfa = sf_lanes + stage * (C::kSfaCols + C::kSfbCols);
        const uint32_t tsfb = tsfa + C::kSfaCols;
        const uint8_t* a_src = sSFA + stage * C::kSfaBytes + lane * 16;
        const uint8_t* b_src = sSFB + stage * C::kSfbBytes + lane * 16;
#pragma unroll
        for (int a = 0; a < C::kAtomsPerStage; a += 2)
          tmem_st_32x32b_x8(tsfa + a * 4, *reinterpret_cast<const uint4*>(a_src + a * kAtom),
                            *reinterpret_cast<const uint4*>(a_src + (a + 1) * kAtom));
#pragma unroll
        for (int a = 0; a < C::kAtomsPerStage; ++a)
          tmem_st_32x32b_x8(tsfb + a * 8, *reinterpret_cast<const uint4*>(b_src + a * kAtom),
                            *reinterpret_cast<const uint4*>(b_src + C::kSfaBytes + a * kAtom));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(full(stage));
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::kTmemCols);
}

template <int BN, bool NV>
lpq_status launch_fp4_t(const CUtensorMap& tmA, const CUtensorMap& tmB, const uint8_t* sfa, const uint8_t* sfb,
                        int64_t kb4, const GemmParams& p, int grid, cudaStream_t st) {
  using C = Fp4Cfg<BN, NV>;
  static uint64_t done_mask = 0;
  lpq_status s = ensure_smem_attr(reinterpret_cast<const void*>(&gemm_fp4_kernel<BN, NV>), C::kSmemBytes, &done_mask);
  if (s != LPQ_OK) return s;
  s = launch_pdl(gemm_fp4_kernel<BN, NV>, dim3(grid), dim3(kThreads), C::kSmemBytes, st, 1, tmA, tmB, sfa, sfb, kb4, p);
  if (s != LPQ_OK || p.tail_s <= 1) return s;
  return launch_tail_reduce<BN>(p, st);
}

}  // namespace

// FP4 plan: 128 x 256 tiles on the natural operands (no swap; the scale
// layouts of A and B are the same 128-row tiles).  A 256-wide tile doubles
// the MMA work per scale copy of A and per staged byte of A over a 128-wide
// one; the price is a single tensor-memory accumulator (the epilogue does not
// overlap the next tile).  Whole tiles in waves, the last partial wave split
// along K when a workspace is given.
Fp8Plan plan_fp4(int64_t M, int64_t N, int64_t K, bool have_ws, size_t ws_bytes) {
  Fp8Plan pl{};
  pl.transposed = 0;
  pl.bn = 256;
  pl.I = M;
  pl.J = N;
  pl.kblocks = static_cast<int>((K + kKPerStage - 1) / kKPerStage);
  finish_plan(pl, have_ws, ws_bytes);
  return pl;
}

lpq_status launch_fp4(bool nv, const Fp8Plan& pl, const CUtensorMap& tmA, const CUtensorMap& tmB, const uint8_t* sfa,
                      const uint8_t* sfb, int64_t K, GemmParams p, void* ws, cudaStream_t st) {
  apply_plan(pl, p, ws);
  p.transposed = 0;
  p.j_fast = j_fastest(pl.I, pl.J, K, 0.5) ? 1 : 0;
  const int64_t kb4 = (K / (nv ? 16 : 32) + 3) / 4;
  if (nv) return launch_fp4_t<256, true>(tmA, tmB, sfa, sfb, kb4, p, pl.grid, st);
  return launch_fp4_t<256, false>(tmA, tmB, sfa, sfb, kb4, p, pl.grid, st);
}

}  // namespace lpq
