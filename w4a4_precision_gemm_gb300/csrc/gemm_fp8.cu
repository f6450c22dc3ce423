// gemm_fp8.cu - FP8 E4M3 x E4M3 GEMM on the 5th-generation tensor cores with
// per-row scales applied in the epilogue:
//   Y = diag(s_X) (X_q W_q^T) diag(s_W)     (fp32 accumulation, bf16 out)
// "FP8 and FP4 inference, SmoothQuant and activation quantization", section
// "Scale granularity"; "FP8 and INT8 Inference", sections 5 and 6-9 (the
// epilogue: acc *= s_a x s_b, store bf16).
//
// Structure (one CTA per SM, persistent over work units):
//   warp 0      TMA producer: 128-byte-swizzled A / B tiles into a STAGES-deep
//               shared-memory ring (mbarrier full/empty pairs);
//   warp 1      allocates tensor memory and issues tcgen05.mma (one thread),
//               accumulating a 128 x BN fp32 tile into one of two TMEM
//               buffers, so the epilogue of tile t overlaps the K loop of t+1;
//   warps 2-5   epilogue: tcgen05.ld -> scales -> bf16 -> global (or, for a
//               K slice, fp32 partial sums: to shared memory for a cluster
//               split, summed over the cluster; to the workspace for a split
//               tail tile, summed by the tail-reduction kernel).
// Every barrier wait is bounded (a timeout sets the device error word and the
// kernel winds down); no trap, no unbounded spin.
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>

#include "gemm_common.cuh"
#include "gemm_fp8.h"
#include "internal.h"
#include "ptx.cuh"

namespace lpq {
namespace {

constexpr int kThreads = 192;
constexpr int kBM = 128;
constexpr int kBKBytes = 128;   // one 128-byte swizzle row of K per stage

template <int BN>
struct Fp8Cfg {
  // small token tiles (decode): two CTAs share an SM (two independent TMA
  // streams per SM, and one CTA's epilogue overlaps the other's loads)
  static constexpr int kCtasPerSm = (BN <= 64) ? 2 : 1;
  static constexpr int kStageBytes = (kBM + BN) * kBKBytes;
  static constexpr int kStages = cmin(12, (kCtasPerSm == 2 ? 108 * 1024 : 200 * 1024) / kStageBytes);
  static constexpr int kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
  // instruction descriptor: D fp32, A/B E4M3, K-major both, N = BN, M = 128
  static constexpr uint32_t kIdesc =
      (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(kBM >> 4) << 24);
};

static_assert(Fp8Cfg<64>::kCtasPerSm == 2 && Fp8Cfg<128>::kCtasPerSm == 1, "planner assumes 2 CTAs/SM for BN <= 64");
static_assert(2 * Fp8Cfg<64>::kSmemBytes <= 227 * 1024, "two CTAs must fit one SM's shared memory");
static_assert(2 * Fp8Cfg<16>::kSmemBytes <= 227 * 1024, "two CTAs must fit one SM's shared memory");

// FQ: fused activation quantization (swap-AB with BN = 16 only): operand B
// is not loaded by TMA; the epilogue warps, idle during the K loop, compute
// the tokens' scales and write every stage's E4M3 token tile into shared
// memory themselves.
template <int BN, bool FQ = false>
__global__ void __launch_bounds__(kThreads, Fp8Cfg<BN>::kCtasPerSm)
    gemm_fp8_rowscale_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const GemmParams p) {
  static_assert(!FQ || BN == 16, "fused quantization: 16-token tiles, 8 threads per token");
  using C = Fp8Cfg<BN>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * kBM * kBKBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + S * BN * kBKBytes);
  // bars: full[S], empty[S], tfull[2], tempty[2], drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // fused quantization: per-rank partial maxima [8][BN] (fp32 bits) and the
  // tokens' scales [BN] (kFqExtraBytes of shared memory past the barriers)
  uint32_t* fq_amax = reinterpret_cast<uint32_t*>(bars + 2 * S + 6);   // [8][BN] per rank
  float* fq_scale = reinterpret_cast<float*>(fq_amax + 8 * BN);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + S + s); };
  auto tfull = [&](int a) { return smem_u32(bars + 2 * S + a); };
  auto tempty = [&](int a) { return smem_u32(bars + 2 * S + 2 + a); };
  const uint32_t drain = smem_u32(bars + 2 * S + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), FQ ? 5 : 1);      // FQ: + one arrival per token-writing warp
      mbar_init(empty(s), 1);
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
  if constexpr (FQ) {
    // every CTA of the cluster is running before any writes into a peer's
    // shared memory (the exchange of the tokens' partial maxima)
    if (p.csplit > 1) cluster_sync();
  }
  // Inputs of this call may come from the previous kernel on the stream:
  // every thread waits for it before touching global memory, except the TMA
  // thread when the weights are declared static, which first starts the
  // weight stream of its opening stages (see the producer below).
  const bool early_w = p.b_static && warp == 0 && lane == 0;
  if (!early_w) {
    pdl_launch();
    pdl_wait();
  }

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    // (lane 0 issues; the other lanes only join the cluster barrier of a
    // fused quantization)
    constexpr uint32_t kTx = FQ ? kBM * kBKBytes : C::kStageBytes;   // FQ: B is written by the epilogue warps
    const uint64_t pol_a = p.transposed ? policy_evict_first() : policy_evict_last();
    const uint64_t pol_b = p.transposed ? policy_evict_last() : policy_evict_first();
    uint32_t stage = 0, phase = 0;
    uint32_t issued = 0, issued_par = 0;   // per-stage: issued at least once / parity of last issue
    bool ok = true;
    WorkIter wi(p, blockIdx.x, gridDim.x);
    Seg w;
    // static weights: claim the first (still free) stages and start their
    // weight tiles before waiting for the previous kernel; the token tiles of
    // those stages follow after the wait
    int pre = 0;
    if (lane == 0 && early_w) {
      WorkIter wi2 = wi;
      Seg w2;
      bool h2 = wi2.next(p, blockIdx.x, gridDim.x, w2);
      int kb2 = h2 ? w2.kb0 : 0;
      while (h2 && pre < S) {
        mbar_arrive_expect_tx(full(pre), kTx);
        if (p.transposed)
          tma_load_2d(smem_u32(sA + pre * kBM * kBKBytes), &tmA, full(pre), kb2 * kBKBytes, w2.i_tile * kBM, pol_a);
        else
          tma_load_2d(smem_u32(sB + pre * BN * kBKBytes), &tmB, full(pre), kb2 * kBKBytes, w2.j_tile * BN, pol_b);
        ++pre;
        if (++kb2 == w2.kb1) {
          h2 = wi2.next(p, blockIdx.x, gridDim.x, w2);
          if (h2) kb2 = w2.kb0;
        }
      }
      pdl_launch();
      pdl_wait();
    }
    if constexpr (FQ) {
      __syncwarp();
      if (p.csplit > 1) cluster_sync();    // exchange of the tokens' partial maxima
    }
    if (lane == 0) {
      int n = 0;                              // stages handled so far
      while (ok && wi.next(p, blockIdx.x, gridDim.x, w)) {
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++n) {
          if (n < pre) {
            // weight tile already on its way; add the token tile
            if (!FQ) {
              if (p.transposed)
                tma_load_2d(smem_u32(sB + stage * BN * kBKBytes), &tmB, full(stage), kb * kBKBytes, w.j_tile * BN,
                            pol_b);
              else
                tma_load_2d(smem_u32(sA + stage * kBM * kBKBytes), &tmA, full(stage), kb * kBKBytes, w.i_tile * kBM,
                            pol_a);
            }
          } else {
            if (!mbar_wait(empty(stage), phase ^ 1u, p.err, 0x101u, abort_flag)) { ok = false; break; }
            mbar_arrive_expect_tx(full(stage), kTx);
            tma_load_2d(smem_u32(sA + stage * kBM * kBKBytes), &tmA, full(stage), kb * kBKBytes, w.i_tile * kBM, pol_a);
            if (!FQ)
              tma_load_2d(smem_u32(sB + stage * BN * kBKBytes), &tmB, full(stage), kb * kBKBytes, w.j_tile * BN, pol_b);
          }
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // let the copies already in flight land before the CTA leaves
        volatile int no_abort = 0;
        for (int s = 0; s < S; ++s)
          if (issued & (1u << s)) mbar_wait(full(s), (issued_par >> s) & 1u, nullptr, 0, &no_abort);
      }
    }
  } else if (warp == 1) {
    if constexpr (FQ) {
      if (p.csplit > 1) cluster_sync();    // exchange of the tokens' partial maxima
    }
    if (lane == 0) {
      // --------------------------------------------------------------- MMA
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      WorkIter wi(p, blockIdx.x, gridDim.x);
      Seg w;
      while (ok && wi.next(p, blockIdx.x, gridDim.x, w)) {
        if (!mbar_wait(tempty(acc), acc_phase ^ 1u, p.err, 0x102u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait(full(stage), phase, p.err, 0x103u, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * kBM * kBKBytes);
          const uint32_t b0 = smem_u32(sB + stage * BN * kBKBytes);
#pragma unroll
          for (int k = 0; k < kBKBytes / 32; ++k) {
            const uint64_t ad = smem_desc(a0 + k * 32, 16, 1024, 2);
            const uint64_t bd = smem_desc(b0 + k * 32, 16, 1024, 2);
            mma_f8f6f4(d, ad, bd, C::kIdesc, (kb > w.kb0 || k > 0) ? 1u : 0u);
          }
          tc_commit(empty(stage));
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(tfull(acc));
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      // wait for every MMA this thread issued before tensor memory is released
      tc_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, nullptr, 0, &no_abort);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int et = threadIdx.x - 64;            // 0 .. 127
    uint32_t acc = 0, acc_phase = 0;
    GemmParams pe = p;                          // FQ: scales from shared memory
    uint32_t pstage = 0, pphase = 0;            // FQ: ring position of the token tiles
    bool ok = true;
    if constexpr (FQ) {
      // ---- tokens' scales: s = max(max_k |x|, 1e-8) / 448, the per-token rule
      // of the standalone quantizer.  8 threads per token; a cluster split
      // takes each rank's K slice and exchanges the partial maxima.
      const int ntok = p.J;
      WorkIter wq(p, blockIdx.x, gridDim.x);
      Seg w0;
      const bool has = wq.next(p, blockIdx.x, gridDim.x, w0);
      int k0 = 0, k1 = p.K;
      if (p.csplit > 1 && has) {
        k0 = w0.kb0 * kBKBytes;
        k1 = min(p.K, w0.kb1 * kBKBytes);
      }
      // 8 threads per token (lanes 8g .. 8g+7 of a warp), 16-byte loads
      const int tok = et >> 3, sub = et & 7;
      float a = 0.0f;
      if (tok < ntok) {
        const uint16_t* xr = p.xa + static_cast<int64_t>(tok) * p.ldxa;
#pragma unroll 4
        for (int k = k0 + sub * 8; k < k1; k += 64) {
          const uint4 u = __ldg(reinterpret_cast<const uint4*>(xr + k));
          a = fmaxf(a, fmaxf(fmaxf(fmaxf(fabsf(bf16lo(u.x)), fabsf(bf16hi(u.x))), fmaxf(fabsf(bf16lo(u.y)), fabsf(bf16hi(u.y)))),
                             fmaxf(fmaxf(fabsf(bf16lo(u.z)), fabsf(bf16hi(u.z))), fmaxf(fabsf(bf16lo(u.w)), fabsf(bf16hi(u.w))))));
        }
      }
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
      const uint32_t rank = p.csplit > 1 ? cluster_ctarank() : 0u;
      if (sub == 0) {
        if (p.csplit > 1) {
          for (int r = 0; r < p.csplit; ++r)
            st_dsmem_u32(map_to_rank(smem_u32(fq_amax + rank * BN + tok), static_cast<uint32_t>(r)), __float_as_uint(a));
        } else {
          fq_amax[tok] = __float_as_uint(a);
        }
      }
      if (p.csplit > 1) {
        __syncwarp();
        cluster_sync();                         // every rank's maxima are in every rank
      } else {
        named_barrier_sync(1, 128);
      }
      if (et < BN) {
        float m = 0.0f;
        for (int r = 0; r < (p.csplit > 1 ? p.csplit : 1); ++r) m = fmaxf(m, __uint_as_float(fq_amax[r * BN + et]));
        const float sc = __fdiv_rn(fmaxf(m, 1e-8f), 448.0f);
        fq_scale[et] = sc;
        if (p.sx_out && et < ntok && has && w0.i_tile == 0 && rank == 0) p.sx_out[et] = sc;
      }
      named_barrier_sync(1, 128);
      pe.sx = fq_scale;
      pe.sx_plain = 1;
      pe.sx_stride = 1;
    }
    WorkIter wi(p, blockIdx.x, gridDim.x);
    Seg w;
    while (ok && wi.next(p, blockIdx.x, gridDim.x, w)) {
      if constexpr (FQ) {
        // ---- this piece's token tiles: 16 E4M3 codes per thread per stage,
        // written in the 128-byte-swizzled K-major layout a TMA load gives
        const int tok = et >> 3, c16 = et & 7;
        const float sc = fq_scale[tok];
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!warp_wait(empty(pstage), pphase ^ 1u, p.err, 0x105u, abort_flag)) { ok = false; break; }
          uint4 code = make_uint4(0u, 0u, 0u, 0u);
          const int k = kb * kBKBytes + c16 * 16;
          if (tok < p.J && k < p.K) {
            const uint16_t* xp = p.xa + static_cast<int64_t>(tok) * p.ldxa + k;
            const uint4 u0 = __ldg(reinterpret_cast<const uint4*>(xp));
            const uint4 u1 = __ldg(reinterpret_cast<const uint4*>(xp + 8));
            const uint32_t w32[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) h[i] = cvt_e4m3x2(__fdiv_rn(bf16lo(w32[i]), sc), __fdiv_rn(bf16hi(w32[i]), sc));
            code = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
          }
          uint8_t* dst = sB + pstage * BN * kBKBytes + tok * kBKBytes + ((c16 ^ (tok & 7)) << 4);
          *reinterpret_cast<uint4*>(dst) = code;
          fence_proxy_async_smem();             // visible to the tensor core's reads
          __syncwarp();
          if (lane == 0) mbar_arrive(full(pstage));
          if (++pstage == S) { pstage = 0; pphase ^= 1u; }
        }
        if (!ok) break;
      }
      if (!warp_wait(tfull(acc), acc_phase, p.err, 0x104u, abort_flag)) break;
      tc_fence_after();
      // a cluster split's partial goes to this CTA's (now idle) stage buffers
      epilogue_tile<BN>(FQ ? pe : p, w, tmem_base + acc * BN, quarter, lane,
                        p.csplit > 1 ? reinterpret_cast<float*>(sA) : nullptr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty(acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  }

  if (p.csplit > 1) {
    // every thread of the cluster takes part in both cluster barriers (also
    // after a timed-out wait), so no CTA can be left waiting at one; the warp
    // is reconverged first (the TMA and MMA lanes leave their loops later)
    __syncwarp();
    cluster_sync();                       // all partials written
    if (warp >= 2) {
      WorkIter wi(p, blockIdx.x, gridDim.x);
      Seg w;
      if (wi.next(p, blockIdx.x, gridDim.x, w)) {
        GemmParams pr = p;
        if (FQ) {
          pr.sx = fq_scale;
          pr.sx_plain = 1;
          pr.sx_stride = 1;
        }
        cluster_reduce_store<BN>(pr, w, smem_u32(sA), threadIdx.x - 64);
      }
    }
    __syncwarp();
    cluster_sync();                       // peers done reading this CTA's partial
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::kTmemCols);
}

constexpr int kFqExtraBytes = 1024;   // partial maxima and scales of a fused quantization
static_assert(2 * (Fp8Cfg<16>::kSmemBytes + kFqExtraBytes) <= 227 * 1024, "two fused CTAs must fit one SM");

template <int BN, bool FQ = false>
lpq_status launch_bn(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid, cudaStream_t st,
                     int cluster) {
  using C = Fp8Cfg<BN>;
  constexpr int kSmem = C::kSmemBytes + (FQ ? kFqExtraBytes : 0);
  static uint64_t done_mask = 0;
  lpq_status s = ensure_smem_attr(reinterpret_cast<const void*>(&gemm_fp8_rowscale_kernel<BN, FQ>), kSmem, &done_mask);
  if (s != LPQ_OK) return s;
  s = launch_pdl(gemm_fp8_rowscale_kernel<BN, FQ>, dim3(grid), dim3(kThreads), kSmem, st, cluster, tmA, tmB, p);
  if (s != LPQ_OK || p.tail_s <= 1) return s;
  return launch_tail_reduce<BN>(p, st);
}

// Clusters of `S` CTAs of the BN kernel that can be resident at once
// (cached per device, BN and S).
template <int BN>
int max_active_clusters_bn(int S) {
  using C = Fp8Cfg<BN>;
  static int cache[64][9] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || S < 1 || S > 8) return 0;
  if (cache[dev][S] != 0) return cache[dev][S] > 0 ? cache[dev][S] : 0;
  static uint64_t done_mask = 0;
  int n = 0;
  if (ensure_smem_attr(reinterpret_cast<const void*>(&gemm_fp8_rowscale_kernel<BN>), C::kSmemBytes, &done_mask) ==
      LPQ_OK) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S * 64);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_fp8_rowscale_kernel<BN>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
  }
  cache[dev][S] = n > 0 ? n : -1;
  return n;
}

int max_active_clusters(int bn, int S) {
  switch (bn) {
    case 16: return max_active_clusters_bn<16>(S);
    case 32: return max_active_clusters_bn<32>(S);
    case 64: return max_active_clusters_bn<64>(S);
    case 128: return max_active_clusters_bn<128>(S);
    case 256: return max_active_clusters_bn<256>(S);
    default: return 0;
  }
}

}  // namespace

// Tile choice: swap-AB (weights on the tensor core's M side) for <= 64
// tokens, N tile = the token count rounded up to a power of two >= 16 (two
// CTAs per SM).  More tokens: 128 x 256 tiles (from 65 to 256 tokens they
// stage each weight tile into shared memory once or twice, where 128-token
// swap-AB tiles would need 1/2 to 1/8 of the tensor rate per staged byte).
// Few tiles (at most a quarter of the CTA slots): K split 4 or 8 ways across
// a thread-block cluster whose CTAs add their partial sums through
// distributed shared memory.  Otherwise whole tiles in waves, the last partial wave split along
// K when a workspace is given (see finish_plan).
Fp8Plan plan_fp8_rowscale(int64_t M, int64_t N, int64_t K, bool have_ws_budget, size_t ws_bytes) {
  Fp8Plan pl{};
  pl.transposed = (M <= 64);
  pl.I = pl.transposed ? N : M;
  pl.J = pl.transposed ? M : N;
  int bn = 256;
  if (pl.transposed) {
    bn = 16;
    while (bn < pl.J && bn < 64) bn *= 2;
  }
  pl.bn = bn;
  pl.ctas_per_sm = (bn <= 64) ? 2 : 1;     // Fp8Cfg<bn>::kCtasPerSm
  pl.kblocks = static_cast<int>((K + kBKBytes - 1) / kBKBytes);
  pl.i_tiles = static_cast<int>((pl.I + kBM - 1) / kBM);
  pl.j_tiles = static_cast<int>((pl.J + pl.bn - 1) / pl.bn);
  const int64_t tiles = static_cast<int64_t>(pl.i_tiles) * pl.j_tiles;
  const int slots = sm_count() * pl.ctas_per_sm;
  pl.csplit = 1;
  pl.tail_s = 1;
  pl.dp_tiles = static_cast<int>(tiles);
  pl.kb_per_split = pl.kblocks;
  if (tiles * 4 <= slots && pl.kblocks >= 4) {
    // the widest power-of-two split (8 or 4: they pack evenly into the GPCs)
    // that keeps tiles x split within the CTA slots and whose clusters fit
    // on the GPU in at most two waves.  (A 2-way split measured slower than
    // whole tiles: half a tile's partial sums per CTA cross the cluster.)
    for (int S = 8; S >= 4; S /= 2) {
      if (tiles * S > slots || S > pl.kblocks) continue;
      const int fit = max_active_clusters(pl.bn, S);
      if (fit > 0 && tiles > 2 * fit) continue;   // (0: unknown / no device)
      pl.kb_per_split = (pl.kblocks + S - 1) / S;
      pl.csplit = (pl.kblocks + pl.kb_per_split - 1) / pl.kb_per_split;   // no empty slice
      break;
    }
    if (pl.csplit > 1) {
      pl.grid = static_cast<int>(tiles * pl.csplit);
      return pl;
    }
    pl.kb_per_split = pl.kblocks;
  }
  if (pl.transposed) {
    pl.grid = static_cast<int>(std::min<int64_t>(tiles, slots));
    return pl;
  }
  finish_plan(pl, have_ws_budget, ws_bytes);
  return pl;
}

// Whole tiles in waves of one CTA per slot.  The tiles of the last, partial
// wave leave CTAs idle; if at least twice as many CTAs as those tiles are
// available (and a workspace is given), each of them is cut into S <= 8
// equal K slices run by S CTAs, and a small reduction kernel adds the slices
// in a fixed order.
void finish_plan(Fp8Plan& pl, bool have_ws, size_t ws_bytes) {
  pl.i_tiles = static_cast<int>((pl.I + kBM - 1) / kBM);
  pl.j_tiles = static_cast<int>((pl.J + pl.bn - 1) / pl.bn);
  const int64_t tiles = static_cast<int64_t>(pl.i_tiles) * pl.j_tiles;
  const int slots = sm_count() * (pl.ctas_per_sm > 0 ? pl.ctas_per_sm : 1);
  pl.csplit = 1;
  pl.kb_per_split = pl.kblocks;
  pl.tail_s = 1;
  pl.dp_tiles = static_cast<int>(tiles);
  pl.grid = static_cast<int>(std::min<int64_t>(tiles, slots));
  const int64_t left = tiles % slots;
  if (!have_ws || left == 0) return;
  int S = static_cast<int>(std::min<int64_t>(8, slots / left));
  S = std::min(S, pl.kblocks);
  if (S < 2) return;
  Fp8Plan t = pl;
  t.kb_per_split = (pl.kblocks + S - 1) / S;
  t.tail_s = (pl.kblocks + t.kb_per_split - 1) / t.kb_per_split;   // no empty slice
  t.dp_tiles = static_cast<int>(tiles - left);
  t.grid = static_cast<int>(tiles >= slots ? slots : left * t.tail_s);
  if (plan_ws_bytes(t) <= ws_bytes) pl = t;
}

size_t plan_ws_bytes(const Fp8Plan& pl) {
  if (pl.tail_s <= 1) return 0;
  const size_t pieces = static_cast<size_t>(static_cast<int64_t>(pl.i_tiles) * pl.j_tiles - pl.dp_tiles) * pl.tail_s;
  return pieces * 128 * pl.bn * sizeof(float);
}

void apply_plan(const Fp8Plan& pl, GemmParams& p, void* ws) {
  p.I = static_cast<int>(pl.I);
  p.J = static_cast<int>(pl.J);
  p.i_tiles = pl.i_tiles;
  p.j_tiles = pl.j_tiles;
  p.kblocks = pl.kblocks;
  p.dp_tiles = pl.dp_tiles;
  p.tail_s = pl.tail_s;
  p.csplit = pl.csplit;
  p.kb_per_split = pl.kb_per_split;
  p.transposed = pl.transposed;
  p.ws = pl.tail_s > 1 ? static_cast<float*>(ws) : nullptr;
}

lpq_status launch_fp8_rowscale(const Fp8Plan& pl, const CUtensorMap& tmA, const CUtensorMap& tmB, GemmParams p,
                               void* ws, cudaStream_t st, bool b_static) {
  apply_plan(pl, p, ws);
  p.j_fast = pl.transposed ? 1 : (j_fastest(pl.I, pl.J, p.K, 1.0) ? 1 : 0);
  p.b_static = b_static ? 1 : 0;
  switch (pl.bn) {
    case 16: return launch_bn<16>(tmA, tmB, p, pl.grid, st, pl.csplit);
    case 32: return launch_bn<32>(tmA, tmB, p, pl.grid, st, pl.csplit);
    case 64: return launch_bn<64>(tmA, tmB, p, pl.grid, st, pl.csplit);
    case 128: return launch_bn<128>(tmA, tmB, p, pl.grid, st, pl.csplit);
    case 256: return launch_bn<256>(tmA, tmB, p, pl.grid, st, pl.csplit);
    default: return LPQ_ERR_UNSUPPORTED;
  }
}

lpq_status launch_fp8_fused(const Fp8Plan& pl, const CUtensorMap& tmW, GemmParams p, cudaStream_t st, bool b_static) {
  if (!pl.transposed || pl.bn != 16 || pl.tail_s > 1) return LPQ_ERR_UNSUPPORTED;
  apply_plan(pl, p, nullptr);
  p.j_fast = 1;
  p.b_static = b_static ? 1 : 0;
  return launch_bn<16, true>(tmW, tmW, p, pl.grid, st, pl.csplit);
}

}  // namespace lpq
