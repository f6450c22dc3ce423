// gemm_common.cuh - pieces shared by the tcgen05 GEMM kernels: work-unit
// decoding (data-parallel tiles or stream-K ranges), the scale epilogue and
// the in-order combination of stream-K partial tiles.
//
// Every GEMM here computes D[i, j] = sum_k A[i, k] B[j, k] for a 128-row tile
// of the "A" operand (the tensor core's M side) and a BN-row tile of the "B"
// operand (its N side), accumulating in tensor memory.  With `transposed`
// set, A holds the weights and B the activations (swap-AB for small token
// counts) and the output is written as Y[j][i].
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace lpq {

struct GemmParams {
  int I, J, K;                 // rows of A, rows of B, reduction length (elements)
  int i_tiles, j_tiles;        // tiles of 128 rows of A, BN rows of B
  int kblocks;                 // K blocks (one pipeline stage each)
  int streamk;                 // 0: whole tiles round-robin; 1: equal K-iteration ranges per CTA
  int csplit;                  // > 1: cluster split-K, one (tile, K slice) per CTA, csplit CTAs per cluster
  int kb_per_split;            // K blocks per cluster rank
  int b_static;                // weights not written by the previous kernel: may be read before its end
  int j_fast;                  // tile order: 1 = consecutive tiles share the A rows (i), 0 = share B rows (j)
  int transposed;              // 0: Y[i][j], 1: Y[j][i]
  // epilogue scales: y = (acc * s_x) * s_w, s_x / s_w read from the i or j side
  const float* sx; int sx_stride;                // sx_stride 0: one scale for all
  const float* sw; int sw_stride;
  const float* gx; const float* gw;              // optional extra factors (NVFP4 g)
  uint16_t* Y; int64_t ldy;
  float* ws;                   // stream-K partials [grid][2][BN/4][128][4]
  int* counters;               // [tiles * 4], zero on entry, zero on exit
  uint32_t* err;
};

// A piece of work for one CTA: K blocks [kb0, kb1) of one output tile.
// `full` pieces cover the whole K range; the others are stream-K pieces whose
// partial sums are combined by the last of the tile's contributors.
struct Seg {
  int tile, i_tile, j_tile, kb0, kb1;
  bool full;
  int g_first, n_contrib, slot;
  // stream-K pieces: the tile's first leftover iteration and the leftover
  // iteration count; with fewer leftover iterations than CTAs some CTAs own
  // none, so contributor s of the tile is the owner of iteration sk_a + s
  int64_t sk_a, sk_T;
};

// Iterates the pieces of CTA `g` of `G`.  Whole tiles are dealt round-robin
// in waves of G (tiles g, g+G, ...: at any moment the CTAs work on G
// consecutive tiles, which share operand rows in L2).  In stream-K mode only
// the full waves are dealt that way; the K iterations of the leftover tiles
// (T = leftover tiles x kblocks, tile-major) are split into G equal,
// contiguous ranges [g T / G, (g+1) T / G), cut at tile boundaries.
struct WorkIter {
  int tile_rr, dp_tiles;
  int64_t it, end, T;
  __device__ __forceinline__ WorkIter(const GemmParams& p, int g, int G) {
    const int tiles = p.i_tiles * p.j_tiles;
    dp_tiles = p.streamk ? (tiles / G) * G : tiles;
    tile_rr = g;
    T = static_cast<int64_t>(tiles - dp_tiles) * p.kblocks;
    it = p.streamk ? (static_cast<int64_t>(g) * T) / G : 0;
    end = p.streamk ? (static_cast<int64_t>(g + 1) * T) / G : 0;
  }
  // CTA whose range holds leftover iteration x: the largest g with floor(g T / G) <= x
  __device__ __forceinline__ static int owner(int64_t x, int64_t T, int G) {
    return static_cast<int>(((x + 1) * G - 1) / T);
  }
  __device__ __forceinline__ bool next(const GemmParams& p, int g, int G, Seg& s) {
    if (p.csplit > 1) {
      // one piece per CTA: rank r of the cluster takes the r-th K slice of
      // tile g / csplit; the slices are summed through shared memory
      if (tile_rr < 0) return false;
      const int rank = g % p.csplit;
      s.tile = g / p.csplit;
      s.kb0 = rank * p.kb_per_split;
      s.kb1 = min(p.kblocks, s.kb0 + p.kb_per_split);
      tile_rr = -1;
      if (p.j_fast) {
        s.j_tile = s.tile % p.j_tiles;
        s.i_tile = s.tile / p.j_tiles;
      } else {
        s.i_tile = s.tile % p.i_tiles;
        s.j_tile = s.tile / p.i_tiles;
      }
      s.full = false;
      s.g_first = g - rank;
      s.n_contrib = p.csplit;
      s.slot = rank;
      return true;
    }
    if (tile_rr < dp_tiles) {
      s.tile = tile_rr;
      tile_rr += G;
      s.kb0 = 0;
      s.kb1 = p.kblocks;
    } else {
      if (it >= end) return false;
      const int t = static_cast<int>(it / p.kblocks);
      s.tile = dp_tiles + t;
      s.kb0 = static_cast<int>(it - static_cast<int64_t>(t) * p.kblocks);
      const int64_t left = end - it;
      s.kb1 = static_cast<int>(s.kb0 + left < p.kblocks ? s.kb0 + left : p.kblocks);
      it += s.kb1 - s.kb0;
    }
    if (p.j_fast) {
      s.j_tile = s.tile % p.j_tiles;
      s.i_tile = s.tile / p.j_tiles;
    } else {
      s.i_tile = s.tile % p.i_tiles;
      s.j_tile = s.tile / p.i_tiles;
    }
    s.full = (s.kb0 == 0 && s.kb1 == p.kblocks);
    s.g_first = g;
    s.n_contrib = 1;
    s.slot = 0;
    if (!s.full) {
      const int64_t a = static_cast<int64_t>(s.tile - dp_tiles) * p.kblocks;
      s.g_first = owner(a, T, G);
      s.sk_a = a;
      s.sk_T = T;
      // T >= G: every CTA owns at least one iteration, so the contributors
      // are consecutive; T < G: every CTA owns at most one, so there is one
      // contributor per iteration of the tile
      s.n_contrib = (T >= G) ? owner(a + p.kblocks - 1, T, G) - s.g_first + 1 : p.kblocks;
      // the first contributor's piece is the last of its range (slot 1); every
      // later contributor's piece is the first of its range (slot 0)
      s.slot = (g == s.g_first) ? 1 : 0;
    }
    return true;
  }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Scale and store N (<= 32) accumulators of row i, columns j0 .. j0+N-1:
// y = ((acc * s_x) * s_w) * (g_x * g_w), each factor only where given, fp32,
// rounded once to bf16.
__device__ __forceinline__ float scale_one(const GemmParams& p, float acc, float sx, float sw, float g) {
  float a = acc;
  if (p.sx) a = __fmul_rn(a, sx);
  if (p.sw) a = __fmul_rn(a, sw);
  if (p.gx) a = __fmul_rn(a, g);
  return a;
}

template <int N>
__device__ __forceinline__ void epilogue_store(const GemmParams& p, int i, int j0, const float (&v)[N]) {
  if (i >= p.I) return;
  const float g = p.gx ? __fmul_rn(__ldg(p.gx), __ldg(p.gw)) : 1.0f;
  if (!p.transposed) {
    // i = token row (x side), j = output channel (w side)
    const float sxi = p.sx ? __ldg(p.sx + static_cast<int64_t>(i) * p.sx_stride) : 1.0f;
    uint16_t* yrow = p.Y + static_cast<int64_t>(i) * p.ldy;
    if (j0 + N <= p.J) {
      uint32_t w[N / 2];
#pragma unroll
      for (int c = 0; c < N; c += 2) {
        const float swa = p.sw ? __ldg(p.sw + static_cast<int64_t>(j0 + c) * p.sw_stride) : 1.0f;
        const float swb = p.sw ? __ldg(p.sw + static_cast<int64_t>(j0 + c + 1) * p.sw_stride) : 1.0f;
        w[c / 2] = pack_bf16x2(scale_one(p, v[c], sxi, swa, g), scale_one(p, v[c + 1], sxi, swb, g));
      }
      if constexpr (N == 4) {
        *reinterpret_cast<uint2*>(yrow + j0) = make_uint2(w[0], w[1]);
      } else {
#pragma unroll
        for (int c = 0; c < N / 2; c += 4)
          *reinterpret_cast<uint4*>(yrow + j0 + 2 * c) = make_uint4(w[c], w[c + 1], w[c + 2], w[c + 3]);
      }
    } else {
#pragma unroll
      for (int c = 0; c < N; ++c) {
        if (j0 + c < p.J) {
          const float sw = p.sw ? __ldg(p.sw + static_cast<int64_t>(j0 + c) * p.sw_stride) : 1.0f;
          yrow[j0 + c] = __bfloat16_as_ushort(__float2bfloat16_rn(scale_one(p, v[c], sxi, sw, g)));
        }
      }
    }
  } else {
    // i = output channel (w side), j = token (x side): Y[j][i]
    const float swi = p.sw ? __ldg(p.sw + static_cast<int64_t>(i) * p.sw_stride) : 1.0f;
#pragma unroll
    for (int c = 0; c < N; ++c) {
      if (j0 + c < p.J) {
        const float sxj = p.sx ? __ldg(p.sx + static_cast<int64_t>(j0 + c) * p.sx_stride) : 1.0f;
        p.Y[static_cast<int64_t>(j0 + c) * p.ldy + i] =
            __bfloat16_as_ushort(__float2bfloat16_rn(scale_one(p, v[c], sxj, swi, g)));
      }
    }
  }
}

// Tensor-memory -> registers -> epilogue for one 128 x BN accumulator, by the
// four epilogue warps (warp q of the CTA reads lanes 32*(q%4) .. +31).  A full
// piece is scaled and stored; a stream-K piece writes its partial sums to its
// slot of the workspace.
template <int BN>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const Seg& w, uint32_t tmem_acc, int quarter,
                                              int lane, float* smem_part = nullptr) {
  constexpr int CW = (BN < 32) ? BN : 32;
  const int row_in_tile = quarter * 32 + lane;
  const int i = w.i_tile * 128 + row_in_tile;
  const uint32_t taddr = tmem_acc + (static_cast<uint32_t>(quarter * 32) << 16);
  // partial slot layout [BN/4][128][4]: for one group of 4 columns the 32
  // lanes of a warp touch 512 contiguous bytes (global stream-K slot, or this
  // CTA's shared-memory buffer for a cluster split)
  float* part = w.full ? nullptr
                : smem_part ? smem_part + row_in_tile * 4
                            : p.ws + (static_cast<int64_t>(blockIdx.x) * 2 + w.slot) * 128 * BN + row_in_tile * 4;
#pragma unroll 1
  for (int c = 0; c < BN; c += CW) {
    float v[CW];
    if constexpr (CW == 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(taddr + c, r);
      tmem_ld_wait();
#pragma unroll
      for (int t = 0; t < 32; ++t) v[t] = __uint_as_float(r[t]);
    } else {
      uint32_t r[16];
      tmem_ld_32x32b_x16(taddr + c, r);
      tmem_ld_wait();
#pragma unroll
      for (int t = 0; t < 16; ++t) v[t] = __uint_as_float(r[t]);
    }
    if (w.full) {
      epilogue_store<CW>(p, i, w.j_tile * BN + c, v);
    } else if (smem_part) {
#pragma unroll
      for (int t = 0; t < CW; t += 4)
        *reinterpret_cast<float4*>(part + ((c + t) / 4) * 512) = make_float4(v[t], v[t + 1], v[t + 2], v[t + 3]);
    } else {
#pragma unroll
      for (int t = 0; t < CW; t += 4)
        __stcg(reinterpret_cast<float4*>(part + static_cast<int64_t>((c + t) / 4) * 512),
               make_float4(v[t], v[t + 1], v[t + 2], v[t + 3]));
    }
  }
}

// Second half of a stream-K piece, run after the accumulator has been handed
// back to the MMA warp: count this quarter-tile in; the last contributor sums
// every contributor's partial in contributor order (a fixed order, so the
// result does not depend on which CTA finishes last) and stores the tile.
template <int BN>
__device__ __forceinline__ void streamk_finish(const GemmParams& p, const Seg& w, int quarter, int lane) {
  constexpr int kSub = 8;          // columns per reduction step
  constexpr int kBatch = 8;        // contributors whose loads are in flight together
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    const int old = atomicAdd(p.counters + w.tile * 4 + quarter, 1);
    last = (old == w.n_contrib - 1);
    if (last) p.counters[w.tile * 4 + quarter] = 0;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
  const int row_in_tile = quarter * 32 + lane;
  const int i = w.i_tile * 128 + row_in_tile;
  const int64_t row_off = static_cast<int64_t>(row_in_tile) * 4;
#pragma unroll 2
  for (int c = 0; c < BN; c += kSub) {
    float v[kSub];
#pragma unroll
    for (int t = 0; t < kSub; ++t) v[t] = 0.0f;
    for (int s0 = 0; s0 < w.n_contrib; s0 += kBatch) {
      float4 f[kBatch][2];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (s0 + b < w.n_contrib) {
          const int G = static_cast<int>(gridDim.x);
          const int g = (w.sk_T >= G) ? w.g_first + s0 + b : WorkIter::owner(w.sk_a + s0 + b, w.sk_T, G);
          const int slot = (s0 + b == 0) ? 1 : 0;
          const float* part = p.ws + (static_cast<int64_t>(g) * 2 + slot) * 128 * BN + row_off +
                              static_cast<int64_t>(c / 4) * 512;
          f[b][0] = __ldcg(reinterpret_cast<const float4*>(part));
          f[b][1] = __ldcg(reinterpret_cast<const float4*>(part + 512));
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (s0 + b < w.n_contrib) {
          v[0] += f[b][0].x; v[1] += f[b][0].y; v[2] += f[b][0].z; v[3] += f[b][0].w;
          v[4] += f[b][1].x; v[5] += f[b][1].y; v[6] += f[b][1].z; v[7] += f[b][1].w;
        }
      }
    }
    epilogue_store<kSub>(p, i, w.j_tile * BN + c, v);
  }
}

// Cluster split-K: after every CTA of the cluster has put its partial tile
// (layout [BN/4][128][4] fp32) in its own shared memory and the cluster has
// synchronised, CTA `rank` sums 1/csplit of the tile's float4 groups over all
// ranks in rank order (a fixed order) through distributed shared memory and
// stores them.  Run by the 128 epilogue threads (t = 0..127).
template <int BN>
__device__ __forceinline__ void cluster_reduce_store(const GemmParams& p, const Seg& w, uint32_t part_saddr, int t) {
  constexpr int F = 32 * BN;                    // float4 groups in the tile
  const int S = p.csplit;
  const int rank = w.slot;
  const int q0 = (rank * F) / S, q1 = ((rank + 1) * F) / S;
  for (int q = q0 + t; q < q1; q += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = 0; r < S; ++r) {
      const float4 v = ld_dsmem_f4(map_to_rank(part_saddr + q * 16, static_cast<uint32_t>(r)));
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    const int c4 = q / 128, row = q % 128;
    const float v4[4] = {acc.x, acc.y, acc.z, acc.w};
    epilogue_store<4>(p, w.i_tile * 128 + row, w.j_tile * BN + 4 * c4, v4);
  }
}

}  // namespace lpq
