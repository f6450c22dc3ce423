// gemm_common.cuh - pieces shared by the tcgen05 GEMM kernels: work-unit
// decoding (whole tiles in waves, split tail tiles, cluster split-K), the
// scale epilogue and the in-order combination of partial tiles.
//
// Every GEMM here computes D[i, j] = sum_k A[i, k] B[j, k] for a 128-row tile
// of the "A" operand (the tensor core's M side) and a BN-row tile of the "B"
// operand (its N side), accumulating in tensor memory.  With `transposed`
// set, A holds the weights and B the activations (swap-AB for small token
// counts) and the output is written as Y[j][i].
#pragma once
#include <cuda_bf16.h>
#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace lpq {

struct GemmParams {
  int I, J, K;                 // rows of A, rows of B, reduction length (elements)
  int i_tiles, j_tiles;        // tiles of 128 rows of A, BN rows of B
  int kblocks;                 // K blocks (one pipeline stage each)
  int dp_tiles;                // tiles dealt whole, round-robin in waves of gridDim.x
  int tail_s;                  // > 1: the remaining tiles are split into tail_s K slices, one per CTA
  int csplit;                  // > 1: cluster split-K, one (tile, K slice) per CTA, csplit CTAs per cluster
  int kb_per_split;            // K blocks per slice (tail split or cluster rank)
  int b_static;                // weights not written by the previous kernel: may be read before its end
  int j_fast;                  // tile order: 1 = consecutive tiles share the A rows (i), 0 = share B rows (j)
  int transposed;              // 0: Y[i][j], 1: Y[j][i]
  // epilogue scales: y = (acc * s_x) * s_w, s_x / s_w read from the i or j side
  const float* sx; int sx_stride;                // sx_stride 0: one scale for all
  int sx_plain;                                  // sx points to shared memory (plain loads)
  const float* sw; int sw_stride;
  const float* gx; const float* gw;              // optional extra factors (NVFP4 g)
  uint16_t* Y; int64_t ldy;
  // fused activation quantization (swap-AB, <= 16 tokens): bf16 activations
  // [J][ldxa] quantized per token inside the kernel; scales written to sx_out
  const uint16_t* xa; int64_t ldxa; float* sx_out;
  float* ws;                   // tail-split partials [tail tiles * tail_s][BN/4][128][4]
  uint32_t* err;
};

// A piece of work for one CTA: K blocks [kb0, kb1) of one output tile.
// `full` pieces cover the whole K range; the others are K slices whose
// partial sums are combined later (by the cluster, or by the tail-reduction
// kernel); `slot` is the slice's cluster rank or its tail piece index.
struct Seg {
  int tile, i_tile, j_tile, kb0, kb1;
  bool full;
  int slot;
};

// Iterates the pieces of CTA `g` of `G`.  Whole tiles are dealt round-robin
// in waves of G (tiles g, g+G, ...: at any moment the CTAs work on G
// consecutive tiles, which share operand rows in L2).  The tiles past
// dp_tiles (fewer than G) are each cut into tail_s K slices; CTA g takes
// tail piece g (tile dp_tiles + g / tail_s, slice g % tail_s) after its
// whole tiles.  With a cluster split every CTA has exactly one piece.
struct WorkIter {
  int tile_rr, tail_piece;
  __device__ __forceinline__ WorkIter(const GemmParams& p, int g, int G) {
    (void)G;
    tile_rr = g;
    const int tail_tiles = p.i_tiles * p.j_tiles - p.dp_tiles;
    tail_piece = (p.tail_s > 1 && g < tail_tiles * p.tail_s) ? g : -1;
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
      s.full = false;
      s.slot = rank;
    } else if (tile_rr < p.dp_tiles) {
      s.tile = tile_rr;
      tile_rr += G;
      s.kb0 = 0;
      s.kb1 = p.kblocks;
      s.full = true;
      s.slot = 0;
    } else if (tail_piece >= 0) {
      s.tile = p.dp_tiles + tail_piece / p.tail_s;
      s.kb0 = (tail_piece % p.tail_s) * p.kb_per_split;
      s.kb1 = min(p.kblocks, s.kb0 + p.kb_per_split);
      s.full = false;
      s.slot = tail_piece;
      tail_piece = -1;
    } else {
      return false;
    }
    if (p.j_fast) {
      s.j_tile = s.tile % p.j_tiles;
      s.i_tile = s.tile / p.j_tiles;
    } else {
      s.i_tile = s.tile % p.i_tiles;
      s.j_tile = s.tile / p.i_tiles;
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

// Activation scale of token t (p.sx non-null): a global array, or the
// kernel's own shared-memory copy when the quantization is fused.
__device__ __forceinline__ float token_scale(const GemmParams& p, int64_t t) {
  const int64_t k = t * p.sx_stride;
  return p.sx_plain ? p.sx[k] : __ldg(p.sx + k);
}

template <int N>
__device__ __forceinline__ void epilogue_store(const GemmParams& p, int i, int j0, const float (&v)[N]) {
  if (i >= p.I) return;
  const float g = p.gx ? __fmul_rn(__ldg(p.gx), __ldg(p.gw)) : 1.0f;
  if (!p.transposed) {
    // i = token row (x side), j = output channel (w side)
    const float sxi = p.sx ? token_scale(p, i) : 1.0f;
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
        const float sxj = p.sx ? token_scale(p, j0 + c) : 1.0f;
        p.Y[static_cast<int64_t>(j0 + c) * p.ldy + i] =
            __bfloat16_as_ushort(__float2bfloat16_rn(scale_one(p, v[c], sxj, swi, g)));
      }
    }
  }
}

// Tensor-memory -> registers -> epilogue for one 128 x BN accumulator, by the
// four epilogue warps (warp q of the CTA reads lanes 32*(q%4) .. +31).  A full
// piece is scaled and stored; a K slice writes its partial sums to its slot
// (this CTA's shared memory for a cluster split, else the workspace).
template <int BN>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const Seg& w, uint32_t tmem_acc, int quarter,
                                              int lane, float* smem_part = nullptr) {
  constexpr int CW = (BN < 32) ? BN : 32;
  const int row_in_tile = quarter * 32 + lane;
  const int i = w.i_tile * 128 + row_in_tile;
  const uint32_t taddr = tmem_acc + (static_cast<uint32_t>(quarter * 32) << 16);
  // partial slot layout [BN/4][128][4]: for one group of 4 columns the 32
  // lanes of a warp touch 512 contiguous bytes
  float* part = w.full ? nullptr
                : smem_part ? smem_part + row_in_tile * 4
                            : p.ws + static_cast<int64_t>(w.slot) * 128 * BN + row_in_tile * 4;
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

// Tail reduction (its own launch, after the GEMM): sums the tail_s partial
// tiles of every split tail tile in slice order (a fixed order) and applies
// the epilogue.  One thread per (tail tile, row, group of 4 columns); the
// 32 lanes of a warp read 512 contiguous bytes of each slice.
template <int BN>
__global__ void __launch_bounds__(256) tail_reduce_kernel(const GemmParams p) {
  pdl_launch();
  pdl_wait();
  constexpr int kQ = 128 * (BN / 4);            // float4 groups per tile
  const int tail_tiles = p.i_tiles * p.j_tiles - p.dp_tiles;
  const int64_t total = static_cast<int64_t>(tail_tiles) * kQ;
  for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < total;
       q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(q / kQ);
    const int r = static_cast<int>(q % kQ);
    const int c4 = r / 128, row = r % 128;
    const float* base = p.ws + static_cast<int64_t>(t) * p.tail_s * 128 * BN + c4 * 512 + row * 4;
    float4 v[8];
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (s < p.tail_s) v[s] = __ldcg(reinterpret_cast<const float4*>(base + static_cast<int64_t>(s) * 128 * BN));
    float4 acc = v[0];
#pragma unroll
    for (int s = 1; s < 8; ++s) {
      if (s < p.tail_s) {
        acc.x += v[s].x; acc.y += v[s].y; acc.z += v[s].z; acc.w += v[s].w;
      }
    }
    const int tile = p.dp_tiles + t;
    const int i_tile = p.j_fast ? tile / p.j_tiles : tile % p.i_tiles;
    const int j_tile = p.j_fast ? tile % p.j_tiles : tile / p.i_tiles;
    const float v4[4] = {acc.x, acc.y, acc.z, acc.w};
    epilogue_store<4>(p, i_tile * 128 + row, j_tile * BN + 4 * c4, v4);
  }
}

// Enqueue the tail reduction for a plan with a tail split (after the GEMM on
// the same stream; programmatic launch lets it wait for the GEMM's end).
template <int BN>
lpq_status launch_tail_reduce(const GemmParams& p, cudaStream_t st) {
  const int64_t total = static_cast<int64_t>(p.i_tiles * p.j_tiles - p.dp_tiles) * 128 * (BN / 4);
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(sm_count()) * 8);
  return launch_pdl(tail_reduce_kernel<BN>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1, p);
}

// Cluster split-K: after every CTA of the cluster has put its partial tile
// (layout [BN/4][128][4] fp32) in its own shared memory and the cluster has
// synchronised, CTA `rank` sums 1/csplit of the tile's float4 groups over all
// ranks in rank order (a fixed order) through distributed shared memory and
// stores them.  Run by the 128 epilogue threads (t = 0..127).
template <int BN>
__device__ __forceinline__ void cluster_reduce_store(const GemmParams& p, const Seg& w, uint32_t part_saddr, int t) {
  constexpr int F = 32 * BN;                    // float4 groups in the tile
  constexpr int U = 2;                          // groups per thread per pass
  const int S = p.csplit;                       // 2 .. 8
  const int rank = w.slot;
  const int q0 = (rank * F) / S, q1 = ((rank + 1) * F) / S;
  for (int qb = q0 + t; qb < q1; qb += 128 * U) {
    // every rank's copy of U groups is requested before any is used
    float4 v[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = qb + u * 128;
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (q < q1 && r < S) v[u][r] = ld_dsmem_f4(map_to_rank(part_saddr + q * 16, static_cast<uint32_t>(r)));
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = qb + u * 128;
      if (q >= q1) break;
      float4 acc = v[u][0];
#pragma unroll
      for (int r = 1; r < 8; ++r) {
        if (r < S) {
          acc.x += v[u][r].x; acc.y += v[u][r].y; acc.z += v[u][r].z; acc.w += v[u][r].w;
        }
      }
      const int c4 = q / 128, row = q % 128;
      const float v4[4] = {acc.x, acc.y, acc.z, acc.w};
      epilogue_store<4>(p, w.i_tile * 128 + row, w.j_tile * BN + 4 * c4, v4);
    }
  }
}

}  // namespace lpq
