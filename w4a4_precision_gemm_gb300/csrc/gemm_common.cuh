// gemm_common.cuh - pieces shared by the tcgen05 GEMM kernels: work-unit
// decoding, the scale epilogue and the split-K reduction.
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
  int splits, kb_per_split;    // split-K
  int transposed;              // 0: Y[i][j], 1: Y[j][i]
  // epilogue scales: y = (acc * s_x) * s_w, s_x / s_w read from the i or j side
  const float* sx; int sx_stride;                // sx_stride 0: one scale for all
  const float* sw; int sw_stride;
  const float* gx; const float* gw;              // optional extra factors (NVFP4 g)
  uint16_t* Y; int64_t ldy;
  float* ws;                   // split-K partials [tiles * splits][128][BN]
  int* counters;               // [tiles * 4], zero on entry, zero on exit
  uint32_t* err;
};

struct Unit {
  int tile, split, i_tile, j_tile, kb0, kb1;
};

__device__ __forceinline__ Unit decode_unit(const GemmParams& p, int u) {
  Unit w;
  w.tile = u / p.splits;
  w.split = u - w.tile * p.splits;
  w.i_tile = w.tile % p.i_tiles;
  w.j_tile = w.tile / p.i_tiles;
  w.kb0 = w.split * p.kb_per_split;
  w.kb1 = min(p.kblocks, w.kb0 + p.kb_per_split);
  return w;
}

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
#pragma unroll
      for (int c = 0; c < N / 2; c += 4)
        *reinterpret_cast<uint4*>(yrow + j0 + 2 * c) = make_uint4(w[c], w[c + 1], w[c + 2], w[c + 3]);
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
// four epilogue warps (warp q of the CTA reads lanes 32*(q%4) .. +31).
// Without split-K the result is scaled and stored; with split-K the partial is
// written to the workspace and the last of the splits of this tile (per
// 32-row quarter) sums all partials in split order and stores the result.
template <int BN>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const Unit& w, uint32_t tmem_acc, int quarter,
                                              int lane) {
  constexpr int CW = (BN < 32) ? BN : 32;
  const int row_in_tile = quarter * 32 + lane;
  const int i = w.i_tile * 128 + row_in_tile;
  const uint32_t taddr = tmem_acc + (static_cast<uint32_t>(quarter * 32) << 16);
  if (p.splits == 1) {
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
      epilogue_store<CW>(p, i, w.j_tile * BN + c, v);
    }
    return;
  }
  // split-K: write this split's partial
  float* part = p.ws + ((static_cast<int64_t>(w.tile) * p.splits + w.split) * 128 + row_in_tile) * BN;
#pragma unroll 1
  for (int c = 0; c < BN; c += CW) {
    if constexpr (CW == 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(taddr + c, r);
      tmem_ld_wait();
#pragma unroll
      for (int t = 0; t < 32; t += 4)
        __stcg(reinterpret_cast<float4*>(part + c + t),
               make_float4(__uint_as_float(r[t]), __uint_as_float(r[t + 1]), __uint_as_float(r[t + 2]),
                           __uint_as_float(r[t + 3])));
    } else {
      uint32_t r[16];
      tmem_ld_32x32b_x16(taddr + c, r);
      tmem_ld_wait();
#pragma unroll
      for (int t = 0; t < 16; t += 4)
        __stcg(reinterpret_cast<float4*>(part + c + t),
               make_float4(__uint_as_float(r[t]), __uint_as_float(r[t + 1]), __uint_as_float(r[t + 2]),
                           __uint_as_float(r[t + 3])));
    }
  }
}

// Second half of the split-K epilogue, run after the accumulator has been
// handed back to the MMA warp.
template <int BN>
__device__ __forceinline__ void splitk_finish(const GemmParams& p, const Unit& w, int quarter, int lane) {
  constexpr int CW = (BN < 32) ? BN : 32;
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    const int old = atomicAdd(p.counters + w.tile * 4 + quarter, 1);
    last = (old == p.splits - 1);
    if (last) p.counters[w.tile * 4 + quarter] = 0;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
  const int row_in_tile = quarter * 32 + lane;
  const int i = w.i_tile * 128 + row_in_tile;
#pragma unroll 1
  for (int c = 0; c < BN; c += CW) {
    float v[CW];
#pragma unroll
    for (int t = 0; t < CW; ++t) v[t] = 0.0f;
#pragma unroll 1
    for (int s = 0; s < p.splits; ++s) {
      const float* part = p.ws + ((static_cast<int64_t>(w.tile) * p.splits + s) * 128 + row_in_tile) * BN + c;
#pragma unroll
      for (int t = 0; t < CW; t += 4) {
        const float4 f = __ldcg(reinterpret_cast<const float4*>(part + t));
        v[t] += f.x; v[t + 1] += f.y; v[t + 2] += f.z; v[t + 3] += f.w;
      }
    }
    epilogue_store<CW>(p, i, w.j_tile * BN + c, v);
  }
}

}  // namespace lpq
