// gemm_fp8.h - host-side planning and launch of the tcgen05 GEMM kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/lpq.h"
#include "gemm_common.cuh"

namespace lpq {

constexpr int cmin(int a, int b) { return a < b ? a : b; }

// Tiling of one FP8 (or FP4) GEMM call.
struct Fp8Plan {
  int transposed;     // swap-AB: weights on the tensor core's M side
  int bn;             // N tile of the tensor core
  int64_t I, J;       // rows of the A / B operands
  int i_tiles, j_tiles, kblocks;
  int dp_tiles;       // tiles dealt whole, in waves of `grid`
  int tail_s;         // > 1: the other tiles split into this many K slices (needs a workspace)
  int ctas_per_sm;    // resident CTAs per SM the kernel is built for (grid = SMs x this)
  int csplit;         // > 1: K split across a cluster of this many CTAs (one tile per cluster)
  int kb_per_split;   // K blocks per slice (tail split or cluster rank)
  int grid;
};

Fp8Plan plan_fp8_rowscale(int64_t M, int64_t N, int64_t K, bool have_ws_budget, size_t ws_bytes);
// workspace a plan needs (0 without a tail split): one fp32 partial tile per
// tail slice
size_t plan_ws_bytes(const Fp8Plan& pl);
// fill in tile counts / tail split / grid for the given tiling
void finish_plan(Fp8Plan& pl, bool have_ws, size_t ws_bytes);
// copy a plan's decomposition into the kernel parameters
void apply_plan(const Fp8Plan& pl, GemmParams& p, void* ws);
lpq_status launch_fp8_rowscale(const Fp8Plan& pl, const CUtensorMap& tmA, const CUtensorMap& tmB, GemmParams p,
                               void* ws, cudaStream_t st, bool b_static = false);
// Tile visiting order for an [I x K] by [J x K] product (bytes per element of
// the operands given): consecutive tiles share the A rows (J fastest) when A
// is too large to stay in L2 while the B operand fits, so that every A row
// block is read from DRAM once and B is re-read from L2; otherwise they share
// the B rows (I fastest).
inline bool j_fastest(int64_t I, int64_t J, int64_t K, double bytes_per_elem) {
  const double a = static_cast<double>(I) * K * bytes_per_elem, b = static_cast<double>(J) * K * bytes_per_elem;
  constexpr double kL2Share = 64.0 * 1024 * 1024;   // half the L2
  return a > kL2Share && b <= kL2Share;
}

// Most tokens the fused-quantization GEMM takes (one 16-token swap-AB tile).
constexpr int64_t kFusedMaxTokens = 16;
// FP8 row-scaled GEMM with the activations' per-token quantization inside the
// kernel (p.xa / p.ldxa bf16, scales to p.sx_out); pl from plan_fp8_rowscale
// for at most kFusedMaxTokens tokens, tmW over the weights.
lpq_status launch_fp8_fused(const Fp8Plan& pl, const CUtensorMap& tmW, GemmParams p, cudaStream_t st, bool b_static);

// Output tile width of the block-scaled FP8 kernel (two 128-column weight blocks).
constexpr int kFp8BlockBN = 256;
lpq_status launch_fp8_block(const CUtensorMap& tmA, const CUtensorMap& tmB, int64_t M, int64_t N, int64_t K,
                            const float* sx, const float* sw, uint16_t* Y, int64_t ldy, cudaStream_t st);

// INT8 GEMM on the tcgen05 tensor cores through exact E4M3 digit planes
// (gemm_int8_tc.cu): the planes of both operands live in a workspace of
// int8_tc_workspace_bytes; K is limited so that every partial sum stays an
// exact fp32 integer.
constexpr int64_t kInt8TcMaxK = 65536;
size_t int8_tc_workspace_bytes(int64_t M, int64_t N, int64_t K, bool b_planes);
lpq_status launch_int8_tc(const int8_t* A, int64_t lda, const void* B, int64_t ldb, bool b_planes, int64_t M,
                          int64_t N, int64_t K, const float* sx, const float* sw, uint16_t* Y, int64_t ldy, void* ws,
                          cudaStream_t st);

lpq_status launch_int8(const CUtensorMap& tmA, const CUtensorMap& tmB, int64_t M, int64_t N, int64_t K,
                       const float* sx, const float* sw, uint16_t* Y, int64_t ldy, cudaStream_t st);

Fp8Plan plan_fp4(int64_t M, int64_t N, int64_t K, bool have_ws, size_t ws_bytes);
lpq_status launch_fp4(bool nv, const Fp8Plan& pl, const CUtensorMap& tmA, const CUtensorMap& tmB, const uint8_t* sfa,
                      const uint8_t* sfb, int64_t K, GemmParams p, void* ws, cudaStream_t st);

// Encode a 2-D tensor map over a row-major byte matrix [rows, row_bytes] with
// row stride ld_bytes, box = box_bytes x box_rows, 128-byte swizzle.
lpq_status make_tmap_u8(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes, int64_t ld_bytes,
                        int box_bytes, int box_rows, bool swizzle128);

// Set the dynamic shared memory limit of a kernel once per device.
lpq_status ensure_smem_attr(const void* func, int bytes, uint64_t* done_mask);

}  // namespace lpq
