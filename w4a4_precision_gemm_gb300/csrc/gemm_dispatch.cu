// gemm_dispatch.cu - validation and dispatch of lpq_gemm_scaled.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/lpq.h"
#include "gemm_fp8.h"
#include "internal.h"

using namespace lpq;

namespace {

bool is_fp8_rowscale(const lpq_gemm_desc* d) {
  return d->fmt == LPQ_FMT_FP8 && (d->a_gran == LPQ_GRAN_ROW || d->a_gran == LPQ_GRAN_TENSOR_STATIC) &&
         d->b_gran == LPQ_GRAN_ROW;
}

lpq_status validate_common(const lpq_gemm_desc* d, int64_t kmult, int64_t ld_mult) {
  LPQ_CHECK_NULL(d);
  LPQ_CHECK_NULL(d->A);
  LPQ_CHECK_NULL(d->B);
  LPQ_CHECK_NULL(d->Y);
  if (d->M <= 0 || d->N <= 0 || d->K <= 0 || d->K % kmult != 0) return LPQ_ERR_SHAPE;
  if (d->M > 0x7FFFFFFFLL || d->N > 0x7FFFFFFFLL || d->K > 0x7FFFFFFFLL) return LPQ_ERR_SHAPE;
  if (d->lda < d->K || d->ldb < d->K || d->ldy < d->N) return LPQ_ERR_SHAPE;
  if (d->lda % ld_mult != 0 || d->ldb % ld_mult != 0 || d->ldy % 8 != 0) return LPQ_ERR_ALIGN;
  LPQ_CHECK_ALIGN(d->A);
  LPQ_CHECK_ALIGN(d->B);
  LPQ_CHECK_ALIGN(d->Y);
  if (d->workspace && !aligned16(d->workspace)) return LPQ_ERR_ALIGN;
  return LPQ_OK;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

// LPQ_GEMM_A_BF16: A is bf16 and is quantized per token by the call itself:
// inside the GEMM kernel for at most kFusedMaxTokens tokens, else into the
// workspace by the standalone quantizer followed by the ordinary GEMM.
lpq_status gemm_fp8_rowscale(const lpq_gemm_desc* d, cudaStream_t st);

lpq_status gemm_fp8_a_bf16(const lpq_gemm_desc* d, cudaStream_t st) {
  lpq_status s = validate_common(d, 16, 16);
  if (s != LPQ_OK) return s;
  if (d->a_gran != LPQ_GRAN_ROW) return LPQ_ERR_UNSUPPORTED;
  LPQ_CHECK_NULL(d->sa);
  LPQ_CHECK_NULL(d->sb);
  if ((reinterpret_cast<uintptr_t>(d->sa) & 3u) != 0) return LPQ_ERR_ALIGN;
  const bool b_static = (d->flags & LPQ_GEMM_B_STATIC) != 0;
  if (d->M <= kFusedMaxTokens) {
    const Fp8Plan pl = plan_fp8_rowscale(d->M, d->N, d->K, false, 0);
    CUtensorMap tmW;
    if ((s = make_tmap_u8(&tmW, d->B, pl.I, d->K, d->ldb, 128, 128, true)) != LPQ_OK) return s;
    GemmParams p{};
    p.K = static_cast<int>(d->K);
    p.sw = static_cast<const float*>(d->sb);
    p.sw_stride = 1;
    p.xa = static_cast<const uint16_t*>(d->A);
    p.ldxa = d->lda;
    p.sx_out = const_cast<float*>(static_cast<const float*>(d->sa));
    p.Y = d->Y;
    p.ldy = d->ldy;
    p.err = error_word_ptr();
    return launch_fp8_fused(pl, tmW, p, st, b_static);
  }
  const size_t codes = align256(static_cast<size_t>(d->M) * static_cast<size_t>(d->K));
  if (!d->workspace || d->workspace_bytes < codes) return LPQ_ERR_WORKSPACE;
  uint8_t* xq = static_cast<uint8_t*>(d->workspace);
  s = lpq_quantize_act_fp8(static_cast<const uint16_t*>(d->A), d->M, d->K, d->lda, LPQ_GRAN_ROW, xq,
                           const_cast<float*>(static_cast<const float*>(d->sa)), st);
  if (s != LPQ_OK) return s;
  lpq_gemm_desc q = *d;
  q.A = xq;
  q.lda = d->K;
  q.flags = d->flags & ~LPQ_GEMM_A_BF16;
  q.workspace = d->workspace_bytes > codes ? xq + codes : nullptr;
  q.workspace_bytes = d->workspace_bytes - codes;
  return gemm_fp8_rowscale(&q, st);
}

lpq_status gemm_fp8_rowscale(const lpq_gemm_desc* d, cudaStream_t st) {
  if (d && (d->flags & LPQ_GEMM_A_BF16)) return gemm_fp8_a_bf16(d, st);
  lpq_status s = validate_common(d, 16, 16);
  if (s != LPQ_OK) return s;
  LPQ_CHECK_NULL(d->sa);
  LPQ_CHECK_NULL(d->sb);
  const Fp8Plan pl = plan_fp8_rowscale(d->M, d->N, d->K, d->workspace != nullptr, d->workspace_bytes);
  // operand A of the tensor core: X (normal) or W (swap-AB)
  const void* opA = pl.transposed ? d->B : d->A;
  const void* opB = pl.transposed ? d->A : d->B;
  const int64_t ldA = pl.transposed ? d->ldb : d->lda;
  const int64_t ldB = pl.transposed ? d->lda : d->ldb;
  CUtensorMap tmA, tmB;
  if ((s = make_tmap_u8(&tmA, opA, pl.I, d->K, ldA, 128, 128, true)) != LPQ_OK) return s;
  if ((s = make_tmap_u8(&tmB, opB, pl.J, d->K, ldB, 128, pl.bn, true)) != LPQ_OK) return s;
  GemmParams p{};
  p.K = static_cast<int>(d->K);
  p.sx = static_cast<const float*>(d->sa);
  p.sx_stride = (d->a_gran == LPQ_GRAN_TENSOR_STATIC) ? 0 : 1;
  p.sw = static_cast<const float*>(d->sb);
  p.sw_stride = 1;
  p.Y = d->Y;
  p.ldy = d->ldy;
  p.err = error_word_ptr();
  return launch_fp8_rowscale(pl, tmA, tmB, p, d->workspace, st, (d->flags & LPQ_GEMM_B_STATIC) != 0);
}

bool is_fp8_block(const lpq_gemm_desc* d) {
  return d->fmt == LPQ_FMT_FP8 && d->a_gran == LPQ_GRAN_BLOCK_1x128 && d->b_gran == LPQ_GRAN_BLOCK_128x128;
}

lpq_status gemm_fp8_block(const lpq_gemm_desc* d, cudaStream_t st) {
  lpq_status s = validate_common(d, 128, 16);
  if (s != LPQ_OK) return s;
  LPQ_CHECK_NULL(d->sa);
  LPQ_CHECK_NULL(d->sb);
  CUtensorMap tmA, tmB;
  if ((s = make_tmap_u8(&tmA, d->A, d->M, d->K, d->lda, 128, 128, true)) != LPQ_OK) return s;
  if ((s = make_tmap_u8(&tmB, d->B, d->N, d->K, d->ldb, 128, kFp8BlockBN, true)) != LPQ_OK) return s;
  return launch_fp8_block(tmA, tmB, d->M, d->N, d->K, static_cast<const float*>(d->sa),
                          static_cast<const float*>(d->sb), d->Y, d->ldy, st);
}

bool is_int8(const lpq_gemm_desc* d) {
  return d->fmt == LPQ_FMT_INT8 && d->a_gran == LPQ_GRAN_ROW && d->b_gran == LPQ_GRAN_ROW;
}

lpq_status gemm_int8(const lpq_gemm_desc* d, cudaStream_t st) {
  lpq_status s = validate_common(d, 16, 16);
  if (s != LPQ_OK) return s;
  LPQ_CHECK_NULL(d->sa);
  LPQ_CHECK_NULL(d->sb);
  // with a workspace for the digit planes: the tcgen05 path
  const bool planes = (d->flags & LPQ_GEMM_B_INT8_PLANES) != 0;
  if (d->workspace && d->K <= kInt8TcMaxK && d->workspace_bytes >= int8_tc_workspace_bytes(d->M, d->N, d->K, planes))
    return launch_int8_tc(static_cast<const int8_t*>(d->A), d->lda, d->B, d->ldb, planes, d->M, d->N, d->K,
                          static_cast<const float*>(d->sa), static_cast<const float*>(d->sb), d->Y, d->ldy,
                          d->workspace, st);
  if (planes) return d->K <= kInt8TcMaxK ? LPQ_ERR_WORKSPACE : LPQ_ERR_SHAPE;   // planes need the tensor-core path
  CUtensorMap tmA, tmB;
  if ((s = make_tmap_u8(&tmA, d->A, d->M, d->K, d->lda, 128, 128, true)) != LPQ_OK) return s;
  if ((s = make_tmap_u8(&tmB, d->B, d->N, d->K, d->ldb, 128, 128, true)) != LPQ_OK) return s;
  return launch_int8(tmA, tmB, d->M, d->N, d->K, static_cast<const float*>(d->sa), static_cast<const float*>(d->sb),
                     d->Y, d->ldy, st);
}

bool is_fp4(const lpq_gemm_desc* d) { return d->fmt == LPQ_FMT_NVFP4 || d->fmt == LPQ_FMT_MXFP4; }

lpq_status gemm_fp4(const lpq_gemm_desc* d, cudaStream_t st) {
  // element strides; two E2M1 codes per byte, byte strides a multiple of 16
  lpq_status s = validate_common(d, 32, 32);
  if (s != LPQ_OK) return s;
  const bool nv = d->fmt == LPQ_FMT_NVFP4;
  LPQ_CHECK_NULL(d->sa);
  LPQ_CHECK_NULL(d->sb);
  LPQ_CHECK_ALIGN(d->sa);
  LPQ_CHECK_ALIGN(d->sb);
  if (nv) {
    LPQ_CHECK_NULL(d->ga);
    LPQ_CHECK_NULL(d->gb);
  }
  const Fp8Plan pl = plan_fp4(d->M, d->N, d->K, d->workspace != nullptr, d->workspace_bytes);
  CUtensorMap tmA, tmB;
  if ((s = make_tmap_u8(&tmA, d->A, d->M, d->K / 2, d->lda / 2, 128, 128, true)) != LPQ_OK) return s;
  if ((s = make_tmap_u8(&tmB, d->B, d->N, d->K / 2, d->ldb / 2, 128, pl.bn, true)) != LPQ_OK) return s;
  GemmParams p{};
  p.K = static_cast<int>(d->K);
  p.gx = nv ? d->ga : nullptr;
  p.gw = nv ? d->gb : nullptr;
  p.Y = d->Y;
  p.ldy = d->ldy;
  p.err = error_word_ptr();
  return launch_fp4(nv, pl, tmA, tmB, static_cast<const uint8_t*>(d->sa), static_cast<const uint8_t*>(d->sb), d->K, p,
                    d->workspace, st);
}

}  // namespace

extern "C" {

size_t lpq_gemm_workspace_bytes(const lpq_gemm_desc* d) {
  if (!d || d->M <= 0 || d->N <= 0 || d->K <= 0) return 0;
  if (is_fp8_rowscale(d)) {
    const size_t plan = plan_ws_bytes(plan_fp8_rowscale(d->M, d->N, d->K, true, SIZE_MAX));
    if ((d->flags & LPQ_GEMM_A_BF16) && d->M > kFusedMaxTokens)
      return align256(static_cast<size_t>(d->M) * static_cast<size_t>(d->K)) + plan;
    return (d->flags & LPQ_GEMM_A_BF16) ? 0 : plan;
  }
  if (is_fp4(d)) {
    return plan_ws_bytes(plan_fp4(d->M, d->N, d->K, true, SIZE_MAX));
  }
  if (is_int8(d))
    return d->K <= kInt8TcMaxK ? int8_tc_workspace_bytes(d->M, d->N, d->K, (d->flags & LPQ_GEMM_B_INT8_PLANES) != 0) : 0;
  return 0;
}

lpq_status lpq_gemm_scaled(const lpq_gemm_desc* d, void* stream) {
  LPQ_CHECK_NULL(d);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // a workspace smaller than lpq_gemm_workspace_bytes still works: the
  // planner then falls back to whole tiles
  if (is_fp8_rowscale(d)) return gemm_fp8_rowscale(d, st);
  if (is_fp8_block(d)) return gemm_fp8_block(d, st);
  if (is_int8(d)) return gemm_int8(d, st);
  if (is_fp4(d)) return gemm_fp4(d, st);
  return LPQ_ERR_UNSUPPORTED;
}

}  // extern "C"
