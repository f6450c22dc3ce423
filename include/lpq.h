/*
 * lpq.h - C ABI of the GB300 (sm_103a) quantized-linear library.
 *
 * The library computes the weight-and-activation quantized linear layer:
 * dynamic activation quantization (FP8 E4M3FN per token or per 1x128 group,
 * INT8 per token with SmoothQuant factors, NVFP4 or MXFP4 block-scaled E2M1),
 * static weight quantization, and a tensor-core GEMM with FP32 (INT32 for
 * INT8) accumulation whose epilogue applies the scales and writes bf16:
 *     Y = diag(s_X) (X_q W_q^T) diag(s_W)
 * ("FP8 and FP4 inference, SmoothQuant and activation quantization", section
 *  "Scale granularity"; "Low-bit LLM Weights and Activations", section 3.4).
 *
 * Conventions for every entry point:
 *  - Pointers to tensors are DEVICE pointers owned by the caller.  The library
 *    never allocates, frees or synchronises; each call only enqueues kernels on
 *    `stream` (a cudaStream_t; NULL = the legacy default stream) and returns.
 *  - bf16 tensors are passed as uint16_t bit patterns.  Matrices are row-major;
 *    `ld*` arguments are row strides in ELEMENTS.  X is [M, K], W is [N, K]
 *    (the [out, in] layout of a linear layer), Y is [M, N].
 *  - Quantized outputs are dense: codes [rows, K] (FP4: [rows, K/2] bytes,
 *    element 2i in the low nibble of byte i), scales as documented per call.
 *  - All device pointers must be 16-byte aligned; bf16 row strides a multiple
 *    of 8 elements.  K must be a multiple of 16 (FP4: 32; block-scaled FP8:
 *    128).  M, N >= 1 and K >= 16 unless a call says otherwise.
 *  - Validation happens on the host before any launch; a failing call
 *    enqueues nothing and returns an error code.  Kernels never trap.  Inputs
 *    are expected to be finite; NaN/Inf inputs give unspecified codes but do
 *    not fault.
 *  - Calls are stateless and thread-safe (the CUDA error of the last failing
 *    launch is kept per host thread).
 */
#ifndef LPQ_H_
#define LPQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LPQ_OK = 0,
  LPQ_ERR_NULL = 1,         /* a required pointer is NULL                          */
  LPQ_ERR_SHAPE = 2,        /* a size is <= 0, K not a multiple of the block, ld < K; quantizers: M or N >= 2^31, K > 2^30 */
  LPQ_ERR_ALIGN = 3,        /* a pointer is not 16-byte aligned / ld not a multiple of 8 */
  LPQ_ERR_UNSUPPORTED = 4,  /* format / granularity combination not provided        */
  LPQ_ERR_CUDA = 5,         /* a launch failed; see lpq_last_cuda_error()          */
  LPQ_ERR_WORKSPACE = 6     /* workspace given but too small for the request       */
} lpq_status;

typedef enum {
  LPQ_GRAN_ROW = 0,           /* one scale per row: per token (X) / per output channel (W) */
  LPQ_GRAN_BLOCK_1x128 = 1,   /* activations: one scale per token and 128-wide K group      */
  LPQ_GRAN_BLOCK_128x128 = 2, /* weights: one scale per 128x128 block                       */
  LPQ_GRAN_TENSOR_STATIC = 3  /* one calibrated scale for the whole tensor (input)          */
} lpq_gran;

typedef enum {
  LPQ_FMT_FP8 = 0,    /* E4M3FN codes, fp32 scales                       */
  LPQ_FMT_INT8 = 1,   /* int8 codes (+-127), fp32 scales                 */
  LPQ_FMT_NVFP4 = 2,  /* E2M1 codes, E4M3 scale per 16, fp32 tensor scale */
  LPQ_FMT_MXFP4 = 3   /* E2M1 codes, E8M0 scale per 32                    */
} lpq_format;

/* ---------------------------------------------------------------- errors -- */
const char* lpq_status_string(lpq_status s);
/* cudaError_t (as int) of the last failing launch on this host thread. */
int lpq_last_cuda_error(void);
/* Device error word, written by kernels whose bounded waits timed out
 * (0 = none).  Synchronises the device; `lpq_clear_error_word` resets it. */
lpq_status lpq_read_error_word(uint32_t* out);
lpq_status lpq_clear_error_word(void);
/* Diagnostics for the failure path: one kernel waits, as every barrier wait
 * in the library's kernels does, on a barrier that nothing completes; after
 * limit_ns (1 .. 2e9) it gives up, writes LPQ_SELFTEST_WAIT_CODE into the
 * device error word (if it was 0) and returns.  No trap and no fault: the
 * context stays usable.  Asynchronous on `stream`. */
#define LPQ_SELFTEST_WAIT_CODE 0x0F0Fu
lpq_status lpq_selftest_bounded_wait(uint64_t limit_ns, void* stream);
/* Library version and the number of kernels launched by this host thread
 * since the last reset (for launch accounting). */
const char* lpq_version(void);
uint64_t lpq_launch_count(void);
void lpq_reset_launch_count(void);

/* ------------------------------------------------------ SmoothQuant (a4) -- */
/* Running per-input-channel activation maximum over a calibration batch:
 * chan_amax[j] = max(chan_amax[j], max_t |X[t, j]|).  chan_amax: [K] fp32,
 * in/out; start it at 0.  "Low-bit LLM Weights and Activations", section 4.3
 * step 1 (measure per-channel activation maxima on calibration data). */
lpq_status lpq_act_absmax_update(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                                 float* chan_amax, void* stream);

/* Smoothing factors s_j = max(ax_j, 1e-5)^alpha / max(aw_j, 1e-5)^(1 - alpha),
 * aw_j = max_n |W[n, j]|; the power is taken in fp64 and rounded once to fp32.
 * "Low-bit LLM Weights and Activations", section 4.2.  chan_amax: [K] fp32;
 * W: [N, K] bf16; s: [K] fp32 out (also used as scratch during the call). */
lpq_status lpq_smooth_calibrate(const float* chan_amax, const uint16_t* W, int64_t N, int64_t K,
                                int64_t ldw, float alpha, float* s, void* stream);

/* ------------------------------------------------------ quantizers (a1-a8) -- */
/* FP8 E4M3FN activation quantization, round-to-nearest-even, saturating to
 * +-448 (never NaN), with s = max(amax, 1e-8) / 448 and q = E4M3(x / s)
 * ("FP8 and FP4 inference ...", section "Implementation sketch", per-token
 * emulation; "FP8 and INT8 Inference", section 5 "What DeepSeek did").
 *   g = LPQ_GRAN_ROW:          sx [M] out.
 *   g = LPQ_GRAN_BLOCK_1x128:  sx [K/128][M] out (K-group major, M contiguous);
 *                              K must be a multiple of 128.
 *   g = LPQ_GRAN_TENSOR_STATIC: sx [1] IN (a calibrated scale); no reduction.
 * Xq: [M, K] uint8 out. */
lpq_status lpq_quantize_act_fp8(const uint16_t* X, int64_t M, int64_t K, int64_t ldx, lpq_gran g,
                                uint8_t* Xq, float* sx, void* stream);

/* FP8 E4M3FN weight quantization (static, at load time).
 *   g = LPQ_GRAN_ROW:             sw [N] out (per output channel).
 *   g = LPQ_GRAN_BLOCK_128x128:   sw [ceil(N/128)][K/128] out; K % 128 == 0.
 * Wq: [N, K] uint8 out.  Same rounding rule as the activation quantizer. */
lpq_status lpq_quantize_weight_fp8(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, lpq_gran g,
                                   uint8_t* Wq, float* sw, void* stream);

/* INT8 per-token activation quantization with optional SmoothQuant factors:
 * x~ = x / smooth[j] (fp32), S = max(max|x~|, 1e-8) / 127,
 * q = clamp(round_half_even(x~ / S), -127, 127).  smooth: [K] or NULL.
 * "Low-bit LLM Weights and Activations", sections 2.1 and 4.3; "FP8 and INT8
 * Inference", section 5 "INT8 in practice".  Xq: [M, K] int8; sx: [M]. */
lpq_status lpq_quantize_act_int8(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                                 const float* smooth, int8_t* Xq, float* sx, void* stream);

/* INT8 per-output-channel weight quantization; w~ = w * smooth[j] (fp32).
 * Wq: [N, K] int8; sw: [N]. */
lpq_status lpq_quantize_weight_int8(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                                    const float* smooth, int8_t* Wq, float* sw, void* stream);

/* INT8 weight codes -> the E4M3 digit planes the tensor-core INT8 GEMM reads,
 * for weights quantized once at load time: every code q = 16 h + l with
 * h = floor(q / 16) in [-8, 7] and l in [0, 15], both exact in E4M3; planes
 * [2][N][K] bytes (all h codes, then all l codes; rows of K, no padding).
 * Pass planes as B with LPQ_GEMM_B_INT8_PLANES (the product stays the exact
 * int32 one).  Wq: [N, ldw] int8, ldw a multiple of 16, K a multiple of 16. */
lpq_status lpq_int8_weight_planes(const int8_t* Wq, int64_t N, int64_t K, int64_t ldw, uint8_t* planes,
                                  void* stream);

/* NVFP4: g = amax / (448 * 6) over the whole tensor (g = 1 if all zero);
 * per block of 16: c = E4M3((amax_b / 6) / g), s = dec(c) * g,
 * q = E2M1(x / s) (a block whose c is 0 stores zero codes).
 * "FP8 and FP4 inference ...", section "Implementation sketch" (nvfp4).
 * Xq: [M, K/2] bytes; sf: lpq_sf_bytes(LPQ_FMT_NVFP4, M, K) bytes in the
 * tensor-core scale layout (see lpq_sf_offset; padding written as 0);
 * gs: [2] fp32 out: gs[0] = tensor amax, gs[1] = g.  K % 32 == 0.
 * Two kernels run in stream order (tensor amax, then the blocks). */
lpq_status lpq_quantize_act_nvfp4(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                                  uint8_t* Xq, uint8_t* sf, float* gs, void* stream);
lpq_status lpq_quantize_weight_nvfp4(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                                     uint8_t* Wq, uint8_t* sf, float* gs, void* stream);

/* MXFP4: per block of 32, e = clamp(floor(log2 amax_b) - 2, -127, 127),
 * stored as the E8M0 code e + 127; q = E2M1(x * 2^-e).  (The pages give
 * "power-of-two scale per 32, E8M0, bias 127"; the exponent rule is the OCP MX
 * one they cite.)  Xq: [M, K/2] bytes; sf: lpq_sf_bytes(LPQ_FMT_MXFP4, M, K).
 * K % 32 == 0. */
lpq_status lpq_quantize_act_mxfp4(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                                  uint8_t* Xq, uint8_t* sf, void* stream);
lpq_status lpq_quantize_weight_mxfp4(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                                     uint8_t* Wq, uint8_t* sf, void* stream);

/* Scale-factor layout of the FP4 formats (host functions, no GPU needed).
 * Rows are grouped by 128 and scale blocks by 4; each 128x4 tile is 512
 * contiguous bytes, tiles ordered row-group major; inside a tile the scale of
 * (row r, block kb) sits at (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 4.
 * This is the order the tensor core reads scales in. */
size_t lpq_sf_bytes(lpq_format fmt, int64_t rows, int64_t K);
size_t lpq_sf_offset(lpq_format fmt, int64_t rows, int64_t K, int64_t r, int64_t kblock);

/* ------------------------------------------------------------ GEMM (a9-a12) -- */
/* Y[M, N] = bf16( dequant(A)[M, K] . dequant(B)[N, K]^T ), A = quantized X,
 * B = quantized W, both K-contiguous ("TN").
 *   fmt FP8, a_gran ROW, b_gran ROW:
 *       Y = bf16((acc * sa[m]) * sb[n]), acc = sum_k A B in fp32 (tensor memory).
 *   fmt FP8, a_gran BLOCK_1x128, b_gran BLOCK_128x128:
 *       acc += (sum_{k in group} A B) * sa[kb][m] * sb[n/128][kb] per 128-wide K
 *       group, in fp32; Y = bf16(acc).  K % 128 == 0.
 *   fmt FP8, a_gran TENSOR_STATIC: sa[0] is the single activation scale.
 *   fmt INT8, ROW, ROW: acc exact in int32; Y = bf16((float(acc) * sa[m]) * sb[n]).
 *       With a workspace of lpq_gemm_workspace_bytes (K <= 65536) the product
 *       runs on the tcgen05 tensor cores through E4M3 digit planes (see
 *       lpq_int8_weight_planes), else on the warp-level int8 MMA; same bits.
 *   fmt NVFP4: sa / sb are the scale-layout buffers of the quantizers; ga / gb
 *       point at the tensor scales g (gs + 1); Y = bf16(acc * ga * gb).
 *   fmt MXFP4: as NVFP4 without ga / gb.
 * lda / ldb are row strides in elements (FP4: elements, two per byte).
 * workspace: optional device buffer for fp32 partial sums: when the output
 * tiles leave the last wave of CTAs mostly idle, those tiles are split along
 * K and a second kernel adds the slices in a fixed order.  If NULL (or too
 * small) the library uses whole tiles only.  Its size for a problem is
 * lpq_gemm_workspace_bytes(desc) (0 when no split would be used); its
 * contents need no initialisation.  Calls sharing one workspace must be
 * ordered on one stream.
 * "FP8 and INT8 Inference", sections 5 and 6-9 (the GEMM epilogue);
 * "Low-bit LLM Weights and Activations", section 3.4. */
typedef struct {
  lpq_format fmt;
  lpq_gran a_gran, b_gran;
  int64_t M, N, K;
  const void* A; int64_t lda;
  const void* B; int64_t ldb;
  const void* sa;              /* activation scales (layout per a_gran / fmt) */
  const void* sb;              /* weight scales                               */
  const float* ga;             /* NVFP4 tensor scale of A (device, [1])       */
  const float* gb;             /* NVFP4 tensor scale of B (device, [1])       */
  uint16_t* Y; int64_t ldy;    /* bf16 output                                 */
  void* workspace; size_t workspace_bytes;
  uint32_t flags;              /* LPQ_GEMM_* bits below; 0 = none          */
} lpq_gemm_desc;

/* flags: the weights B are not written by the kernel that immediately
 * precedes this call on the stream (true for weights quantized at load time).
 * The GEMM may then start streaming B before that kernel has finished; its
 * activations, scales and output still wait for it.  FP8 row-scaled GEMMs. */
#define LPQ_GEMM_B_STATIC 1u
/* flags: A holds the bf16 activations X [M][lda] (lda in elements, a multiple
 * of 16), not codes; the call quantizes them per token itself, by the rule of
 * lpq_quantize_act_fp8 with LPQ_GRAN_ROW (s = max(max_k |x|, 1e-8) / 448,
 * codes E4M3FN(x / s)), writes the scales to sa ([M] fp32, an output here) and
 * computes the same Y as lpq_quantize_act_fp8 followed by lpq_gemm_scaled.
 * fmt FP8, a_gran ROW, b_gran ROW only.  For M <= 16 the quantization runs
 * inside the GEMM kernel and the codes never reach memory: the 8-bit
 * activations do not make a round trip through HBM ("FP8 and INT8
 * Inference", sections 6-9, where the quantization sits in the producing
 * GEMM's epilogue; here it sits in the consuming GEMM, for bf16 activations
 * from any producer).  For larger M the codes go through the workspace
 * (lpq_gemm_workspace_bytes includes them; a missing or smaller workspace
 * returns LPQ_ERR_WORKSPACE).  Not accepted by lpq_gemm_scaled_noalloc. */
#define LPQ_GEMM_A_BF16 2u
/* flags: fmt INT8; B holds the planes of lpq_int8_weight_planes ([2][N][K],
 * ldb ignored) instead of the int8 codes.  Needs a workspace of
 * lpq_gemm_workspace_bytes (the activations' planes), else LPQ_ERR_WORKSPACE. */
#define LPQ_GEMM_B_INT8_PLANES 4u

size_t lpq_gemm_workspace_bytes(const lpq_gemm_desc* d);
lpq_status lpq_gemm_scaled(const lpq_gemm_desc* d, void* stream);

/* ------------------------------------------- GEMM without a workspace -- */
/* The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory: a plugin inside a serving runtime that owns
 * all device memory through its own pool and hands over only the operation's
 * tensors, or a latency-critical path where cudaMalloc's implicit device-wide
 * synchronisation is not acceptable and no workspace was set aside.
 *
 * Same operation and arguments as lpq_gemm_scaled for fmt LPQ_FMT_FP8 with
 * a_gran ROW or TENSOR_STATIC and b_gran ROW (other combinations return
 * LPQ_ERR_UNSUPPORTED); d->workspace is ignored.  The split-K scratch comes
 * from one array of LPQ_NOALLOC_SCRATCH_BYTES inside the library, which every
 * GPU that loads the library holds until the process exits.  A problem whose
 * split-K scratch would exceed that size returns LPQ_ERR_WORKSPACE and
 * enqueues nothing; nothing is allocated or freed.
 * The first call on a device looks up the array's device address (a one-time
 * set-up per device, done with that device current); make that first call
 * before any stream capture.  All calls share the array (no call depends on
 * what an earlier one left in it), so calls that may run at the same time on
 * the GPU race on it; order them on one stream. */
#define LPQ_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
lpq_status lpq_gemm_scaled_noalloc(const lpq_gemm_desc* d, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* LPQ_H_ */
