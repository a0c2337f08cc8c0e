/*
 * nvfp4.h -- C ABI of the B300 (sm_103a) NVFP4 quantisation and block-scaled
 * NVFP4 GEMM library.
 *
 * What the library computes, with the passages that define it:
 *   - NVFP4 is a two-level micro-scaled 4-bit format: E2M1 elements (1 sign,
 *     2 exponent, 1 mantissa bit), one FP8 E4M3 scale per 16 consecutive
 *     elements, and one FP32 scale for the whole tensor.
 *       "NVFP4: cos'è e come supera FP8 e BF16 nell'intelligenza artificiale"
 *       (guiahardware.es), section "Cos'è NVFP4 e in che modo migliora FP8 e
 *       BF16?"; "FP4" (chaitex.ru/fp4), section "Математическая структура
 *       FP4", items 1-2; "Mastering Low-Precision AI: FP8 and FP4 Support
 *       Across Frameworks in Mid-2026", first paragraph.
 *   - The training recipe uses NVFP4 for the three GEMMs of each MLP layer
 *     (fprop, dgrad, wgrad), all with NVFP4 operands and BF16 results; weights
 *     use 2D (16x16) blocks so that quantising W and W^T agree; the wgrad
 *     operands get a random Hadamard transform before quantisation; gradient
 *     quantisers use stochastic rounding.
 *       readjensen.com NVFP4 training-recipe article (2026-06-08), paragraphs
 *       on the recipe and on the data flow inside the MLP GEMMs.
 *
 * Numeric definition (every step IEEE fp32 round-to-nearest-even):
 *   amax  = max |x| over the tensor (over the transformed values with RHT)
 *   s_g   = amax / 2688                      (2688 = 6 * 448)
 *   block : sc = E4M3_RNE_satfinite(amax_b / (s_g * 6)), 0 if s_g == 0
 *   elem  : v = x * (1 / (s_g * decode(sc))) (0 if decode(sc) == 0);
 *           code = E2M1 round-to-nearest-even (or stochastic), saturating at
 *           +-6, sign bit kept (negative values that round to 0 give 0x8)
 *   RHT   : y = 1/4 * H16 * (d (.) x) per 16-chunk along the quantisation axis,
 *           Sylvester H16, d_j = -1 iff bit j of mix32(key(rht_seed, 0x5248))
 *   SR    : round |v| up iff u16 * 2^-16 < (|v| - lo) / (hi - lo); u16 comes
 *           from the lowbias32 hash of (sr_seed, output element index)
 *   GEMM  : C[m,n] = bf16_rne( s_gA * s_gB * sum_k A[m,k] * B[n,k] ), fp32
 *           accumulation on the tensor cores.
 *
 * Conventions for every call:
 *   - All pointers are DEVICE pointers unless stated.  The caller owns all
 *     memory; the library allocates nothing and keeps no reference after the
 *     call returns.
 *   - Calls are asynchronous on the given stream (a cudaStream_t; NULL means
 *     the legacy default stream).  Errors found on the host are returned
 *     immediately and nothing is launched.  Errors found on the device (a
 *     bounded wait that expired, a non-finite amax) set a per-device status
 *     word that nvfp4_check_status() reads and clears.
 *   - Shapes use int64_t; a NVFP4 operand [rows, cols] is quantised along
 *     cols (the GEMM contraction dimension K).
 */
#ifndef NVFP4_B300_H
#define NVFP4_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* nvfp4_stream_t; /* same type as cudaStream_t */

/* ---- status codes ------------------------------------------------------- */
#define NVFP4_OK 0
#define NVFP4_ERR_INVALID_ARG (-1) /* null pointer, bad shape, misalignment  */
#define NVFP4_ERR_UNSUPPORTED (-2) /* device is not sm_100-family / sm_103a  */
#define NVFP4_ERR_CUDA (-3)        /* a CUDA runtime call or launch failed    */
#define NVFP4_ERR_TIMEOUT (-4)     /* a bounded device-side wait expired      */
#define NVFP4_ERR_NONFINITE (-5)   /* an input tensor held NaN or Inf         */

/* ---- quantiser flags ---------------------------------------------------- */
#define NVFP4_BLOCK_1D 0x0u       /* 16 consecutive elements along a row     */
#define NVFP4_BLOCK_2D 0x1u       /* aligned 16x16 tiles (weights)           */
#define NVFP4_ROUND_RNE 0x0u      /* round to nearest even                   */
#define NVFP4_ROUND_SR 0x2u       /* stochastic rounding                     */
#define NVFP4_TRANSPOSE_OUT 0x4u  /* quantise x^T: output is [cols, rows]    */

/* ---- scale-factor layouts ------------------------------------------------ */
/* CANONICAL: row-major [rows, cols/16] bytes.
 * MMA: the layout the GEMM consumes.  Rows are padded to a multiple of 128
 * and cols must be a multiple of 64.  For row r and 16-element block kb the
 * byte offset is
 *     ((r / 128) * (cols / 64) + kb / 4) * 512
 *   + (r % 32) * 16 + ((r / 32) % 4) * 4 + kb % 4,
 * i.e. one 512-byte atom per (128 rows, 64 columns) holding 4 scales per
 * row, row r's 4-byte word at (r % 32, r / 32).  Padding rows read as 0. */
#define NVFP4_SCALES_CANONICAL 0
#define NVFP4_SCALES_MMA 1

/* A quantised operand.  All buffers are device memory owned by the caller.
 *   codes        [rows, cols/2] bytes: element 2j in the low nibble of byte j.
 *   scales       E4M3 block scales (sign bit 0) in `scale_layout`;
 *                nvfp4_scales_bytes() gives the size.
 *   amax         fp32 scalar, written by the quantiser.
 *   global_scale fp32 scalar s_g, written by the quantiser, read by the GEMM.
 *   rows, cols   logical shape of the quantised operand (cols = K). */
typedef struct nvfp4_tensor {
  uint8_t* codes;
  uint8_t* scales;
  float* amax;
  float* global_scale;
  int64_t rows;
  int64_t cols;
  int32_t scale_layout;
  int32_t reserved; /* must be 0 */
} nvfp4_tensor;

/* Bytes of the scale buffer for an operand [rows, cols] in `layout`
 * (0 for an invalid combination). */
size_t nvfp4_scales_bytes(int64_t rows, int64_t cols, int32_t layout);

/* Quantise a bf16 matrix x [rows, cols] (row stride ld elements) to NVFP4:
 * E2M1 elements with one E4M3 scale per 16 values and one FP32 tensor scale
 * ("NVFP4: cos'è e come supera FP8 e BF16 ...", section "Cos'è NVFP4 ...";
 * "FP4" (chaitex.ru/fp4), section "Математическая структура FP4"), with the
 * recipe's 16x16 weight blocks and stochastic rounding as options
 * (readjensen.com NVFP4 training-recipe article, MLP data-flow paragraph).
 * flags: NVFP4_BLOCK_1D or NVFP4_BLOCK_2D, NVFP4_ROUND_RNE or NVFP4_ROUND_SR,
 * optionally NVFP4_TRANSPOSE_OUT (then out is [cols, rows], blocks run along
 * the input's rows).  out->rows/out->cols must equal the output shape.
 * sr_seed keys the stochastic rounding (ignored for RNE).  amax_in (device
 * fp32, nullable) supplies the tensor amax and skips the amax pass.
 * Requirements: x 16-byte aligned, ld % 8 == 0, cols % 8 == 0, the output's
 * cols % 16 == 0 (and % 64 for the MMA scale layout), both output dims % 16
 * for 2D.  Returns NVFP4_OK or a negative status code. */
int nvfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld,
                   uint32_t flags, uint64_t sr_seed, const float* amax_in,
                   const nvfp4_tensor* out, nvfp4_stream_t stream);

/* Quantise with the 16-point random Hadamard transform and stochastic
 * rounding: the recipe's treatment of the wgrad operands (readjensen.com
 * NVFP4 training-recipe article, MLP data-flow paragraph: a random Hadamard
 * transform before 4-bit quantisation of the weight-gradient inputs,
 * stochastic rounding for gradients).  The transform runs along the output's
 * quantisation axis, so with NVFP4_TRANSPOSE_OUT (the usual wgrad case) it
 * mixes 16 consecutive rows (tokens) of x.  Both wgrad operands must use the
 * same rht_seed; use different sr_seeds.  The amax is taken after the
 * transform.  NVFP4_BLOCK_2D is not allowed; other arguments as for
 * nvfp4_quantize(). */
int nvfp4_quantize_rht_sr(const void* x, int64_t rows, int64_t cols, int64_t ld,
                          uint32_t flags, uint64_t rht_seed, uint64_t sr_seed,
                          const float* amax_in, const nvfp4_tensor* out,
                          nvfp4_stream_t stream);

/* Dual-orientation quantisation: one pass over x [rows, cols] produces both
 * operands a training step takes from the same tensor (the activations X
 * feed fprop and wgrad, the output gradient dY feeds dgrad and wgrad):
 *   out_row [rows, cols]  = nvfp4_quantize(x, row_flags, row_sr_seed, amax_row_in)
 *                           with 1D blocks (row_flags: NVFP4_ROUND_RNE or
 *                           NVFP4_ROUND_SR; nothing else),
 *   out_col [cols, rows]  = nvfp4_quantize_rht_sr(x, NVFP4_TRANSPOSE_OUT,
 *                           rht_seed, col_sr_seed, amax_col_in),
 * bit-identical to those two calls.  The recipe's data flow inside the MLP
 * GEMMs (readjensen.com NVFP4 training-recipe article, MLP data-flow
 * paragraph) quantises each of X and dY once per orientation; this call reads
 * x twice (one pass for both amaxes unless both are supplied, one for both
 * encodings) instead of four times.  Both outputs must use the same scale
 * layout.  Requirements: rows % 16 == 0 and cols % 16 == 0 (% 64 for the MMA
 * layout), x 16-byte aligned, ld % 8 == 0, codes 8-byte aligned.  Returns
 * NVFP4_OK or a negative status code; nothing is launched on an error. */
int nvfp4_quantize_dual(const void* x, int64_t rows, int64_t cols, int64_t ld, uint32_t row_flags,
                        uint64_t row_sr_seed, uint64_t rht_seed, uint64_t col_sr_seed,
                        const float* amax_row_in, const float* amax_col_in, const nvfp4_tensor* out_row,
                        const nvfp4_tensor* out_col, nvfp4_stream_t stream);

/* MXFP4 quantisation, for comparison with NVFP4: the power-of-two-scaled
 * open format the pages set NVFP4 against ("NVFP4: cos'è e come supera FP8 e
 * BF16 ...", section "Cos'è NVFP4 ...", second paragraph: NVFP4 has much less
 * quantisation error than power-of-two solutions such as MXFP4; "FP4"
 * (chaitex.ru/fp4), section "Сравнительный ландшафт низкоразрядных
 * форматов": NVFP4 uses smaller blocks and exact scale factors).  Format
 * (the open microscaling layout; the pages give no detail): 32 consecutive
 * elements of a row share the scale 2^e, e = floor(log2(block amax)) - 2
 * clamped to [-127, 127] (-127 for a zero or subnormal block maximum), stored
 * as the E8M0 byte e + 127; elements are E2M1, round-to-nearest-even of
 * x / 2^e saturating at 6, sign kept; no tensor scale.
 *   x       bf16 [rows, cols], row stride ld elements (16-byte aligned,
 *           ld % 8 == 0, cols % 32 == 0)
 *   codes   [rows, cols/2] bytes, element 2j in the low nibble of byte j
 *           (16-byte aligned)
 *   scales  [rows, cols/32] E8M0 bytes, row-major
 * Returns NVFP4_OK or a negative status code (nothing launched on error). */
int nvfp4_quantize_mxfp4(const void* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* codes,
                         uint8_t* scales_e8m0, nvfp4_stream_t stream);

/* Block-scaled NVFP4 GEMM, "TN": C[M, N] = s_gA * s_gB * A[M, K] * B[N, K]^T
 * with fp32 accumulation and a BF16 (round-to-nearest-even) result: the
 * recipe's three MLP GEMMs take NVFP4 operands and return BF16
 * (readjensen.com NVFP4 training-recipe article, MLP data-flow paragraph),
 * and the fifth-generation tensor cores apply the block scales in hardware
 * ("NVFP4: cos'è e come supera FP8 e BF16 ...", section "Blackwell
 * Architecture: la potenza dietro NVFP4").
 * A and B must use NVFP4_SCALES_MMA, K = A->cols = B->cols, K % 256 == 0.
 * c is bf16 [M, N] with row stride ldc elements (ldc >= N, ldc % 8 == 0,
 * c 16-byte aligned).  The same call serves fprop (X * W^T), dgrad
 * (dY * (W^T)^T) and wgrad (dY^T * (X^T)^T) given suitably quantised operands. */
int nvfp4_gemm(const nvfp4_tensor* A, const nvfp4_tensor* B, void* c, int64_t ldc,
               nvfp4_stream_t stream);

/* Up to NVFP4_GEMM_GROUP_MAX independent GEMMs in one launch:
 * c[i] = s_gA[i] * s_gB[i] * A[i] * B[i]^T, each exactly as nvfp4_gemm()
 * computes it (same bits).  The backward pass of the MLP layer has two such
 * GEMMs, dgrad and wgrad, that read different operands and write different
 * outputs (readjensen.com NVFP4 training-recipe article, MLP data-flow
 * paragraph).  One persistent grid shares out both problems' output tiles,
 * longer contractions first, so neither GEMM leaves multiprocessors idle in
 * a last partial round of tiles.  A, B, c and ldc are HOST arrays of count
 * (1 .. NVFP4_GEMM_GROUP_MAX) entries; the tensors' buffers are device
 * memory as for nvfp4_gemm().  Every problem is checked as nvfp4_gemm()
 * checks it, and nothing is launched if one fails.  The outputs must not
 * overlap each other or any operand. */
#define NVFP4_GEMM_GROUP_MAX 2
int nvfp4_gemm_group(int32_t count, const nvfp4_tensor* const* A, const nvfp4_tensor* const* B, void* const* c,
                     const int64_t* ldc, nvfp4_stream_t stream);

/* Synchronise `stream`, then read the device status word of the current
 * device and clear the bits it read (a bit raised meanwhile by a kernel on
 * another stream stays set for the next call).  Returns NVFP4_OK,
 * NVFP4_ERR_TIMEOUT, NVFP4_ERR_NONFINITE or NVFP4_ERR_CUDA. */
int nvfp4_check_status(nvfp4_stream_t stream);

/* Static description of a status code. */
const char* nvfp4_status_string(int status);

/* Library version (major * 10000 + minor * 100 + patch). */
int nvfp4_version(void);

/* ---- failure-detection self-test ------------------------------------------ */
/* Launch a one-warp kernel whose bounded mbarrier waits (the same two wait
 * helpers every kernel of the library uses) wait on a barrier that nothing
 * completes: after limit_us microseconds (1 .. 2,000,000) each wait gives up,
 * raises the timeout bit of the device status word, and the kernel exits.
 * The next nvfp4_check_status() returns NVFP4_ERR_TIMEOUT and the context
 * stays usable.  This is how a lost arrival inside a kernel surfaces; no
 * kernel traps or spins without a limit.  Not part of the pages' method. */
int nvfp4_selftest_wait_timeout(uint32_t limit_us, nvfp4_stream_t stream);

/* ---- FP4 tensor-core rate probe ------------------------------------------- */
/* Measure the dense FP4 tensor-core rate this library's GEMM is bounded by:
 * one CTA pair per two multiprocessors issues n_mma (1 .. 2^20) back-to-back
 * block-scaled pair MMAs (kind::mxf4nvf4, scale_vec::4X, M = 256 over the
 * pair, N = mma_n (128 or 256), K = 64) on fixed on-chip operands, with no
 * memory traffic.  For pair p, out[2 p] receives the SM cycles and
 * out[2 p + 1] the nanoseconds from the first issue to the completion of the
 * last MMA (0 if a bounded wait expired).  out is device memory with room for
 * 2 * (multiprocessors / 2) uint64 values (8-byte aligned); *pairs_launched
 * (host) receives the number of pairs.  FLOP per SM per MMA = 2 * 128 *
 * mma_n * 64.  The fifth-generation tensor cores' NVFP4 block scaling in
 * hardware is the pages' basis for this path ("NVFP4: cos'è e come supera
 * FP8 e BF16 ...", section "Blackwell Architecture: la potenza dietro NVFP4");
 * the probe is the measured denominator of the GEMM's roofline. */
int nvfp4_mma_rate_probe(int32_t n_mma, int32_t mma_n, uint64_t* out, int32_t* pairs_launched,
                         nvfp4_stream_t stream);

/* ---- operand delivery-rate probe ----------------------------------------- */
/* Measure how fast global memory (L2 when src_bytes fits in it) fills one
 * multiprocessor's shared memory by asynchronous copies, the path the GEMM's
 * operand tiles take: each of `ctas` CTAs (one per multiprocessor,
 * 1 .. multiprocessors) streams `iters` (1 .. 2^20) 16 KiB copies from src
 * into a 12-slot shared-memory ring, cycling through src.  mode 0: plain
 * bulk copies of consecutive 16 KiB chunks (src_bytes >= 16384, whole chunks
 * used).  mode 1: the GEMM's own operand boxes, 128 rows x 128 bytes with
 * 128-byte swizzle, through a tensor map over src viewed as rows of 2048
 * bytes (an NVFP4 operand with K = 4096; src_bytes >= 262144, whole 128-row
 * bands used).  src is device memory, 16-byte aligned.  For CTA c, out[3 c]
 * receives the nanoseconds from its first copy to the arrival of its last (0
 * if a bounded wait expired), out[3 c + 1] the bytes it received and
 * out[3 c + 2] the SM cycles of the same interval; out is device memory with
 * room for 3 * ctas uint64 values (8-byte aligned).  Not
 * part of the pages' method: it is the measured per-multiprocessor operand
 * delivery rate that bounds the GEMM alongside the tensor-core rate. */
int nvfp4_copy_rate_probe(const void* src, int64_t src_bytes, int32_t mode, int32_t ctas, int32_t iters,
                          uint64_t* out, nvfp4_stream_t stream);

/* ---- codec diagnostics (exhaustive conversion checks) -------------------- */
/* out[i] = E2M1 code (low nibble) of v[i] with round-to-nearest-even,
 * saturating, sign kept -- the element encoder the quantiser uses.
 * v and out are device arrays of n elements. */
int nvfp4_encode_e2m1_rne(const float* v, int64_t n, uint8_t* out, nvfp4_stream_t stream);

/* out[i] = E2M1 code of v[i] rounded stochastically with the 16 random bits
 * u16[i] (the quantiser's SR encoder). */
int nvfp4_encode_e2m1_sr(const float* v, const uint16_t* u16, int64_t n, uint8_t* out,
                         nvfp4_stream_t stream);

/* out[i] = E4M3 code of t[i] >= 0, round-to-nearest-even, saturating at 448,
 * NaN -> 0 (the quantiser's block-scale encoder). */
int nvfp4_encode_e4m3(const float* t, int64_t n, uint8_t* out, nvfp4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_B300_H */
