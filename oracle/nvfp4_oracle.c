/*
 * nvfp4_oracle.c -- plain, slow, obviously-correct CPU reference for NVFP4
 * quantisation and the block-scaled NVFP4 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline / reference arm may load this library.  It shares no
 * code, header, table or constant generator with the CUDA path.
 *
 * Sources (each function cites the passage it follows):
 *   [P3] "NVFP4: cos'è e come supera FP8 e BF16 nell'intelligenza artificiale"
 *        (guiahardware.es), section "Cos'è NVFP4 e in che modo migliora FP8 e
 *        BF16?": E2M1 elements (1 sign, 2 exponent, 1 mantissa bit), an FP8 E4M3
 *        scale per 16-value micro-block and an FP32 tensor-level scale.
 *   [P4] "FP4" (chaitex.ru/fp4), section "Математическая структура FP4": the
 *        1-2-1 bit split, items 1 (16-element micro-blocks with an E4M3 scale)
 *        and 2 (a 32-bit whole-tensor multiplier).
 *   [P5] "Mastering Low-Precision AI: FP8 and FP4 Support Across Frameworks in
 *        Mid-2026", first paragraph: shared FP8 scale per 16 elements plus a
 *        tensor-level scale.
 *   [P2] readjensen.com article on the Blackwell NVFP4 training recipe
 *        (2026-06-08), paragraph on the data flow inside the MLP GEMMs: all three
 *        GEMMs take NVFP4 inputs and emit BF16; weights use 2D block
 *        quantisation so fprop and dgrad agree under transposition; a random
 *        Hadamard transform is applied to the wgrad inputs; gradient quantisers
 *        use stochastic rounding.
 *
 * Readings where the pages are silent (all listed in the design notes):
 *   - tensor scale s_g = amax / (6 * 448), one fp32 division;
 *   - block scale sc = E4M3_RNE_satfinite(amax_b / (6 * s_g)); 0 when the
 *     denominator is 0 or the quotient is NaN;
 *   - element v = x * (1 / (s_g * decode(sc))), E2M1 round-to-nearest-even (or
 *     stochastic), saturating at 6, sign kept (so -0 encodes as 0x8);
 *   - 2D blocks are aligned 16x16 tiles; the tile scale is stored on each of the
 *     tile's 16 rows;
 *   - RHT: y = 1/4 * H16 * (d (.) x) on each 16-chunk along the quantisation
 *     axis, Sylvester H16, d_j = -1 iff bit j of mix32(K(rht_seed, 0x5248));
 *   - SR random bits: 16 bits per element from the "lowbias32" integer hash
 *     (C. Wellons, hash-prospector, 2018, public domain) keyed by the seed and
 *     the element's row-major index in the OUTPUT orientation;
 *   - packing: the even column goes to the low nibble;
 *   - MXFP4 (the comparison format): 32-element row blocks, scale 2^e stored
 *     as E8M0, e = floor(log2(block amax)) - 2 clamped to [-127, 127],
 *     elements E2M1 round-to-nearest-even of x / 2^e.
 * Every fp32 operation below is a single IEEE round-to-nearest-even operation;
 * build with -ffp-contract=off so no multiply-add is fused.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OFLAG_BLOCK_2D 0x1u
#define OFLAG_SR 0x2u
#define OFLAG_TRANSPOSE 0x4u
#define OFLAG_RHT 0x8u

/* ---------------------------------------------------------------- bf16 --- */

/* bf16 is the upper half of an fp32 pattern: widening is exact. */
static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round a double to bf16 with round-to-nearest-even in ONE step (no detour
 * through fp32, which would round twice).  bf16 has 8 significant bits and
 * the fp32 exponent range (normals down to 2^-126, subnormal quantum 2^-133). */
uint16_t o_bf16_rne(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);          /* a = f * 2^e, f in [0.5, 1) -> a in [2^(e-1), 2^e) */
  int ulp_exp = (e - 1) - 7; /* quantum of an 8-significant-bit number */
  if (ulp_exp < -133) ulp_exp = -133;
  double q = ldexp(a, -ulp_exp);       /* exact scaling by a power of two */
  double n = nearbyint(q);             /* default rounding: to nearest, ties even */
  double r = ldexp(n, ulp_exp);
  if (r >= ldexp(1.0, 128)) return sign | 0x7F80; /* overflow -> inf */
  float f = (float)r; /* exact: r has <= 8 significant bits and fits fp32 */
  uint32_t u;
  memcpy(&u, &f, 4);
  return sign | (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------- E2M1 --- */

/* [P4] 1 sign bit, 2 exponent bits, 1 mantissa bit; exponent bias 1, so the
 * exponent-0 codes are 0 and 0.5 and the others are 2^(e-1) * (1 + m/2). */
float o_e2m1_decode(uint8_t code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  float mag = (e == 0) ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, e - 1);
  return s ? -mag : mag;
}

/* Round-to-nearest-even onto the eight E2M1 magnitudes, saturating at 6:
 * walk the ascending magnitude list and compare with the exact midpoints; a
 * value equal to a midpoint goes to the even code (even mantissa bit). */
uint8_t o_e2m1_encode_rne(float v) {
  uint8_t sign = signbit(v) ? 0x8 : 0x0;
  float a = fabsf(v);
  uint8_t code = 7; /* saturate: anything above the last midpoint is 6 */
  for (uint8_t c = 0; c < 7; ++c) {
    float lo = o_e2m1_decode(c), hi = o_e2m1_decode((uint8_t)(c + 1));
    float mid = 0.5f * (lo + hi); /* exact: small dyadic rationals */
    if (a < mid) { code = c; break; }
    if (a == mid) { code = (c % 2 == 0) ? c : (uint8_t)(c + 1); break; }
  }
  return sign | code;
}

/* Stochastic rounding onto E2M1 ([P2] recipe: gradient quantisers round
 * stochastically so that small updates stay unbiased).  With lo <= |v| < hi adjacent
 * magnitudes, round up iff u16 * 2^-16 < (|v| - lo) / (hi - lo).  The
 * subtraction is exact (Sterbenz or lo = 0) and hi - lo is a power of two, so
 * p is exact; |v| >= 6 saturates to 6. */
uint8_t o_e2m1_encode_sr(float v, uint32_t u16) {
  uint8_t sign = signbit(v) ? 0x8 : 0x0;
  float a = fabsf(v);
  if (!(a < 6.0f)) return sign | 7;
  uint8_t c = 0;
  while (c < 7 && o_e2m1_decode((uint8_t)(c + 1)) <= a) ++c; /* lo = decode(c) */
  float lo = o_e2m1_decode(c), hi = o_e2m1_decode((uint8_t)(c + 1));
  float p = (a - lo) * (1.0f / (hi - lo));
  float u = (float)(u16 & 0xFFFFu) * 0x1p-16f;
  return sign | (uint8_t)(u < p ? c + 1 : c);
}

/* ---------------------------------------------------------------- E4M3 --- */

/* FP8 E4M3 (the micro-block scale type named by [P3], [P4] item 1, [P5]):
 * 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is subnormal
 * (m * 2^-9); 0x7F/0xFF are NaN, so the largest finite value is 0x7E = 448. */
float o_e4m3_decode(uint8_t code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  float mag = (e == 0) ? ldexpf((float)m, -9) : ldexpf(1.0f + (float)m / 8.0f, e - 7);
  return s ? -mag : mag;
}

/* Non-negative scale encoding: round-to-nearest-even among the 127 finite
 * non-negative codes, saturating at 448; NaN (0/0) gives code 0.  Binary
 * search on the monotone code order, then the exact-midpoint tie rule. */
uint8_t o_e4m3_encode(float t) {
  if (isnan(t) || t <= 0.0f) return 0;
  if (t >= 448.0f) return 0x7E;
  int lo = 0, hi = 0x7E; /* invariant: decode(lo) <= t < decode(hi) */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (o_e4m3_decode((uint8_t)mid) <= t) lo = mid; else hi = mid;
  }
  float a = o_e4m3_decode((uint8_t)lo), b = o_e4m3_decode((uint8_t)hi);
  float m = 0.5f * (a + b); /* exact: one extra mantissa bit */
  if (t < m) return (uint8_t)lo;
  if (t > m) return (uint8_t)hi;
  return (uint8_t)((lo % 2 == 0) ? lo : hi);
}

/* ------------------------------------------------------ hash and signs --- */

/* "lowbias32" 32-bit integer finaliser (C. Wellons, hash-prospector, 2018):
 * xorshift 16, multiply 0x7feb352d, xorshift 15, multiply 0x846ca68b,
 * xorshift 16, all modulo 2^32. */
uint32_t o_mix32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

/* Stream key for a 64-bit seed and a 32-bit stream tag. */
uint32_t o_stream_key(uint64_t seed, uint32_t stream) {
  return o_mix32((uint32_t)seed ^ o_mix32((uint32_t)(seed >> 32) ^ stream));
}

/* 16 random bits for output element i: one hash word per pair of elements,
 * the even element takes the low half-word, the odd one the high half-word. */
uint32_t o_sr_bits(uint64_t sr_seed, uint64_t i) {
  uint32_t k = o_stream_key(sr_seed, 0x5352u);
  uint64_t q = i >> 1;
  uint32_t w = o_mix32(o_mix32(k ^ (uint32_t)(q >> 32)) ^ (uint32_t)q);
  return (i & 1) ? (w >> 16) : (w & 0xFFFFu);
}

/* The 16 signs of the random diagonal: bit j set means d_j = -1. */
uint32_t o_rht_signs(uint64_t rht_seed) {
  return o_mix32(o_stream_key(rht_seed, 0x5248u)) & 0xFFFFu;
}

/* 16-point randomised Hadamard transform [P2 recipe: random Hadamard
 * transform on the wgrad inputs]: y = 1/4 * H16 * (d (.) x) with the Sylvester
 * H16, evaluated as the fast Walsh-Hadamard butterfly with strides 1, 2, 4, 8
 * ((a, b) -> (a + b, a - b) on pairs (i, i + h) with i & h == 0), then the
 * exact scaling by 1/4. */
void o_rht16(const float* in, float* out, uint32_t signs) {
  float w[16];
  for (int j = 0; j < 16; ++j) w[j] = ((signs >> j) & 1) ? -in[j] : in[j];
  for (int h = 1; h < 16; h <<= 1)
    for (int i = 0; i < 16; ++i)
      if ((i & h) == 0) {
        float a = w[i], b = w[i + h];
        w[i] = a + b;
        w[i + h] = a - b;
      }
  for (int j = 0; j < 16; ++j) out[j] = w[j] * 0.25f;
}

/* ----------------------------------------------------------- quantise --- */

/* Gather output-orientation row `orow`, columns [oc, oc+16) as fp32, applying
 * the RHT when asked.  Output orientation is the input itself, or its
 * transpose when OFLAG_TRANSPOSE is set. */
static void gather16(const uint16_t* x, int64_t ld, uint32_t flags, uint32_t signs,
                     int64_t orow, int64_t oc, float* out) {
  float v[16];
  for (int j = 0; j < 16; ++j) {
    int64_t r = (flags & OFLAG_TRANSPOSE) ? oc + j : orow;
    int64_t c = (flags & OFLAG_TRANSPOSE) ? orow : oc + j;
    v[j] = bf16_to_f32(x[r * ld + c]);
  }
  if (flags & OFLAG_RHT) o_rht16(v, out, signs);
  else memcpy(out, v, sizeof v);
}

/* Two-level NVFP4 quantisation of x[rows, cols] (bf16 bit patterns, row
 * stride ld) into codes [orows, ocols/2] and canonical scales
 * [orows, ocols/16], where (orows, ocols) = (rows, cols), or (cols, rows)
 * with OFLAG_TRANSPOSE.  Steps follow [P3]/[P4]/[P5] for the format and [P2]
 * for the 2D, RHT and SR options.  Returns 0, or -1 on a shape it cannot
 * block.  amax_in (nullable) replaces the amax pass. */
int o_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
               uint32_t flags, uint64_t rht_seed, uint64_t sr_seed,
               const float* amax_in, uint8_t* codes, uint8_t* scales,
               float* amax_out, float* sg_out) {
  int64_t orows = (flags & OFLAG_TRANSPOSE) ? cols : rows;
  int64_t ocols = (flags & OFLAG_TRANSPOSE) ? rows : cols;
  if (ocols % 16 != 0) return -1;
  if ((flags & OFLAG_BLOCK_2D) && orows % 16 != 0) return -1;
  uint32_t signs = o_rht_signs(rht_seed);
  int64_t nb = ocols / 16;

  /* 1. tensor amax (after the transform in RHT mode) */
  float amax = 0.0f;
  if (amax_in) {
    amax = *amax_in;
  } else {
#pragma omp parallel for reduction(max : amax) schedule(static)
    for (int64_t o = 0; o < orows; ++o)
      for (int64_t b = 0; b < nb; ++b) {
        float v[16];
        gather16(x, ld, flags, signs, o, b * 16, v);
        for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
      }
  }
  /* 2. tensor scale s_g = amax / (6 * 448) */
  float sg = amax / 2688.0f;
  float den = sg * 6.0f;

  /* 3. per block: scale code, then element codes */
  int64_t tile_rows = (flags & OFLAG_BLOCK_2D) ? 16 : 1;
#pragma omp parallel for schedule(static)
  for (int64_t ot = 0; ot < orows / tile_rows; ++ot) {
    for (int64_t b = 0; b < nb; ++b) {
      float v[16][16];
      float amax_b = 0.0f;
      for (int64_t i = 0; i < tile_rows; ++i) {
        gather16(x, ld, flags, signs, ot * tile_rows + i, b * 16, v[i]);
        for (int j = 0; j < 16; ++j) amax_b = fmaxf(amax_b, fabsf(v[i][j]));
      }
      float t = amax_b / den;
      uint8_t sc = (den == 0.0f || isnan(t)) ? 0 : o_e4m3_encode(t);
      float scf = o_e4m3_decode(sc);
      float enc = (scf == 0.0f) ? 0.0f : 1.0f / (sg * scf);
      for (int64_t i = 0; i < tile_rows; ++i) {
        int64_t o = ot * tile_rows + i;
        scales[o * nb + b] = sc;
        for (int j = 0; j < 16; j += 2) {
          uint8_t q[2];
          for (int h = 0; h < 2; ++h) {
            float val = v[i][j + h] * enc;
            if (flags & OFLAG_SR) {
              uint64_t idx = (uint64_t)o * (uint64_t)ocols + (uint64_t)(b * 16 + j + h);
              q[h] = o_e2m1_encode_sr(val, o_sr_bits(sr_seed, idx));
            } else {
              q[h] = o_e2m1_encode_rne(val);
            }
          }
          codes[o * (ocols / 2) + (b * 16 + j) / 2] = (uint8_t)(q[0] | (q[1] << 4));
        }
      }
    }
  }
  if (amax_out) *amax_out = amax;
  if (sg_out) *sg_out = sg;
  return 0;
}

/* --------------------------------------------------------------- MXFP4 --- */

/* MXFP4, the power-of-two-scaled open format the pages set NVFP4 against
 * ([P3] section "Cos'è NVFP4 ...", second paragraph: NVFP4 has much less
 * error than power-of-two solutions such as MXFP4; [P4] section
 * "Сравнительный ландшафт низкоразрядных форматов": NVFP4 uses smaller
 * quantisation blocks and exact scale factors than the open MXFP4 standard).
 * The pages give no further detail; the reading (the open microscaling
 * layout): 32 consecutive elements of a row share one scale 2^e stored as an
 * E8M0 biased exponent (byte = e + 127), e = floor(log2(amax_b)) - 2 so that
 * the block amax lies in [4, 8) * 2^e, clamped to [-127, 127], and e = -127
 * for an all-zero block; elements are E2M1 round-to-nearest-even of x / 2^e,
 * saturating at 6, sign kept.  No tensor-level scale. */
int o_mx_block_exponent(float amax_b) {
  if (!(amax_b > 0.0f)) return -127;
  int ex = 0;
  (void)frexp((double)amax_b, &ex);  /* amax_b = m * 2^ex, m in [0.5, 1) */
  int e = (ex - 1) - 2;              /* floor(log2(amax_b)) - 2 */
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

int o_quantize_mx(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* codes,
                  uint8_t* scales) {
  if (cols % 32 != 0) return -1;
  int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      float amax_b = 0.0f;
      for (int j = 0; j < 32; ++j) amax_b = fmaxf(amax_b, fabsf(bf16_to_f32(x[r * ld + b * 32 + j])));
      int e = o_mx_block_exponent(amax_b);
      scales[r * nb + b] = (uint8_t)(e + 127);
      for (int j = 0; j < 32; j += 2) {
        uint8_t q[2];
        for (int h = 0; h < 2; ++h) {
          /* x / 2^e is exact in double and representable in float: the
           * bf16 significand has 8 bits and |x / 2^e| < 8 */
          double v = ldexp((double)bf16_to_f32(x[r * ld + b * 32 + j + h]), -e);
          q[h] = o_e2m1_encode_rne((float)v);
        }
        codes[r * (cols / 2) + (b * 32 + j) / 2] = (uint8_t)(q[0] | (q[1] << 4));
      }
    }
  }
  return 0;
}

/* --------------------------------------------------------------- GEMM --- */

/* Dequantised element k of row r: E2M1 value times its block's E4M3 scale;
 * both factors and their product are exact in fp64. */
static double dq(const uint8_t* codes, const uint8_t* scales, int64_t K, int64_t r, int64_t k) {
  uint8_t byte = codes[r * (K / 2) + k / 2];
  uint8_t c = (k & 1) ? (byte >> 4) : (byte & 0xF);
  return (double)o_e2m1_decode(c) * (double)o_e4m3_decode(scales[r * (K / 16) + k / 16]);
}

/* One output of the block-scaled GEMM C = s_gA * s_gB * A * B^T in fp64
 * [P2 recipe: the three MLP GEMMs take NVFP4 operands and return BF16].
 * A is [M, K], B is [N, K], both K-contiguous, canonical scales. */
double o_gemm_elem(const uint8_t* ca, const uint8_t* sa, float sga,
                   const uint8_t* cb, const uint8_t* sb, float sgb,
                   int64_t K, int64_t m, int64_t n) {
  double acc = 0.0;
  for (int64_t k = 0; k < K; ++k) acc += dq(ca, sa, K, m, k) * dq(cb, sb, K, n, k);
  return (double)sga * (double)sgb * acc;
}

/* Full GEMM into out[M, N] (fp64). */
void o_gemm(const uint8_t* ca, const uint8_t* sa, float sga,
            const uint8_t* cb, const uint8_t* sb, float sgb,
            int64_t M, int64_t N, int64_t K, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) out[m * N + n] = o_gemm_elem(ca, sa, sga, cb, sb, sgb, K, m, n);
}

/* Selected outputs (mi[i], ni[i]) into out[i] (fp64). */
void o_gemm_sampled(const uint8_t* ca, const uint8_t* sa, float sga,
                    const uint8_t* cb, const uint8_t* sb, float sgb, int64_t K,
                    const int64_t* mi, const int64_t* ni, int64_t count, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) out[i] = o_gemm_elem(ca, sa, sga, cb, sb, sgb, K, mi[i], ni[i]);
}

/* Element-wise bf16 rounding of an fp64 array. */
void o_bf16_rne_array(const double* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = o_bf16_rne(in[i]);
}

/* Threads the parallel loops may use (1 = single-threaded). */
void o_set_threads(int n) {
#ifdef _OPENMP
  omp_set_num_threads(n > 0 ? n : 1);
#else
  (void)n;
#endif
}

int o_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Element-wise encoders over arrays (used by the exhaustive codec checks). */
void o_e2m1_encode_rne_array(const float* v, uint8_t* out, int64_t n) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = o_e2m1_encode_rne(v[i]);
}

void o_e4m3_encode_array(const float* v, uint8_t* out, int64_t n) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = o_e4m3_encode(v[i]);
}
