// nvfp4_device.cuh -- device helpers shared by the library's kernels:
// element/scale codecs, the counter hash, the 16-point transform, and thin
// inline-PTX wrappers for mbarrier, TMA and tcgen05 (sm_100-family).
#pragma once

#include <cuda.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

// Device status word bits (mirrored by the host's status codes).
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusNonFinite = 2u;

// ------------------------------------------------------------------ bf16 --
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ------------------------------------------------------------------ E4M3 --
// Non-negative block scale -> E4M3 code: round-to-nearest-even, saturating at
// 448 (the hardware conversion with satfinite).  NaN is mapped to 0 by the
// caller before this point.
__device__ __forceinline__ uint32_t e4m3_encode(float t) {
  return (uint32_t)__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3);
}

// E4M3 code -> fp32 (exact: every E4M3 value is an fp16 value).
__device__ __forceinline__ float e4m3_decode(uint32_t code) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
  return __half2float(__half(h));
}

// ------------------------------------------------------------------ E2M1 --
// Two values -> one byte of E2M1 codes, round-to-nearest-even, saturating at
// +-6, sign kept (a negative value that rounds to zero keeps its sign bit:
// code 0x8); s0 lands in the low nibble.  The hardware conversion.
__device__ __forceinline__ uint32_t e2m1x2_rne(float s0, float s1) {
  return (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(s0, s1), __NV_E2M1, cudaRoundNearest);
}

// Stochastic rounding of two values s0, s1 (already scaled by their block's
// encoding factor) with one 32-bit random word r: s0 takes the low half-word
// u0, s1 the high half-word u1.  With lo <= a = |s| < hi adjacent E2M1
// magnitudes, a rounds up iff u * 2^-16 < (a - lo) / (hi - lo); a >= 6
// saturates to 6; the sign is kept.  Returns a word whose top byte is
// code0 | code1 << 4 (the other bytes are scratch).
//
// Scaled by 2^-126, every E2M1 magnitude below 8 lands on a multiple of 2^22
// in the fp32 bit pattern b (0.5 -> 1 << 22, 1 -> 2 << 22, 1.5 -> 3 << 22,
// 2 -> 4 << 22, 3 -> 5 << 22, 4 -> 6 << 22, 6 -> 7 << 22): below 2 the scaled
// values are subnormal or in the first normal binade (uniform spacing
// 2^-149, i.e. b = a * 2^23), above 2 the top mantissa bit is the E2M1 one.
// So lo = b >> 22 and (a - lo) / (hi - lo) = (b mod 2^22) / 2^22, and the
// rule is "round up iff (b mod 2^22) > 64 u": the magnitude code is
// (b + 2^22 - 1 - 64 u) >> 22.  The scaling is exact for a >= 1; below 1 it
// is rounded UP (ceil(a * 2^23)), which leaves every comparison of a * 2^23
// against an integer threshold unchanged, so the decision equals the exact
// rule.  Clamping a to 6 first keeps the code at most 7 (b <= 7 << 22, and 6
// itself never rounds up).
//
// The code of s0 is formed directly in bits 24..27 of
//   x0 = 4 b0 + (2^24 - 1 - 256 u0) + sign0 * 2^27
// (four times the sum above plus 3, which does not change the quotient by
// 2^24; x0 < 2^28), and the code of s1 in bits 28..31 of
//   x1 = 64 b1 + (2^28 - 1 - 4096 u1) + sign1 * 2^31,
// so the pair's byte is the top byte of x0 | (x1 & 0xF0000000).  256 u0 and
// 256 u1 are byte permutations of r.
__device__ __forceinline__ uint32_t sr_pair_b3(float s0, float s1, uint32_t r) {
  const float a0 = fminf(fabsf(s0), 6.0f), a1 = fminf(fabsf(s1), 6.0f);
  const uint32_t b0 = __float_as_uint(__fmul_ru(a0, 0x1p-126f));
  const uint32_t b1 = __float_as_uint(__fmul_ru(a1, 0x1p-126f));
  const uint32_t m0 = __byte_perm(r, 0u, 0x4104);  // u0 << 8
  const uint32_t m1 = __byte_perm(r, 0u, 0x4324);  // u1 << 8
  const uint32_t g0 = ((__float_as_uint(s0) >> 4) & 0x08000000u) | 0x00FFFFFFu;
  const uint32_t g1 = (__float_as_uint(s1) & 0x80000000u) | 0x0FFFFFFFu;
  const uint32_t x0 = b0 * 4u + (g0 - m0);
  const uint32_t x1 = b1 * 64u + (g1 - m1 * 16u);
  return x0 | (x1 & 0xF0000000u);
}

// The top bytes of four words, in order, as one word.
__device__ __forceinline__ uint32_t top_bytes4(uint32_t p0, uint32_t p1, uint32_t p2, uint32_t p3) {
  return __byte_perm(__byte_perm(p0, p1, 0x0073), __byte_perm(p2, p3, 0x0073), 0x5410);
}

// ------------------------------------------------------------------ hash --
// "lowbias32" 32-bit integer finaliser (C. Wellons, hash-prospector, 2018):
// xorshift 16, *0x7feb352d, xorshift 15, *0x846ca68b, xorshift 16 (mod 2^32).
// mix32_tail is everything after the first xorshift.
__host__ __device__ __forceinline__ uint32_t mix32_tail(uint32_t x) {
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}
__host__ __device__ __forceinline__ uint32_t mix32(uint32_t x) { return mix32_tail(x ^ (x >> 16)); }

// Key of a (64-bit seed, 32-bit stream tag) pair.
__host__ __device__ __forceinline__ uint32_t stream_key(uint64_t seed, uint32_t tag) {
  return mix32((uint32_t)seed ^ mix32((uint32_t)(seed >> 32) ^ tag));
}

constexpr uint32_t kTagSR = 0x5352u;   // stochastic-rounding stream
constexpr uint32_t kTagRHT = 0x5248u;  // Hadamard sign stream

// 16 random-sign bits of the transform's diagonal (bit j set: d_j = -1).
__host__ __device__ __forceinline__ uint32_t rht_sign_bits(uint64_t rht_seed) {
  return mix32(stream_key(rht_seed, kTagRHT)) & 0xFFFFu;
}

// --------------------------------------------------------------- RHT-16 --
// y = 1/4 * H16 * (d (.) x): sign flips, Walsh-Hadamard butterflies with
// strides 1, 2, 4, 8 ((a, b) -> (a + b, a - b)), then the exact 1/4 scaling.
// Same operation order as the definition, so results are bit-reproducible.
__device__ __forceinline__ void rht16(float (&v)[16], uint32_t signs) {
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = ((signs >> j) & 1u) ? -v[j] : v[j];
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], 0.25f);
}

// ---- packed fp32 pairs (each lane an IEEE round-to-nearest op, the same
// result as the scalar instruction; two values per instruction) ----
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// The 16-point transform of two columns at once (lane 0: column a, lane 1:
// column b) without the final 1/4: sign flips, then butterflies with strides
// 1, 2, 4, 8, in the definition's operation order.  Every result lies on the
// 2^-133 grid of its bf16 inputs, so the 1/4 that follows is exact and can be
// applied wherever it is cheapest (once to an amax, for instance).
__device__ __forceinline__ void rht16x2_unscaled(float (&a)[16], float (&b)[16], uint32_t signs, uint64_t (&v)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float d = ((signs >> j) & 1u) ? -1.0f : 1.0f;
    v[j] = f2_mul(f2_pack(a[j], b[j]), f2_pack(d, d));
  }
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const uint64_t x = v[i], y = v[i + h];
        v[i] = f2_add(x, y);
        v[i + h] = f2_sub(x, y);
      }
    }
  }
}

__device__ __forceinline__ void rht16x2_unscaled(float (&a)[16], float (&b)[16], uint32_t signs) {
  uint64_t v[16];
  rht16x2_unscaled(a, b, signs, v);
#pragma unroll
  for (int j = 0; j < 16; ++j) f2_unpack(v[j], a[j], b[j]);
}

// The full transform of two columns: the butterflies, then the exact 1/4.
__device__ __forceinline__ void rht16x2(float (&a)[16], float (&b)[16], uint32_t signs) {
  uint64_t v[16];
  rht16x2_unscaled(a, b, signs, v);
  const uint64_t q = f2_pack(0.25f, 0.25f);
#pragma unroll
  for (int j = 0; j < 16; ++j) f2_unpack(f2_mul(v[j], q), a[j], b[j]);
}

// ---------------------------------------------------------- block encode --
// Scale of one block from its amax: sc = E4M3(amax_b / (s_g * 6)) or 0.
__device__ __forceinline__ uint32_t block_scale_code(float amax_b, float den) {
  if (den == 0.0f) return 0u;
  const float t = __fdiv_rn(amax_b, den);
  return (t != t) ? 0u : e4m3_encode(t);
}

// Encoding factor 1 / (s_g * decode(sc)), 0 when the scale is 0.
__device__ __forceinline__ float block_enc(float sg, uint32_t sc) {
  const float scf = e4m3_decode(sc);
  return (scf == 0.0f) ? 0.0f : __frcp_rn(__fmul_rn(sg, scf));
}

// Every encoding factor of a tensor (one per E4M3 code; codes above 0x7E
// never occur) into shared memory, by the whole CTA.  The caller
// synchronises before use.
__device__ __forceinline__ void fill_enc_table(float* tab, float sg) {
  for (int c = threadIdx.x; c < 128; c += blockDim.x) tab[c] = block_enc(sg, (uint32_t)c);
}

// Random words of the 8 pairs q0 .. q0 + 7 of a 16-element block (q0 a
// multiple of 8, so the pairs share hi32 and hk).  w[j] = mix32(hk ^ (q0lo +
// j)); since q0lo + j == q0lo ^ j and j < 8 leaves bits 16 and up unchanged,
// the first xorshift is taken once for the block: mix32(g ^ j) ==
// mix32_tail((g ^ (g >> 16)) ^ j) with g = hk ^ q0lo.
__device__ __forceinline__ void sr_words8(uint32_t hk, uint32_t q0lo, uint32_t (&w)[8]) {
  uint32_t g = hk ^ q0lo;
  g ^= g >> 16;
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = mix32_tail(g ^ (uint32_t)j);
}

// SR codes of 16 values already multiplied by the block's encoding factor:
// hk is the hash key of the block's pair range, q0 the pair index of element
// 0 (8 pairs, one hash word each; the even element uses the low half-word).
__device__ __forceinline__ uint2 encode16_sr_scaled(const float (&sv)[16], uint32_t hk, uint64_t q0) {
  uint32_t r[8];
  sr_words8(hk, (uint32_t)q0, r);
  uint32_t p[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) p[j] = sr_pair_b3(sv[2 * j], sv[2 * j + 1], r[j]);
  return make_uint2(top_bytes4(p[0], p[1], p[2], p[3]), top_bytes4(p[4], p[5], p[6], p[7]));
}

// RNE codes of 16 values already multiplied by the block's encoding factor.
__device__ __forceinline__ uint2 encode16_rne_scaled(const float (&sv)[16]) {
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 16; j += 2) w[j / 8] |= e2m1x2_rne(sv[j], sv[j + 1]) << (8 * ((j / 2) % 4));
  return make_uint2(w[0], w[1]);
}

// Scale 16 values by a common factor (packed pairs; each lane one IEEE
// round-to-nearest multiply).
__device__ __forceinline__ void scale16(float (&v)[16], float enc) {
  const uint64_t e2 = f2_pack(enc, enc);
#pragma unroll
  for (int j = 0; j < 16; j += 2) f2_unpack(f2_mul(f2_pack(v[j], v[j + 1]), e2), v[j], v[j + 1]);
}

__device__ __forceinline__ uint2 encode16_rne(float (&v)[16], float enc) {
  scale16(v, enc);
  return encode16_rne_scaled(v);
}

__device__ __forceinline__ uint2 encode16_sr(float (&v)[16], float enc, uint32_t hk, uint64_t q0) {
  scale16(v, enc);
  return encode16_sr_scaled(v, hk, q0);
}

// Offset of scale (row r, block kb) in the MMA layout (cols/64 atoms per
// 128-row band, 512 bytes per atom).
__host__ __device__ __forceinline__ int64_t mma_scale_offset(int64_t r, int64_t kb, int64_t atoms_per_band) {
  return ((r >> 7) * atoms_per_band + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3);
}

// --------------------------------------------------------------- PTX ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase.  Returns false (and raises the timeout
// bit in *status) if the phase did not complete within `limit_ns`.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* status,
                                          uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++spins & 1023u) == 0u && globaltimer_ns() - t0 > limit_ns) {
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
  return true;
}

// Bounded wait with the whole spin inside one asm block (no data-dependent
// control flow in the caller's code): true once the phase with `parity` has
// completed; after about limit_ns it raises the timeout bit and returns false.
// Loops that issue tcgen05.mma keep their full rate only with this form.
__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity, uint32_t* status,
                                               uint64_t limit_ns = 2000000000ull) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P1, P2;\n\t.reg .u64 t0, t1;\n\t.reg .u32 n;\n\t"
      "mov.u64 t0, %%globaltimer;\n\tmov.u32 n, 0;\n"
      "WAIT_%=:\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
      "@P1 bra.uni DONE_%=;\n\t"
      "add.u32 n, n, 1;\n\t"
      "and.b32 n, n, 1023;\n\t"
      "setp.ne.u32 P2, n, 0;\n\t"
      "@P2 bra.uni WAIT_%=;\n\t"
      "mov.u64 t1, %%globaltimer;\n\t"
      "sub.u64 t1, t1, t0;\n\t"
      "setp.lt.u64 P2, t1, %3;\n\t"
      "@P2 bra.uni WAIT_%=;\n\t"
      "mov.u32 %0, 0;\n\t"
      "bra.uni END_%=;\n"
      "DONE_%=:\n\t"
      "mov.u32 %0, 1;\n"
      "END_%=:\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "l"(limit_ns)
      : "memory");
  if (!ok) atomicOr(status, kStatusTimeout);
  return ok != 0;
}

// True in exactly one lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}" : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D TMA tile load into this CTA's shared memory whose completion is
// counted on an mbarrier given by its cluster address, which may lie in the
// other CTA of the pair (CTA-pair form).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

// 2-D TMA tile load into this CTA's shared memory, completion counted on
// this CTA's mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 3-D TMA tile load into this CTA's shared memory, completion counted on
// this CTA's mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"((uint64_t)src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 16 consecutive 32-bit columns: thread i writes lane (base + i).
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread i receives lane (base + i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// ---- clusters (CTA pairs) ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive on an mbarrier given by its cluster address (possibly in the peer
// CTA).  Default (CTA-scope release) semantics: what it publishes are
// completed tensor-memory accesses ordered by tcgen05 fences, and a
// cluster-scope release here measured 2x slower for the whole GEMM.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for barriers that receive arrivals from the peer CTA or from
// a multicast tcgen05.commit.  Same contract as mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint32_t* status,
                                                  uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (!mbar_try_wait_cluster(bar, parity)) {
    if ((++spins & 1023u) == 0u && globaltimer_ns() - t0 > limit_ns) {
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
  return true;
}

// ---- bulk tensor stores ----
// 2-D TMA store of a shared-memory box to global memory (bulk-group
// completion); elements outside the tensor map's extent are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
               ::"l"((uint64_t)map), "r"(src), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N committed bulk groups are still in flight.
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// ---- tcgen05, CTA-pair forms ----
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Arrive on the mbarrier at the same shared-memory offset in every CTA of
// `mask` once this thread's previously issued pair MMAs have completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
      ::"r"(bar), "h"(mask)
      : "memory");
}

// Pair MMA (M = 256 over the two CTAs): D (+)= (A * SFA) x (B * SFB)^T.  Each
// CTA supplies half of A's rows and half of B's rows from the same
// shared-memory offsets, holds its half of D in its own tensor memory, and
// holds its own A scales and all of B's scales in its own tensor memory.
__device__ __forceinline__ void tc_mma_nvf4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

}  // namespace nvfp4
