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
// Two magnitudes (>= 0) -> one byte of E2M1 codes, round-to-nearest-even with
// saturation at 6; a0 lands in the low nibble.  Feeding magnitudes keeps the
// sign decision out of the conversion; the caller ORs the sign bits in.
__device__ __forceinline__ uint32_t e2m1x2_rne_mag(float a0, float a1) {
  return (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(a0, a1), __NV_E2M1, cudaRoundNearest);
}

// Stochastic rounding of a magnitude a >= 0: the E2M1 code (0..7) given
// u64 = u << 6 for 16 random bits u.  With lo <= a < hi adjacent E2M1
// magnitudes the value rounds up iff u * 2^-16 < (a - lo) / (hi - lo).
//
// Scaled by 2^-126, every E2M1 magnitude below 8 lands on a multiple of 2^22
// in the fp32 bit pattern b (0.5 -> 1 << 22, 1 -> 2 << 22, 1.5 -> 3 << 22,
// 2 -> 4 << 22, 3 -> 5 << 22, 4 -> 6 << 22, 6 -> 7 << 22): below 2 the scaled
// values are subnormal or in the first normal binade (uniform spacing
// 2^-149, i.e. b = a * 2^23), above 2 the top mantissa bit is the E2M1 one.
// So lo = b >> 22 and (a - lo) / (hi - lo) = (b mod 2^22) / 2^22, and the
// rule is "round up iff (b mod 2^22) > u * 64", i.e. add 2^22 - 1 - 64 u and
// keep the bits above 22.  The scaling is exact for a >= 1; below 1 it is
// rounded UP (ceil(a * 2^23)), which leaves every comparison of a * 2^23
// against an integer threshold unchanged, so the decision equals the exact
// rule.  Codes above 7 (a >= 6, after rounding) saturate to 7.
__device__ __forceinline__ uint32_t e2m1_sr_code(float a, uint32_t u64) {
  const uint32_t b = __float_as_uint(__fmul_ru(a, 0x1p-126f));
  return min((b + 0x3FFFFFu - u64) >> 22, 7u);
}

__device__ __forceinline__ uint32_t sign_nibble(float v) { return (__float_as_uint(v) >> 31) << 3; }

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
// column b), same operation order as rht16: sign flips, butterflies with
// strides 1, 2, 4, 8, then the exact 1/4.
__device__ __forceinline__ void rht16x2(float (&a)[16], float (&b)[16], uint32_t signs) {
  uint64_t v[16];
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

// Encode 16 values with a common factor into 8 bytes (two 32-bit words),
// round-to-nearest-even.
__device__ __forceinline__ uint2 encode16_rne(const float (&v)[16], float enc) {
  const uint64_t e2 = f2_pack(enc, enc);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    float s0, s1;
    f2_unpack(f2_mul(f2_pack(v[j], v[j + 1]), e2), s0, s1);
    uint32_t byte = e2m1x2_rne_mag(fabsf(s0), fabsf(s1));
    byte |= sign_nibble(s0) | (sign_nibble(s1) << 4);
    w[j / 8] |= byte << (8 * ((j / 2) % 4));
  }
  return make_uint2(w[0], w[1]);
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

// SR codes (sign included) of two values s0, s1 (already scaled by the
// block's encoding factor) from one random word r: s0 uses the low
// half-word, s1 the high half-word.  Returns c0 | c1 << 4.  (Moving the
// threshold and packing arithmetic onto high products and multiply-adds
// measured slower.)
__device__ __forceinline__ uint32_t sr_pair_codes(float s0, float s1, uint32_t r) {
  const uint32_t c0 = e2m1_sr_code(fabsf(s0), (r << 6) & 0x3FFFC0u) | sign_nibble(s0);
  const uint32_t c1 = e2m1_sr_code(fabsf(s1), (r >> 10) & 0x3FFFC0u) | sign_nibble(s1);
  return c0 | (c1 << 4);
}

// SR codes of 16 values already multiplied by the block's encoding factor.
__device__ __forceinline__ uint2 encode16_sr_scaled(const float (&sv)[16], uint32_t hk, uint64_t q0) {
  uint32_t r[8];
  sr_words8(hk, (uint32_t)q0, r);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 16; j += 2) w[j / 8] += sr_pair_codes(sv[j], sv[j + 1], r[j / 2]) << (8 * ((j / 2) % 4));
  return make_uint2(w[0], w[1]);
}

// RNE codes of 16 values already multiplied by the block's encoding factor.
__device__ __forceinline__ uint2 encode16_rne_scaled(const float (&sv)[16]) {
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    uint32_t byte = e2m1x2_rne_mag(fabsf(sv[j]), fabsf(sv[j + 1]));
    byte |= sign_nibble(sv[j]) | (sign_nibble(sv[j + 1]) << 4);
    w[j / 8] |= byte << (8 * ((j / 2) % 4));
  }
  return make_uint2(w[0], w[1]);
}

// Same with stochastic rounding: hk is the per-block hash key, q0 the pair
// index of element 0 (8 pairs, one hash word each; the even element uses the
// low half-word).
__device__ __forceinline__ uint2 encode16_sr(const float (&v)[16], float enc, uint32_t hk,
                                             uint64_t q0) {
  uint32_t r[8];
  sr_words8(hk, (uint32_t)q0, r);
  const uint64_t e2 = f2_pack(enc, enc);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    float s0, s1;
    f2_unpack(f2_mul(f2_pack(v[j], v[j + 1]), e2), s0, s1);
    w[j / 8] += sr_pair_codes(s0, s1, r[j / 2]) << (8 * ((j / 2) % 4));
  }
  return make_uint2(w[0], w[1]);
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
