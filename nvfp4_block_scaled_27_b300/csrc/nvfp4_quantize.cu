// nvfp4_quantize.cu -- HBM-bound NVFP4 quantisers for sm_103a.
//
// Format (E2M1 elements, one E4M3 scale per 16 values, one FP32 tensor
// scale): "NVFP4: cos'è e come supera FP8 e BF16 nell'intelligenza
// artificiale", section "Cos'è NVFP4 ..."; "FP4" (chaitex.ru/fp4), section
// "Математическая структура FP4".  Recipe options (2D weight blocks, random
// Hadamard transform for wgrad operands, stochastic rounding for gradients):
// readjensen.com NVFP4 training-recipe article, MLP data-flow paragraph.
//
// Kernels
//   amax_plain    : one read of the input, eight 16-byte loads in flight per
//                   thread, packed bf16 integer max, one atomicMax per CTA.
//   amax_tile     : 64 x 256 input tiles staged in shared memory; the plain
//                   amax and/or the amax after the column-wise transform.
//   amax_rht_rows : amax after the row-wise transform.
//   quant_rows_*  : row-wise blocks straight from registers (1D) or from a
//                   staged tile (2D); a warp reads 1 KiB of contiguous input
//                   per 16-element step and writes 256 contiguous code bytes.
//   quant_cols    : blocks along the input's rows (transposed output): a
//                   64 x 256 input tile is staged in shared memory with
//                   coalesced 16-byte copies, then each thread owns a column
//                   pair and walks four 16-row chunks.
//   quant_dual    : both operands of one tensor from one staged tile.
// Every CTA keeps the tensor's 128 encoding factors 1 / (s_g * scale) in
// shared memory, so a block's factor is one lookup.  All arithmetic on
// values is single-rounded IEEE fp32 (no contraction), so results are
// bit-reproducible.
#include <float.h>

#include <mutex>
#include <unordered_map>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

struct QuantParams {
  const uint16_t* x;
  int64_t rows, cols, ld;  // input shape and row stride (elements)
  int64_t orows, ocols;    // output shape
  uint8_t* codes;
  uint8_t* scales;
  const float* amax_src;  // amax to use (caller's amax_in, or the amax pass result)
  float* amax_out;        // written once when amax came from the caller, else null
  float* sg_out;
  uint32_t* status;
  uint32_t sr_hk[2];      // hash key of pair indices with hi32 = 0 and 1: mix32(key ^ hi32)
  uint32_t rht_signs;
};

// ------------------------------------------------------------- helpers --
__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float (&v)[16]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16_lo(w[i]);
    v[2 * i + 1] = bf16_hi(w[i]);
  }
}

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// max(|a|, |b|, |c|) in one instruction (three-input max over magnitudes).
__device__ __forceinline__ float absmax3(float a, float b, float c) {
  float r;
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// max |v[j]| over 16 values.
__device__ __forceinline__ float absmax16(const float (&v)[16]) {
  float m = absmax3(v[0], v[1], v[2]);
#pragma unroll
  for (int j = 3; j < 15; j += 2) m = absmax3(m, v[j], v[j + 1]);
  return absmax3(m, v[15], v[15]);
}

// CTA-wide max of a non-negative fp32 bit pattern, then one atomicMax.
__device__ __forceinline__ void cta_amax_commit(uint32_t m, float* out) {
  __shared__ uint32_t red[32];
  m = warp_max_u32(m);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = (lane < (int)(blockDim.x >> 5)) ? red[lane] : 0u;
    m = warp_max_u32(m);
    if (lane == 0 && m != 0u) atomicMax(reinterpret_cast<unsigned int*>(out), m);
  }
}

// Max |bf16| over a packed pair, as a 15-bit magnitude pattern per half.
__device__ __forceinline__ uint32_t absmax_pairs(uint32_t m, const uint4& u) {
  m = __vmaxu2(m, u.x & 0x7FFF7FFFu);
  m = __vmaxu2(m, u.y & 0x7FFF7FFFu);
  m = __vmaxu2(m, u.z & 0x7FFF7FFFu);
  m = __vmaxu2(m, u.w & 0x7FFF7FFFu);
  return m;
}

__device__ __forceinline__ uint32_t pairs_to_f32_bits(uint32_t m) {
  return max(m & 0xFFFFu, m >> 16) << 16;  // bf16 magnitude -> fp32 pattern
}

// Tensor scale and the first-CTA bookkeeping (s_g, amax copy, non-finite flag).
__device__ __forceinline__ float tensor_scale(const QuantParams& p, float& amax) {
  amax = *p.amax_src;
  const float sg = __fdiv_rn(amax, 2688.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *p.sg_out = sg;
    if (p.amax_out) *p.amax_out = amax;
    if (!(amax <= FLT_MAX)) atomicOr(p.status, kStatusNonFinite);
  }
  return sg;
}

// Hash key of the pair range starting at pair index q0 (the tensor has fewer
// than 2^34 elements, so hi32(q0) is 0 or 1).
__device__ __forceinline__ uint32_t pair_key(const QuantParams& p, uint64_t q0) {
  return (q0 >> 32) ? p.sr_hk[1] : p.sr_hk[0];
}

// ----------------------------------------------------------------- amax --
// Plain amax of a bf16 matrix (vpr 16-byte vectors per row, row stride ldv
// vectors).  Magnitudes are compared as integers (exact for bf16).  Eight
// 16-byte loads in flight per thread keep enough bytes outstanding per SM to
// cover DRAM latency.
__global__ void __launch_bounds__(256) amax_plain_kernel(const uint4* __restrict__ x, int64_t rows,
                                                         int64_t vpr, int64_t ldv, float* out) {
  uint32_t m = 0u;
  if (vpr == ldv) {
    const int64_t n = rows * vpr;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 7 * stride < n; i += 8 * stride) {
      uint4 a[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) a[k] = ldg_nc(x + i + k * stride);
#pragma unroll
      for (int k = 0; k < 8; ++k) m = absmax_pairs(m, a[k]);
    }
    for (; i < n; i += stride) m = absmax_pairs(m, ldg_nc(x + i));
  } else {
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x)
      for (int64_t v = threadIdx.x; v < vpr; v += blockDim.x) m = absmax_pairs(m, ldg_nc(x + r * ldv + v));
  }
  cta_amax_commit(pairs_to_f32_bits(m), out);
}

// amax after the row-wise transform: every 16 consecutive elements of a row.
// max |1/4 w| = 1/4 max |w| exactly, so the 1/4 is applied once at the end.
__global__ void __launch_bounds__(256) amax_rht_rows_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                            int64_t cols, int64_t ld, uint32_t signs,
                                                            float* out) {
  float m = 0.0f;
  const uint32_t nb = (uint32_t)(cols / 16);
  const uint32_t total = (uint32_t)(rows * nb);
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const uint32_t r = i / nb, b = i - r * nb;
    const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)r * ld + (int64_t)b * 16);
    float v[16];
    unpack16(ldg_nc(src), ldg_nc(src + 1), v);
    rht16(v, signs);
    m = fmaxf(m, absmax16(v));
  }
  cta_amax_commit(__float_as_uint(m), out);
}

// Two CTA-wide maxima at once (one shared scratch, one barrier), then one
// atomicMax each (a null output is skipped).
__device__ __forceinline__ void cta_amax_commit2(uint32_t m1, float* out1, uint32_t m2, float* out2) {
  __shared__ uint32_t red2[2][32];
  m1 = warp_max_u32(m1);
  m2 = warp_max_u32(m2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red2[0][warp] = m1;
    red2[1][warp] = m2;
  }
  __syncthreads();
  if (warp == 0) {
    const bool in = lane < (int)(blockDim.x >> 5);
    m1 = warp_max_u32(in ? red2[0][lane] : 0u);
    m2 = warp_max_u32(in ? red2[1][lane] : 0u);
    if (lane == 0) {
      if (out1 && m1 != 0u) atomicMax(reinterpret_cast<unsigned int*>(out1), m1);
      if (out2 && m2 != 0u) atomicMax(reinterpret_cast<unsigned int*>(out2), m2);
    }
  }
}

// ------------------------------------------------------ staged tiles --
constexpr int kColTileRows = 64;   // input rows per tile (4 blocks)
constexpr int kColTileCols = 256;  // input columns per tile
constexpr int kColThreads = 128;   // one thread per column pair

constexpr uint32_t kTileBytes = kColTileRows * kColTileCols * 2;

// Shared memory of a tile-staged kernel: the input tile (the TMA box,
// row-major, 512 bytes per row) and the mbarrier its copy completes on.
struct TileSmem {
  __align__(128) uint32_t tile[kColTileRows][kColTileCols / 2];
  __align__(8) uint64_t bar;
};

// Walks the input's 64 x 256 tiles (forwards, or backwards with kReverse)
// with a grid stride; each tile arrives in shared memory by one TMA copy
// that thread 0 issues and every thread waits for (elements outside the
// input read as zero), then body(r0, c0) runs on it.  One barrier per tile
// separates the body's reads from the next copy; a wait that expires (the
// timeout bit is then raised) ends the walk for the whole CTA.  The caller
// initialises ts.bar and synchronises before the first call.
template <bool kReverse, typename Body>
__device__ __forceinline__ void for_each_tile(const CUtensorMap& map, TileSmem& ts, int64_t rows, int64_t cols,
                                              uint32_t* status, Body&& body) {
  const int64_t tiles_c = (cols + kColTileCols - 1) / kColTileCols;
  const int64_t ntiles = ((rows + kColTileRows - 1) / kColTileRows) * tiles_c;
  const int64_t step = kReverse ? -(int64_t)gridDim.x : (int64_t)gridDim.x;
  int64_t t = kReverse ? ntiles - 1 - blockIdx.x : blockIdx.x;
  if (t < 0 || t >= ntiles) return;
  const uint32_t bar = smem_u32(&ts.bar), dst = smem_u32(&ts.tile[0][0]);
  auto issue = [&](int64_t tt) {
    const int64_t tr = tt / tiles_c, tc = tt - tr * tiles_c;
    fence_proxy_async();  // earlier generic reads of the tile before the async-proxy write
    mbar_arrive_expect_tx(bar, kTileBytes);
    tma_load_2d(dst, &map, (int32_t)(tc * kColTileCols), (int32_t)(tr * kColTileRows), bar);
  };
  if (threadIdx.x == 0) issue(t);
  uint32_t phase = 0u;
  while (true) {
    const bool ok = mbar_wait(bar, phase, status);
    phase ^= 1u;
    const int64_t tr = t / tiles_c, tc = t - tr * tiles_c;
    body(tr * kColTileRows, tc * kColTileCols);
    const int64_t tn = t + step;
    if (__syncthreads_or(!ok) || tn < 0 || tn >= ntiles) break;
    t = tn;
    if (threadIdx.x == 0) issue(t);
  }
}

__device__ __forceinline__ void tile_smem_init(TileSmem& ts) {
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ts.bar), 1);
    fence_barrier_init();
  }
}

// The 32 values of a thread's column pair in one 16-row chunk of a staged
// tile (v0: column 2 tid, v1: column 2 tid + 1).
__device__ __forceinline__ void load_chunk_cols(const uint32_t (&tile)[kColTileRows][kColTileCols / 2], int k,
                                                float (&v0)[16], float (&v1)[16]) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t w = tile[16 * k + i][tid];
    v0[i] = bf16_lo(w);
    v1[i] = bf16_hi(w);
  }
}

// amax of a bf16 matrix over staged 64 x 256 tiles: the plain amax (kPlain)
// and/or the amax after the column-wise transform (kCols: every 16
// consecutive rows of a column, 1/4 applied once at the end).  Zero-filled
// padding does not change either maximum.
template <bool kPlain, bool kCols>
__global__ void __launch_bounds__(kColThreads) amax_tile_kernel(const __grid_constant__ CUtensorMap map, int64_t rows,
                                                                int64_t cols, uint32_t signs, float* out_plain,
                                                                float* out_cols, uint32_t* status) {
  __shared__ TileSmem ts;
  tile_smem_init(ts);
  __syncthreads();
  uint32_t mp = 0u;
  float mc = 0.0f;
  for_each_tile<false>(map, ts, rows, cols, status, [&](int64_t, int64_t) {
#pragma unroll 1
    for (int k = 0; k < kColTileRows / 16; ++k) {
      if (kPlain) {
#pragma unroll
        for (int i = 0; i < 16; ++i) mp = __vmaxu2(mp, ts.tile[16 * k + i][threadIdx.x] & 0x7FFF7FFFu);
      }
      if (kCols) {
        float v0[16], v1[16];
        load_chunk_cols(ts.tile, k, v0, v1);
        rht16x2_unscaled(v0, v1, signs);
        mc = absmax3(mc, absmax16(v0), absmax16(v1));
      }
    }
  });
  cta_amax_commit2(pairs_to_f32_bits(mp), kPlain ? out_plain : nullptr, __float_as_uint(__fmul_rn(mc, 0.25f)),
                   kCols ? out_cols : nullptr);
}

// ------------------------------------------------------- row-wise, 1D --
template <bool kSR, bool kRHT, bool kMMA>
__device__ __forceinline__ void quant_block_1d(const QuantParams& p, const float* enc_tab, uint32_t i, uint32_t nb,
                                               const uint4& a, const uint4& b4, float den) {
  float v[16];
  unpack16(a, b4, v);
  if (kRHT) rht16(v, p.rht_signs);
  const uint32_t sc = block_scale_code(absmax16(v), den);
  const float enc = enc_tab[sc];
  uint2 q;
  if (kSR) {
    const uint64_t q0 = (uint64_t)i * 8u;  // element index 16 i, pair index 8 i
    q = encode16_sr(v, enc, pair_key(p, q0), q0);
  } else {
    q = encode16_rne(v, enc);
  }
  *reinterpret_cast<uint2*>(p.codes + (int64_t)i * 8) = q;
  const uint32_t r = i / nb, kb = i - r * nb;
  const int64_t off = kMMA ? mma_scale_offset(r, kb, nb / 4) : (int64_t)i;
  p.scales[off] = (uint8_t)sc;
}

// One thread per 16-element block, two blocks in flight per thread.  The
// output [rows, cols/2] is contiguous, so block i's codes sit at byte 8 i and
// its elements have output indices 16 i .. 16 i + 15.
template <bool kSR, bool kRHT, bool kMMA>
__global__ void __launch_bounds__(256) quant_rows_1d_kernel(QuantParams p) {
  __shared__ float enc_tab[128];
  float amax;
  const float sg = tensor_scale(p, amax);
  const float den = __fmul_rn(sg, 6.0f);
  fill_enc_table(enc_tab, sg);
  __syncthreads();
  const uint32_t nb = (uint32_t)(p.ocols / 16);
  const uint32_t total = (uint32_t)(p.orows * nb);
  const uint32_t stride = gridDim.x * blockDim.x;
  uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + stride < total; i += 2 * stride) {
    const uint32_t j = i + stride;
    const uint32_t ri = i / nb, rj = j / nb;
    const uint4* si = reinterpret_cast<const uint4*>(p.x + (int64_t)ri * p.ld + (int64_t)(i - ri * nb) * 16);
    const uint4* sj = reinterpret_cast<const uint4*>(p.x + (int64_t)rj * p.ld + (int64_t)(j - rj * nb) * 16);
    const uint4 a0 = ldg_nc(si), a1 = ldg_nc(si + 1), b0 = ldg_nc(sj), b1 = ldg_nc(sj + 1);
    quant_block_1d<kSR, kRHT, kMMA>(p, enc_tab, i, nb, a0, a1, den);
    quant_block_1d<kSR, kRHT, kMMA>(p, enc_tab, j, nb, b0, b1, den);
  }
  if (i < total) {
    const uint32_t ri = i / nb;
    const uint4* si = reinterpret_cast<const uint4*>(p.x + (int64_t)ri * p.ld + (int64_t)(i - ri * nb) * 16);
    quant_block_1d<kSR, kRHT, kMMA>(p, enc_tab, i, nb, ldg_nc(si), ldg_nc(si + 1), den);
  }
}

// ------------------------------------------------- column-wise (x^T) --
// Column-wise (transposed) quantisation of a staged tile.  Output row c =
// input column c, output column r = input row r.  Blocks run along the
// input's rows; with kTwoD the 16x16 tile amax is shared by the 8 threads
// (16 columns) of a tile via shuffles.
template <bool kSR, bool kRHT, bool kTwoD, bool kMMA>
__device__ __forceinline__ void cols_tile(const QuantParams& p, const float* enc_tab,
                                          const uint32_t (&tile)[kColTileRows][kColTileCols / 2],
                                          int64_t r0, int64_t c0, float den) {
  const int64_t R = p.rows, C = p.cols;
  const int tid = threadIdx.x;
  const int64_t kb_per_row = R / 16;  // output blocks per output row
  const int64_t c = c0 + 2 * tid;  // this thread's two output rows: c, c + 1
  const bool col_ok = c < C;
  // Codes and scales of the tile's four 16-row chunks are collected and
  // written together when the tile is whole: 32 contiguous code bytes per
  // output row (two 16-byte stores) and one 32-bit word of four scales.
  const bool whole = (r0 + kColTileRows <= R) && ((R & 31) == 0) &&
                     ((reinterpret_cast<uintptr_t>(p.codes) & 15u) == 0);
  // Codes shift through four registers per output row, oldest chunk first,
  // so the chunk loop needs no indexed arrays and can stay rolled (the
  // unrolled body overflows the instruction cache).
  uint2 qa0 = make_uint2(0u, 0u), qa1 = qa0, qa2 = qa0, qa3 = qa0;
  uint2 qb0 = qa0, qb1 = qa0, qb2 = qa0, qb3 = qa0;
  uint32_t sca = 0u, scb = 0u;
  // pair indices of the two output rows' first elements in this tile; each
  // 16-row chunk advances them by 8
  uint64_t pa = ((uint64_t)c * (uint64_t)R + (uint64_t)r0) >> 1;
  uint64_t pb = pa + (uint64_t)(R >> 1);
#pragma unroll 1
  for (int k = 0; k < kColTileRows / 16; ++k, pa += 8u, pb += 8u) {
    const int64_t rb = r0 + 16 * k;  // first input row of the block
    if (rb >= R) break;              // uniform across the CTA
    float v0[16], v1[16];
    load_chunk_cols(tile, k, v0, v1);
    if (kRHT) rht16x2(v0, v1, p.rht_signs);
    float a0 = absmax16(v0), a1 = absmax16(v1);
    if (kTwoD) {
      float a = fmaxf(a0, a1);
      a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
      a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
      a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));
      a0 = a1 = a;
    }
    if (!col_ok) continue;
    const uint32_t sc0 = block_scale_code(a0, den), sc1 = block_scale_code(a1, den);
    const uint64_t e01 = f2_pack(enc_tab[sc0], enc_tab[sc1]);
#pragma unroll
    for (int i = 0; i < 16; ++i) f2_unpack(f2_mul(f2_pack(v0[i], v1[i]), e01), v0[i], v1[i]);
    uint2 q0, q1;
    if (kSR) {
      q0 = encode16_sr_scaled(v0, pair_key(p, pa), pa);
      q1 = encode16_sr_scaled(v1, pair_key(p, pb), pb);
    } else {
      q0 = encode16_rne_scaled(v0);
      q1 = encode16_rne_scaled(v1);
    }
    qa0 = qa1; qa1 = qa2; qa2 = qa3; qa3 = q0;
    qb0 = qb1; qb1 = qb2; qb2 = qb3; qb3 = q1;
    sca = (sca >> 8) | (sc0 << 24);
    scb = (scb >> 8) | (sc1 << 24);
    if (!whole) {
      *reinterpret_cast<uint2*>(p.codes + c * (R / 2) + rb / 2) = q0;
      *reinterpret_cast<uint2*>(p.codes + (c + 1) * (R / 2) + rb / 2) = q1;
      const int64_t kb = rb / 16;
      if (kMMA) {
        p.scales[mma_scale_offset(c, kb, kb_per_row / 4)] = (uint8_t)sc0;
        p.scales[mma_scale_offset(c + 1, kb, kb_per_row / 4)] = (uint8_t)sc1;
      } else {
        p.scales[c * kb_per_row + kb] = (uint8_t)sc0;
        p.scales[(c + 1) * kb_per_row + kb] = (uint8_t)sc1;
      }
    }
  }
  if (whole && col_ok) {
    uint8_t* o0 = p.codes + c * (R / 2) + r0 / 2;
    uint8_t* o1 = o0 + R / 2;
    *reinterpret_cast<uint4*>(o0) = make_uint4(qa0.x, qa0.y, qa1.x, qa1.y);
    *reinterpret_cast<uint4*>(o0 + 16) = make_uint4(qa2.x, qa2.y, qa3.x, qa3.y);
    *reinterpret_cast<uint4*>(o1) = make_uint4(qb0.x, qb0.y, qb1.x, qb1.y);
    *reinterpret_cast<uint4*>(o1 + 16) = make_uint4(qb2.x, qb2.y, qb3.x, qb3.y);
    const int64_t kb0 = r0 / 16;  // a multiple of 4: the four scales share one word
    if (kMMA) {
      *reinterpret_cast<uint32_t*>(p.scales + mma_scale_offset(c, kb0, kb_per_row / 4)) = sca;
      *reinterpret_cast<uint32_t*>(p.scales + mma_scale_offset(c + 1, kb0, kb_per_row / 4)) = scb;
    } else {
      uint8_t* s0 = p.scales + c * kb_per_row + kb0;
      uint8_t* s1 = s0 + kb_per_row;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        s0[k] = (uint8_t)(sca >> (8 * k));
        s1[k] = (uint8_t)(scb >> (8 * k));
      }
    }
  }
}

template <bool kSR, bool kRHT, bool kTwoD, bool kMMA>
__global__ void __launch_bounds__(kColThreads, 6) quant_cols_kernel(const __grid_constant__ CUtensorMap map,
                                                                    QuantParams p) {
  __shared__ TileSmem ts;
  __shared__ float enc_tab[128];
  float amax;
  const float sg = tensor_scale(p, amax);
  const float den = __fmul_rn(sg, 6.0f);
  fill_enc_table(enc_tab, sg);
  tile_smem_init(ts);
  __syncthreads();
  // Tiles in reverse order: the amax pass walked them forwards, so the first
  // tiles encoded are the ones it left in L2.
  for_each_tile<true>(map, ts, p.rows, p.cols, p.status, [&](int64_t r0, int64_t c0) {
    cols_tile<kSR, kRHT, kTwoD, kMMA>(p, enc_tab, ts.tile, r0, c0, den);
  });
}

// Row-wise 1D quantisation of a staged tile: thread t owns the two
// 16-column blocks 2 (t % 8) and 2 (t % 8) + 1 of rows t / 8 + 16 i
// (i = 0..3); 8 threads write 128 contiguous code bytes of a row.  Row and
// pair indices advance by 16 rows per step, so a step costs no divisions.
template <bool kSR>
__device__ __forceinline__ uint2 rows_block(const QuantParams& p, const float* enc_tab, const uint4& a,
                                            const uint4& b, float den, uint64_t q0, uint32_t& sc) {
  float v[16];
  unpack16(a, b, v);
  sc = block_scale_code(absmax16(v), den);
  const float enc = enc_tab[sc];
  return kSR ? encode16_sr(v, enc, pair_key(p, q0), q0) : encode16_rne(v, enc);
}

template <bool kSR, bool kMMA>
__device__ __forceinline__ void rows_tile(const QuantParams& p, const float* enc_tab,
                                          const uint32_t (&tile)[kColTileRows][kColTileCols / 2],
                                          int64_t r0, int64_t c0, float den) {
  const int tid = threadIdx.x;
  const int bp = tid & 7;                 // block pair within the tile row
  const int64_t col = c0 + 32 * bp;       // first column of the pair
  if (col >= p.cols) return;              // cols % 16 == 0: blocks are wholly in or out
  const bool two = col + 16 < p.cols;     // the pair's second block exists
  // 16-byte code stores and 16-bit scale stores when every pair is whole and aligned
  const bool whole = (p.cols % 32) == 0 && ((reinterpret_cast<uintptr_t>(p.codes) & 15u) == 0) &&
                     ((reinterpret_cast<uintptr_t>(p.scales) & 1u) == 0);
  const int64_t nb = p.cols / 16, kb = col / 16;
  const int rl0 = tid >> 3;
  int64_t r = r0 + rl0;
  uint64_t q0 = ((uint64_t)r * (uint64_t)p.cols + (uint64_t)col) >> 1;  // pair index of element (r, col)
  uint8_t* codes = p.codes + r * (p.cols / 2) + col / 2;
  const uint64_t q_step = (uint64_t)p.cols * 8u;       // 16 rows of pairs
  const int64_t c_step = p.cols * 8;                    // 16 rows of code bytes
#pragma unroll 1
  for (int i = 0; i < kColTileRows / 16; ++i, r += 16, q0 += q_step, codes += c_step) {
    if (r >= p.rows) break;
    const int rl = rl0 + 16 * i;
    const uint4 a0 = *reinterpret_cast<const uint4*>(&tile[rl][16 * bp]);
    const uint4 a1 = *reinterpret_cast<const uint4*>(&tile[rl][16 * bp + 4]);
    const uint4 b0 = *reinterpret_cast<const uint4*>(&tile[rl][16 * bp + 8]);
    const uint4 b1 = *reinterpret_cast<const uint4*>(&tile[rl][16 * bp + 12]);
    uint32_t sc0, sc1 = 0u;
    const uint2 qa = rows_block<kSR>(p, enc_tab, a0, a1, den, q0, sc0);
    uint2 qb = make_uint2(0u, 0u);
    if (two) qb = rows_block<kSR>(p, enc_tab, b0, b1, den, q0 + 8u, sc1);
    const int64_t so = kMMA ? mma_scale_offset(r, kb, nb / 4) : r * nb + kb;
    if (whole) {
      *reinterpret_cast<uint4*>(codes) = make_uint4(qa.x, qa.y, qb.x, qb.y);
      *reinterpret_cast<uint16_t*>(p.scales + so) = (uint16_t)(sc0 | (sc1 << 8));
    } else {
      *reinterpret_cast<uint2*>(codes) = qa;
      p.scales[so] = (uint8_t)sc0;
      if (two) {
        *reinterpret_cast<uint2*>(codes + 8) = qb;
        p.scales[kMMA ? mma_scale_offset(r, kb + 1, nb / 4) : so + 1] = (uint8_t)sc1;
      }
    }
  }
}

// Row-wise 2D (16x16 tile) quantisation of a staged tile: threads 2u and
// 2u + 1 own the 16x16 tile u (tile row u / 16, tile column u % 16), eight
// rows each; the integer tile amax (exact for bf16) is combined with one
// shuffle, then each row is re-read from shared memory and encoded, and the
// tile's scale is written on each of its 16 rows.  16 threads write 128
// contiguous code bytes of a row.
template <bool kSR, bool kMMA>
__device__ __forceinline__ void rows2d_tile(const QuantParams& p, const float* enc_tab,
                                            const uint32_t (&tile)[kColTileRows][kColTileCols / 2], int64_t r0,
                                            int64_t c0, float den) {
  const int tid = threadIdx.x;
  const int h = tid & 1, tcol = (tid >> 1) & 15, trow = tid >> 5;
  const int64_t col = c0 + 16 * tcol;
  const int lr0 = 16 * trow + 8 * h;  // first of this thread's 8 rows in the tile
  uint32_t m = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 a = *reinterpret_cast<const uint4*>(&tile[lr0 + i][8 * tcol]);
    const uint4 b = *reinterpret_cast<const uint4*>(&tile[lr0 + i][8 * tcol + 4]);
    m = absmax_pairs(absmax_pairs(m, a), b);
  }
  m = pairs_to_f32_bits(m);
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  if (col >= p.cols || r0 + 16 * trow >= p.rows) return;  // whole 16x16 tiles only (rows, cols % 16 == 0)
  const uint32_t sc = block_scale_code(__uint_as_float(m), den);
  const float enc = enc_tab[sc];
  const int64_t nb = p.cols / 16, kb = col / 16;
#pragma unroll 2
  for (int i = 0; i < 8; ++i) {
    const int64_t r = r0 + lr0 + i;
    const uint4 a = *reinterpret_cast<const uint4*>(&tile[lr0 + i][8 * tcol]);
    const uint4 b = *reinterpret_cast<const uint4*>(&tile[lr0 + i][8 * tcol + 4]);
    float v[16];
    unpack16(a, b, v);
    uint2 q;
    if (kSR) {
      const uint64_t q0 = ((uint64_t)r * (uint64_t)p.cols + (uint64_t)col) >> 1;
      q = encode16_sr(v, enc, pair_key(p, q0), q0);
    } else {
      q = encode16_rne(v, enc);
    }
    *reinterpret_cast<uint2*>(p.codes + r * (p.cols / 2) + col / 2) = q;
    p.scales[kMMA ? mma_scale_offset(r, kb, nb / 4) : r * nb + kb] = (uint8_t)sc;
  }
}

template <bool kSR, bool kMMA>
__global__ void __launch_bounds__(kColThreads) quant_rows_2d_kernel(const __grid_constant__ CUtensorMap map,
                                                                   QuantParams p) {
  __shared__ TileSmem ts;
  __shared__ float enc_tab[128];
  float amax;
  const float sg = tensor_scale(p, amax);
  const float den = __fmul_rn(sg, 6.0f);
  fill_enc_table(enc_tab, sg);
  tile_smem_init(ts);
  __syncthreads();
  for_each_tile<true>(map, ts, p.rows, p.cols, p.status, [&](int64_t r0, int64_t c0) {
    rows2d_tile<kSR, kMMA>(p, enc_tab, ts.tile, r0, c0, den);
  });
}

// Row-wise 1D quantisation through staged tiles (no transform): the tile's
// copies are asynchronous, so a CTA keeps a whole 32 KiB tile in flight
// without holding registers, and six CTAs per SM cover DRAM latency.
template <bool kSR, bool kMMA>
__global__ void __launch_bounds__(kColThreads, 6) quant_rows_tile_kernel(const __grid_constant__ CUtensorMap map,
                                                                         QuantParams p) {
  __shared__ TileSmem ts;
  __shared__ float enc_tab[128];
  float amax;
  const float sg = tensor_scale(p, amax);
  const float den = __fmul_rn(sg, 6.0f);
  fill_enc_table(enc_tab, sg);
  tile_smem_init(ts);
  __syncthreads();
  for_each_tile<true>(map, ts, p.rows, p.cols, p.status, [&](int64_t r0, int64_t c0) {
    rows_tile<kSR, kMMA>(p, enc_tab, ts.tile, r0, c0, den);
  });
}

// Dual-orientation quantisation: one read of each input tile produces the
// row-wise 1D operand (pr: RNE or SR) and the transposed RHT + SR operand
// (pc).  Results are bit-identical to the two separate kernels.
// Six CTAs per SM (80 registers, 6 x 32 KiB tiles): the encodes are bound
// by instruction issue, and more resident warps hide their latencies.
template <bool kRowSR, bool kMMA>
__global__ void __launch_bounds__(kColThreads, 6) quant_dual_kernel(const __grid_constant__ CUtensorMap map,
                                                                    QuantParams pr, QuantParams pc) {
  __shared__ TileSmem ts;
  __shared__ float enc_r[128], enc_c[128];
  float amax_r, amax_c;
  const float sg_r = tensor_scale(pr, amax_r);
  const float sg_c = tensor_scale(pc, amax_c);
  const float den_r = __fmul_rn(sg_r, 6.0f), den_c = __fmul_rn(sg_c, 6.0f);
  fill_enc_table(enc_r, sg_r);
  fill_enc_table(enc_c, sg_c);
  tile_smem_init(ts);
  __syncthreads();
  for_each_tile<true>(map, ts, pr.rows, pr.cols, pr.status, [&](int64_t r0, int64_t c0) {
    rows_tile<kRowSR, kMMA>(pr, enc_r, ts.tile, r0, c0, den_r);
    cols_tile<true, true, false, kMMA>(pc, enc_c, ts.tile, r0, c0, den_c);
  });
}

// ------------------------------------------------------------- launch --
// CTAs that fit on the device at once for `kernel` (cached per kernel and
// device).  Grid-stride kernels are launched with at most this many CTAs, so
// every CTA is resident from the start and no partial second wave trails.
static int64_t resident_ctas(const void* kernel, int threads, const DeviceInfo& dev) {
  static std::mutex mu;
  static std::unordered_map<const void*, int> per_sm[64];
  std::lock_guard<std::mutex> lock(mu);
  auto& m = per_sm[dev.device & 63];
  auto it = m.find(kernel);
  if (it == m.end()) {
    int n = 0;
    // Kernels that stage tiles in shared memory ask for the largest carveout
    // so shared memory does not cap the CTAs per SM below the register limit.
    // Both calls are hints: a failure falls back to one CTA per SM and its
    // error is cleared, so the launch check that follows does not see it.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
    if (e == cudaSuccess && fa.sharedSizeBytes > 1024)
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) (void)cudaGetLastError();
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1) {
      (void)cudaGetLastError();
      n = 1;
    }
    it = m.emplace(kernel, n).first;
  }
  return (int64_t)it->second * dev.sm_count;
}

template <typename Kernel>
static int grid_for(Kernel kernel, const DeviceInfo& dev, int64_t work_items, int threads) {
  const int64_t need = (work_items + threads - 1) / threads;
  const int64_t cap = resident_ctas(reinterpret_cast<const void*>(kernel), threads, dev);
  return (int)(need < 1 ? 1 : (need < cap ? need : cap));
}

static int64_t tile_count(int64_t rows, int64_t cols) {
  return ((rows + kColTileRows - 1) / kColTileRows) * ((cols + kColTileCols - 1) / kColTileCols);
}

// TMA map of the input as 64 x 256 tiles.
static bool input_map(CUtensorMap* m, const void* x, int64_t rows, int64_t cols, int64_t ld) {
  return make_bf16_tile_map(m, x, rows, cols, ld, kColTileCols, kColTileRows);
}

// Tile-staged amax pass: the plain amax into out_plain and/or the amax after
// the column-wise transform into out_cols (null: not computed).
static void launch_amax_tiles(const DeviceInfo& dev, const CUtensorMap& map, int64_t rows, int64_t cols,
                              uint32_t signs, float* out_plain, float* out_cols, cudaStream_t s) {
  const int64_t work = tile_count(rows, cols) * kColThreads;
  if (out_plain && out_cols) {
    auto k = amax_tile_kernel<true, true>;
    k<<<grid_for(k, dev, work, kColThreads), kColThreads, 0, s>>>(map, rows, cols, signs, out_plain, out_cols,
                                                                   dev.status);
  } else if (out_cols) {
    auto k = amax_tile_kernel<false, true>;
    k<<<grid_for(k, dev, work, kColThreads), kColThreads, 0, s>>>(map, rows, cols, signs, nullptr, out_cols,
                                                                   dev.status);
  } else if (out_plain) {
    auto k = amax_tile_kernel<true, false>;
    k<<<grid_for(k, dev, work, kColThreads), kColThreads, 0, s>>>(map, rows, cols, signs, out_plain, nullptr,
                                                                   dev.status);
  }
}

template <bool kSR, bool kRHT>
static void launch_rows_1d(const DeviceInfo& dev, const CUtensorMap& map, const QuantParams& p, bool mma,
                           cudaStream_t s) {
  // Round-to-nearest rows go through staged tiles (HBM-bound: the TMA keeps
  // a whole tile in flight per CTA); stochastic rounding and the row-wise
  // transform keep the register-resident kernel, which measured faster for
  // those instruction-bound modes.
  if constexpr (!kRHT && !kSR) {
    const int64_t tiles = tile_count(p.rows, p.cols);
    if (mma) {
      auto k = quant_rows_tile_kernel<kSR, true>;
      k<<<grid_for(k, dev, tiles * kColThreads, kColThreads), kColThreads, 0, s>>>(map, p);
    } else {
      auto k = quant_rows_tile_kernel<kSR, false>;
      k<<<grid_for(k, dev, tiles * kColThreads, kColThreads), kColThreads, 0, s>>>(map, p);
    }
    return;
  }
  const int64_t items = p.orows * (p.ocols / 16) / 2;  // two blocks per thread
  if (mma) {
    auto k = quant_rows_1d_kernel<kSR, kRHT, true>;
    k<<<grid_for(k, dev, items, 256), 256, 0, s>>>(p);
  } else {
    auto k = quant_rows_1d_kernel<kSR, kRHT, false>;
    k<<<grid_for(k, dev, items, 256), 256, 0, s>>>(p);
  }
}

template <bool kSR>
static void launch_rows_2d(const DeviceInfo& dev, const CUtensorMap& map, const QuantParams& p, bool mma,
                           cudaStream_t s) {
  const int64_t tiles = tile_count(p.rows, p.cols);
  if (mma) {
    auto k = quant_rows_2d_kernel<kSR, true>;
    k<<<grid_for(k, dev, tiles * kColThreads, kColThreads), kColThreads, 0, s>>>(map, p);
  } else {
    auto k = quant_rows_2d_kernel<kSR, false>;
    k<<<grid_for(k, dev, tiles * kColThreads, kColThreads), kColThreads, 0, s>>>(map, p);
  }
}

template <bool kSR, bool kRHT, bool kTwoD>
static void launch_cols(const DeviceInfo& dev, const CUtensorMap& map, const QuantParams& p, bool mma,
                        cudaStream_t s) {
  const int64_t tiles = tile_count(p.rows, p.cols);
  if (mma) {
    auto k = quant_cols_kernel<kSR, kRHT, kTwoD, true>;
    k<<<grid_for(k, dev, tiles * kColThreads, kColThreads), kColThreads, 0, s>>>(map, p);
  } else {
    auto k = quant_cols_kernel<kSR, kRHT, kTwoD, false>;
    k<<<grid_for(k, dev, tiles * kColThreads, kColThreads), kColThreads, 0, s>>>(map, p);
  }
}

static void set_sr_keys(QuantParams& p, uint64_t sr_seed) {
  const uint32_t key = stream_key(sr_seed, kTagSR);
  p.sr_hk[0] = mix32(key);
  p.sr_hk[1] = mix32(key ^ 1u);
}

int quantize_launch(const DeviceInfo& dev, const void* x, int64_t rows, int64_t cols, int64_t ld,
                    uint32_t flags, bool rht, uint64_t rht_seed, uint64_t sr_seed, const float* amax_in,
                    const nvfp4_tensor& out, cudaStream_t stream) {
  const bool two_d = (flags & NVFP4_BLOCK_2D) != 0;
  const bool sr = rht || (flags & NVFP4_ROUND_SR) != 0;
  const bool tr = (flags & NVFP4_TRANSPOSE_OUT) != 0;
  const bool mma = out.scale_layout == NVFP4_SCALES_MMA;
  const uint32_t signs = rht_sign_bits(rht_seed);

  QuantParams p;
  p.x = static_cast<const uint16_t*>(x);
  p.rows = rows;
  p.cols = cols;
  p.ld = ld;
  p.orows = out.rows;
  p.ocols = out.cols;
  p.codes = out.codes;
  p.scales = out.scales;
  p.sg_out = out.global_scale;
  p.status = dev.status;
  set_sr_keys(p, sr_seed);
  p.rht_signs = signs;

  // Padding rows of the MMA scale layout read as zero.
  if (mma && (p.orows % 128) != 0) {
    const int64_t band = (p.ocols / 64) * 512;
    if (cudaMemsetAsync(out.scales + (p.orows / 128) * band, 0, band, stream) != cudaSuccess)
      return NVFP4_ERR_CUDA;
  }

  CUtensorMap map;
  if (!input_map(&map, x, rows, cols, ld)) return NVFP4_ERR_CUDA;

  // Pass 1: tensor amax (unless supplied).
  if (amax_in) {
    p.amax_src = amax_in;
    p.amax_out = out.amax;
  } else {
    p.amax_src = out.amax;
    p.amax_out = nullptr;
    if (cudaMemsetAsync(out.amax, 0, sizeof(float), stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (!rht) {
      const int64_t vpr = cols / 8;
      amax_plain_kernel<<<grid_for(amax_plain_kernel, dev, rows * vpr, 256), 256, 0, stream>>>(
          reinterpret_cast<const uint4*>(x), rows, vpr, ld / 8, out.amax);
    } else if (tr) {
      launch_amax_tiles(dev, map, rows, cols, signs, nullptr, out.amax, stream);
    } else {
      amax_rht_rows_kernel<<<grid_for(amax_rht_rows_kernel, dev, rows * (cols / 16), 256), 256, 0, stream>>>(
          p.x, rows, cols, ld, signs, out.amax);
    }
  }

  // Pass 2: scales and codes.
  if (!tr) {
    if (two_d) {
      if (sr) launch_rows_2d<true>(dev, map, p, mma, stream);
      else launch_rows_2d<false>(dev, map, p, mma, stream);
    } else {
      if (sr && rht) launch_rows_1d<true, true>(dev, map, p, mma, stream);
      else if (sr) launch_rows_1d<true, false>(dev, map, p, mma, stream);
      else if (rht) launch_rows_1d<false, true>(dev, map, p, mma, stream);
      else launch_rows_1d<false, false>(dev, map, p, mma, stream);
    }
  } else {
    if (two_d) {
      if (sr) launch_cols<true, false, true>(dev, map, p, mma, stream);
      else launch_cols<false, false, true>(dev, map, p, mma, stream);
    } else if (rht) {
      launch_cols<true, true, false>(dev, map, p, mma, stream);
    } else if (sr) {
      launch_cols<true, false, false>(dev, map, p, mma, stream);
    } else {
      launch_cols<false, false, false>(dev, map, p, mma, stream);
    }
  }
  return cudaPeekAtLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// ---------------------------------------------------------------- MXFP4 --
// The power-of-two-scaled open format NVFP4 is compared with: 32-element row
// blocks, scale 2^e with e = floor(log2(amax_b)) - 2 (clamped to
// [-127, 127]; -127 for zero and subnormal block maxima) stored as the E8M0
// byte e + 127, elements E2M1 round-to-nearest-even of x * 2^-e (exact),
// saturating at 6.  One thread per block (four 16-byte loads).
__global__ void __launch_bounds__(256) quant_mx_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                                                       int64_t ld, uint8_t* __restrict__ codes,
                                                       uint8_t* __restrict__ scales) {
  const uint32_t nb = (uint32_t)(cols / 32);
  const uint32_t total = (uint32_t)(rows * nb);
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const uint32_t r = i / nb, b = i - r * nb;
    const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)r * ld + (int64_t)b * 32);
    const uint4 u0 = ldg_nc(src), u1 = ldg_nc(src + 1), u2 = ldg_nc(src + 2), u3 = ldg_nc(src + 3);
    const uint32_t mbits = pairs_to_f32_bits(absmax_pairs(absmax_pairs(absmax_pairs(absmax_pairs(0u, u0), u1), u2), u3));
    const int ef = (int)((mbits >> 23) & 0xFFu);
    const int e = (ef == 0) ? -127 : min(ef - 127 - 2, 127);
    const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e, a normal float for e in [-127, 125]
    float v0[16], v1[16];
    unpack16(u0, u1, v0);
    unpack16(u2, u3, v1);
    const uint2 q0 = encode16_rne(v0, inv), q1 = encode16_rne(v1, inv);
    *reinterpret_cast<uint4*>(codes + (int64_t)r * (cols / 2) + (int64_t)b * 16) = make_uint4(q0.x, q0.y, q1.x, q1.y);
    scales[(int64_t)r * nb + b] = (uint8_t)(e + 127);
  }
}

int quantize_mx_launch(const DeviceInfo& dev, const void* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* codes,
                       uint8_t* scales, cudaStream_t stream) {
  quant_mx_kernel<<<grid_for(quant_mx_kernel, dev, rows * (cols / 32), 256), 256, 0, stream>>>(
      static_cast<const uint16_t*>(x), rows, cols, ld, codes, scales);
  return cudaPeekAtLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// Dual-orientation quantisation (row-wise 1D + transposed RHT/SR).
int quantize_dual_launch(const DeviceInfo& dev, const void* x, int64_t rows, int64_t cols, int64_t ld,
                         bool row_sr, uint64_t row_sr_seed, uint64_t rht_seed, uint64_t col_sr_seed,
                         const float* amax_row_in, const float* amax_col_in, const nvfp4_tensor& out_row,
                         const nvfp4_tensor& out_col, cudaStream_t stream) {
  const uint32_t signs = rht_sign_bits(rht_seed);
  QuantParams pr, pc;
  for (QuantParams* q : {&pr, &pc}) {
    q->x = static_cast<const uint16_t*>(x);
    q->rows = rows;
    q->cols = cols;
    q->ld = ld;
    q->status = dev.status;
    q->rht_signs = signs;
  }
  pr.orows = out_row.rows; pr.ocols = out_row.cols; pr.codes = out_row.codes; pr.scales = out_row.scales;
  pr.sg_out = out_row.global_scale;
  set_sr_keys(pr, row_sr_seed);
  pc.orows = out_col.rows; pc.ocols = out_col.cols; pc.codes = out_col.codes; pc.scales = out_col.scales;
  pc.sg_out = out_col.global_scale;
  set_sr_keys(pc, col_sr_seed);
  const bool mma = out_row.scale_layout == NVFP4_SCALES_MMA;  // the caller checks both layouts agree

  for (const nvfp4_tensor* o : {&out_row, &out_col}) {
    if (o->scale_layout == NVFP4_SCALES_MMA && (o->rows % 128) != 0) {
      const int64_t band = (o->cols / 64) * 512;
      if (cudaMemsetAsync(o->scales + (o->rows / 128) * band, 0, band, stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    }
  }
  CUtensorMap map;
  if (!input_map(&map, x, rows, cols, ld)) return NVFP4_ERR_CUDA;
  // Pass 1: the amaxes that were not supplied, from one read.  A supplied
  // amax is never written here, so it may alias its operand's own amax.
  if (!amax_row_in && cudaMemsetAsync(out_row.amax, 0, sizeof(float), stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (!amax_col_in && cudaMemsetAsync(out_col.amax, 0, sizeof(float), stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (!amax_row_in && !amax_col_in) {
    launch_amax_tiles(dev, map, rows, cols, signs, out_row.amax, out_col.amax, stream);
  } else if (!amax_row_in) {
    const int64_t vpr = cols / 8;
    amax_plain_kernel<<<grid_for(amax_plain_kernel, dev, rows * vpr, 256), 256, 0, stream>>>(
        reinterpret_cast<const uint4*>(x), rows, vpr, ld / 8, out_row.amax);
  } else if (!amax_col_in) {
    launch_amax_tiles(dev, map, rows, cols, signs, nullptr, out_col.amax, stream);
  }
  pr.amax_src = amax_row_in ? amax_row_in : out_row.amax;
  pr.amax_out = amax_row_in ? out_row.amax : nullptr;
  pc.amax_src = amax_col_in ? amax_col_in : out_col.amax;
  pc.amax_out = amax_col_in ? out_col.amax : nullptr;

  // Pass 2: one read, both outputs.
  const int64_t tiles = tile_count(rows, cols);
  if (row_sr) {
    if (mma) {
      auto k = quant_dual_kernel<true, true>;
      k<<<grid_for(k, dev, tiles * kColThreads, kColThreads), kColThreads, 0, stream>>>(map, pr, pc);
    } else {
      auto k = quant_dual_kernel<true, false>;
      k<<<grid_for(k, dev, tiles * kColThreads, kColThreads), kColThreads, 0, stream>>>(map, pr, pc);
    }
  } else {
    if (mma) {
      auto k = quant_dual_kernel<false, true>;
      k<<<grid_for(k, dev, tiles * kColThreads, kColThreads), kColThreads, 0, stream>>>(map, pr, pc);
    } else {
      auto k = quant_dual_kernel<false, false>;
      k<<<grid_for(k, dev, tiles * kColThreads, kColThreads), kColThreads, 0, stream>>>(map, pr, pc);
    }
  }
  return cudaPeekAtLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// ----------------------------------------------------- codec diagnostics --
// The element encoders exactly as the quantisers run them, through both
// lanes of a pair (even element: low nibble; odd element: high nibble); a
// disagreement between the lanes is reported as 0xFF, which is never a code.
__global__ void encode_e2m1_rne_kernel(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float a = v[i];
    const uint32_t lo = e2m1x2_rne(a, 0.0f) & 0xFu, hi = e2m1x2_rne(0.0f, a) >> 4;
    out[i] = (uint8_t)(lo == hi ? lo : 0xFFu);
  }
}

__global__ void encode_e2m1_sr_kernel(const float* v, const uint16_t* u, int64_t n, uint8_t* out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float a = v[i];
    const uint32_t r = (uint32_t)u[i];
    const uint32_t lo = (sr_pair_b3(a, 0.0f, r) >> 24) & 0xFu, hi = sr_pair_b3(0.0f, a, r << 16) >> 28;
    out[i] = (uint8_t)(lo == hi ? lo : 0xFFu);
  }
}

__global__ void encode_e4m3_kernel(const float* t, int64_t n, uint8_t* out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float a = t[i];
    out[i] = (uint8_t)((a != a) ? 0u : e4m3_encode(a));
  }
}

// Self-test of the bounded waits: one warp waits, with both helpers the
// kernels use (the C++ spin and the single-asm-block spin), on an mbarrier
// that nothing arrives on; each gives up after limit_ns, raising the
// timeout bit, and the kernel returns.
__global__ void selftest_wait_kernel(uint64_t limit_ns, uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&bar), 0, status, limit_ns);
  __syncwarp();
  (void)mbar_wait_spin(smem_u32(&bar), 0, status, limit_ns);
}

int selftest_wait_launch(const DeviceInfo& dev, uint64_t limit_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, dev.status);
  return cudaPeekAtLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

static int diag_grid(int64_t n) {
  const int64_t g = (n + 255) / 256;
  return (int)(g < 1 ? 1 : (g > 65536 ? 65536 : g));
}

int encode_e2m1_rne_launch(const float* v, int64_t n, uint8_t* out, cudaStream_t stream) {
  encode_e2m1_rne_kernel<<<diag_grid(n), 256, 0, stream>>>(v, n, out);
  return cudaPeekAtLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

int encode_e2m1_sr_launch(const float* v, const uint16_t* u, int64_t n, uint8_t* out, cudaStream_t stream) {
  encode_e2m1_sr_kernel<<<diag_grid(n), 256, 0, stream>>>(v, u, n, out);
  return cudaPeekAtLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

int encode_e4m3_launch(const float* t, int64_t n, uint8_t* out, cudaStream_t stream) {
  encode_e4m3_kernel<<<diag_grid(n), 256, 0, stream>>>(t, n, out);
  return cudaPeekAtLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace nvfp4
