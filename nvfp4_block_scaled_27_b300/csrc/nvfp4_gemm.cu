// nvfp4_gemm.cu -- block-scaled NVFP4 GEMM on the sm_103a tensor cores.
//
// C[M, N] = s_gA * s_gB * A[M, K] * B[N, K]^T, BF16 out.  The operands are
// NVFP4 (E2M1 codes, one E4M3 scale per 16 elements along K): "NVFP4: cos'è e
// come supera FP8 e BF16 nell'intelligenza artificiale", sections "Cos'è
// NVFP4 ..." (format) and "Blackwell Architecture: la potenza dietro NVFP4"
// (fifth-generation tensor cores scale NVFP4 blocks in hardware and keep
// results in tensor memory next to the units).  All three MLP GEMMs of the
// training recipe (fprop, dgrad, wgrad) take NVFP4 operands and return BF16:
// readjensen.com NVFP4 training-recipe article, MLP data-flow paragraph.
//
// Design (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0      TMA producer: per 256-wide K step, the A tile (128 rows x
//               128 B) and B tile (256 rows x 128 B) with 128-byte swizzle,
//               plus the matching scale atoms (contiguous 512-byte blocks in
//               the MMA scale layout) by bulk copy; 4-stage mbarrier ring.
//   warp 1      MMA issuer: four tcgen05.mma kind::mxf4nvf4
//               block_scale.scale_vec::4X (M=128, N=256, K=64) per stage into
//               a 128 x 256 fp32 accumulator in tensor memory; tcgen05.commit
//               frees the stage and, after the last K step, hands the tile to
//               the epilogue.
//   warps 2-5   scale writers, one per 32-lane tensor-memory quadrant: each
//               lane reads its 16-byte rows of the stage's scale atoms from
//               shared memory and writes them with tcgen05.st into that
//               stage's scale columns (each quadrant holds the full
//               128-row / 256-column scale set the MMA reads).  Moving scales
//               this way keeps them off the MMA's in-order pipe; copying them
//               with tcgen05.cp (12 copies per stage) stretched every MMA by
//               about half.
//   warps 6-13  epilogue: two warps per lane quadrant each pull 128 fp32
//               columns out of tensor memory, scale by s_gA * s_gB and round
//               to packed BF16 in registers, release the accumulator (the
//               next tile's MMAs start) and only then store.
// Tensor memory: 512 columns = accumulator [0, 256) + per-stage scale
// columns (SFA 4 x 4, SFB 4 x 8 per stage).  Every mbarrier wait is bounded
// (2 s); on expiry the kernel raises the timeout bit and winds down.
#include <cuda_bf16.h>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

#include <mutex>

namespace nvfp4 {
namespace gemm {

constexpr int BM = 128;            // tile rows (A rows)
constexpr int BN = 256;            // tile cols (B rows)
constexpr int BK = 256;            // K elements per stage
constexpr int BKB = BK / 2;        // bytes per row per stage (128: one swizzle row)
constexpr int MMA_K = 64;          // K per tcgen05.mma for kind::mxf4nvf4
constexpr int KSTEPS = BK / MMA_K; // 4 MMAs per stage
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BKB;                     // 16 KiB
constexpr int B_BYTES = BN * BKB;                     // 32 KiB
constexpr int SFA_BYTES = (BM / 128) * KSTEPS * 512;  // 2 KiB
constexpr int SFB_BYTES = (BN / 128) * KSTEPS * 512;  // 4 KiB
constexpr int STAGE_TX = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr int NUM_THREADS = 448;
constexpr int NUM_SF_WARPS = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr int FIRST_SF_WARP = 2;
constexpr int FIRST_EPI_WARP = FIRST_SF_WARP + NUM_SF_WARPS;
constexpr int TMEM_COLS = 512;
constexpr int SF_COLS_PER_STAGE = KSTEPS * 4 + KSTEPS * 8;  // 48

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
constexpr int NUM_BARS = 3 * STAGES + 2;
constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
constexpr int SMEM_USED = OFF_ABORT + 4;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(256 + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "tensor memory budget");

// Instruction descriptor for kind::mxf4nvf4 (dense, K-major A and B, E2M1
// operands, UE4M3 scales, scale-factor ids 0):
//   [7,10) A format = E2M1 (1), [10,13) B format = E2M1 (1),
//   [17,23) N >> 3, [23] scale type UE4M3 = 0, [24,29) M >> 4.
constexpr uint32_t make_idesc(int m, int n) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
constexpr uint32_t IDESC = make_idesc(BM, BN);

// Shared-memory matrix descriptor: start address, leading/stride byte
// offsets (in 16-byte units), descriptor version 1 (bit 46), swizzle mode in
// bits [61,64) (2 = 128-byte swizzle, 0 = none).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swz << 61);
}

// Two accumulator values scaled by alpha and rounded to BF16 (nearest even),
// packed with `lo` in the low half-word.  The product is rounded to fp32
// first; the result differs from rounding the exact product only when that
// fp32 value sits exactly on a BF16 tie.
__device__ __forceinline__ uint32_t scale_pack_bf16x2(float lo, float hi, float alpha) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(lo, alpha), __fmul_rn(hi, alpha));
  return *reinterpret_cast<const uint32_t*>(&h);
}

struct Params {
  const uint8_t* sfa;  // A scales, MMA layout
  const uint8_t* sfb;  // B scales, MMA layout
  const float* sga;
  const float* sgb;
  uint16_t* c;  // bf16 output
  int64_t ldc;
  int M, N, K;
  int tiles_m, tiles_n, num_tiles;
  uint32_t* status;
};

// Tile order: groups of 16 M-tiles, M fastest inside a group, so the tiles
// in flight across the GPU share A and B panels in L2.
__device__ __forceinline__ void tile_coords(const Params& p, int t, int& tm, int& tn) {
  constexpr int G = 16;
  const int group_span = G * p.tiles_n;
  const int g = t / group_span;
  const int first_m = g * G;
  const int gm = min(G, p.tiles_m - first_m);
  const int r = t - g * group_span;
  tm = first_m + r % gm;
  tn = r / gm;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                  const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + OFF_BAR;                // STAGES barriers
  const uint32_t bar_empty = bar_full + STAGES * 8;         // STAGES barriers
  const uint32_t bar_sf = bar_empty + STAGES * 8;           // STAGES barriers
  const uint32_t bar_tmem_full = bar_sf + STAGES * 8;
  const uint32_t bar_tmem_empty = bar_tmem_full + 8;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM_SLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_sf + 8 * s, NUM_SF_WARPS);
    }
    mbar_init(bar_tmem_full, 1);
    mbar_init(bar_tmem_empty, NUM_EPI_WARPS);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmap_a);
    prefetch_tensormap(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(sbase + OFF_TMEM_SLOT, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_kb = p.K / BK;
  const int64_t atoms_per_band = p.K / 64;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      const int bands_b = (p.N + 127) / 128;
      for (int t = blockIdx.x; t < p.num_tiles && !*abort_flag; t += gridDim.x) {
        int tm, tn;
        tile_coords(p, t, tm, tn);
        const bool second_band = (2 * tn + 1) < bands_b;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, p.status)) { *abort_flag = 1; break; }
          const uint32_t full = bar_full + 8 * stage;
          const uint32_t tx = STAGE_TX - (second_band ? 0 : SFB_BYTES / 2);
          mbar_arrive_expect_tx(full, tx);
          tma_load_2d(sbase + OFF_A + stage * A_BYTES, &tmap_a, kb * BKB, tm * BM, full);
          tma_load_2d(sbase + OFF_B + stage * B_BYTES, &tmap_b, kb * BKB, tn * BN, full);
          const uint8_t* sa = p.sfa + ((int64_t)tm * atoms_per_band + (int64_t)kb * KSTEPS) * 512;
          bulk_load(sbase + OFF_SFA + stage * SFA_BYTES, sa, SFA_BYTES, full);
          const uint8_t* sb0 = p.sfb + ((int64_t)(2 * tn) * atoms_per_band + (int64_t)kb * KSTEPS) * 512;
          bulk_load(sbase + OFF_SFB + stage * SFB_BYTES, sb0, SFB_BYTES / 2, full);
          if (second_band)
            bulk_load(sbase + OFF_SFB + stage * SFB_BYTES + SFB_BYTES / 2, sb0 + atoms_per_band * 512,
                      SFB_BYTES / 2, full);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // Let in-flight copies land before the CTA can exit: wait (bounded)
      // for the last loads of every stage to complete.
      for (int s = 0; s < STAGES; ++s) {
        // stages issued in the current lap have parity `phase`, the others
        // belong to the previous lap; waiting on either is bounded.
        const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
        mbar_wait(bar_full + 8 * s, par, p.status, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int t = blockIdx.x; t < p.num_tiles && !*abort_flag; t += gridDim.x, ++it) {
        if (!mbar_wait(bar_tmem_empty, (uint32_t)(it & 1) ^ 1u, p.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(bar_full + 8 * stage, phase, p.status) || !mbar_wait(bar_sf + 8 * stage, phase, p.status)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf_col = tmem_base + 256u + (uint32_t)(stage * SF_COLS_PER_STAGE);
          const uint32_t a_s = sbase + OFF_A + stage * A_BYTES;
          const uint32_t b_s = sbase + OFF_B + stage * B_BYTES;
#pragma unroll
          for (int j = 0; j < KSTEPS; ++j) {
            // K-major, 128-byte swizzle: 8-row groups 1024 B apart; the K
            // offset inside the swizzle row advances the start address.
            const uint64_t ad = smem_desc(a_s + 32 * j, 16, 1024, 2);
            const uint64_t bd = smem_desc(b_s + 32 * j, 16, 1024, 2);
            tc_mma_nvf4(tmem_base, ad, bd, IDESC, sf_col + 4 * j, sf_col + 16 + 8 * j,
                        (kb > 0 || j > 0) ? 1u : 0u);
          }
          tc_commit(bar_empty + 8 * stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(bar_tmem_full);
      }
    }
  } else if (warp < FIRST_EPI_WARP) {
    // ---------------------------------------------------- scale writers --
    // Quadrant q (= warp % 4) lanes 32q + r.  Scale atom row r holds the four
    // 32-bit scale words of rows r, 32 + r, 64 + r, 96 + r (one per column),
    // which is exactly what tensor-memory lane 32q + r needs in the four
    // columns of a 128-row group.
    const int quad = warp & 3;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    int stage = 0;
    uint32_t phase = 0;
    for (int t = blockIdx.x; t < p.num_tiles && !*abort_flag; t += gridDim.x) {
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!mbar_wait(bar_full + 8 * stage, phase, p.status)) { *abort_flag = 1; ok = false; break; }
        const uint8_t* sfa_s = smem + OFF_SFA + stage * SFA_BYTES + lane * 16;
        const uint8_t* sfb_s = smem + OFF_SFB + stage * SFB_BYTES + lane * 16;
        uint32_t va[16], vb[32];
#pragma unroll
        for (int j = 0; j < KSTEPS; ++j) {
          const uint4 a = *reinterpret_cast<const uint4*>(sfa_s + 512 * j);
          const uint4 b0 = *reinterpret_cast<const uint4*>(sfb_s + 512 * j);
          const uint4 b1 = *reinterpret_cast<const uint4*>(sfb_s + SFB_BYTES / 2 + 512 * j);
          va[4 * j + 0] = a.x; va[4 * j + 1] = a.y; va[4 * j + 2] = a.z; va[4 * j + 3] = a.w;
          vb[8 * j + 0] = b0.x; vb[8 * j + 1] = b0.y; vb[8 * j + 2] = b0.z; vb[8 * j + 3] = b0.w;
          vb[8 * j + 4] = b1.x; vb[8 * j + 5] = b1.y; vb[8 * j + 6] = b1.z; vb[8 * j + 7] = b1.w;
        }
        const uint32_t col = tmem_base + lane_off + 256u + (uint32_t)(stage * SF_COLS_PER_STAGE);
        tmem_st_32x32b_x16(col, va);
        tmem_st_32x32b_x16(col + 16, vb);
        tmem_st_32x32b_x16(col + 32, vb + 16);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sf + 8 * stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
    }
  } else {
    // --------------------------------------------------------- epilogue --
    const int quad = warp & 3;                     // lane quadrant this warp may access
    const int half = (warp - FIRST_EPI_WARP) >> 2;  // which 128 accumulator columns
    const float alpha = __fmul_rn(*p.sga, *p.sgb);
    int it = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++it) {
      if (!mbar_wait(bar_tmem_full, (uint32_t)(it & 1), p.status)) { *abort_flag = 1; break; }
      if (*abort_flag) break;
      tc_fence_after();
      int tm, tn;
      tile_coords(p, t, tm, tn);
      const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(half * 128);
      const int row = tm * BM + quad * 32 + lane;
      const int col0 = tn * BN + half * 128;
      uint16_t* out = p.c + (int64_t)row * p.ldc + col0;
      if (col0 + 128 <= p.N) {
        // Pull this warp's 32 x 128 accumulator block out of tensor memory
        // in 32-column chunks, scaling and rounding each into 16 packed
        // bf16x2 words; release the accumulator as soon as the last chunk is
        // in registers so the next tile's MMAs overlap the stores.
        uint32_t w[64];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(taddr + 32 * ch, v);
          tc_wait_ld();
#pragma unroll
          for (int q = 0; q < 16; ++q)
            w[16 * ch + q] = scale_pack_bf16x2(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]), alpha);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_tmem_empty);
        if (row < p.M) {
#pragma unroll
          for (int g = 0; g < 16; ++g)
            *reinterpret_cast<uint4*>(out + 8 * g) = make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
        }
      } else {
        // Ragged right edge (N not a multiple of the tile): chunk by chunk
        // with per-element bounds, releasing the accumulator at the end.
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(taddr + 32 * ch, v);
          tc_wait_ld();
          if (row < p.M) {
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const int n = col0 + 32 * ch + 2 * q;
              const uint32_t pk =
                  scale_pack_bf16x2(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]), alpha);
              if (n < p.N) out[32 * ch + 2 * q] = (uint16_t)(pk & 0xFFFFu);
              if (n + 1 < p.N) out[32 * ch + 2 * q + 1] = (uint16_t)(pk >> 16);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_tmem_empty);
      }
    }
  }

  // ----------------------------------------------------------- teardown --
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace gemm

// ----------------------------------------------------------------- host --
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Byte-granular 2-D map over packed codes [rows, K/2] with a box of
// (128 bytes, box_rows) and 128-byte swizzle; out-of-range rows read as zero.
static bool make_code_map(CUtensorMap* map, const void* base, int64_t rows, int64_t kbytes, uint32_t box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kbytes, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kbytes};
  const cuuint32_t box[2] = {(cuuint32_t)gemm::BKB, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gemm_launch(const DeviceInfo& dev, const nvfp4_tensor& A, const nvfp4_tensor& B, void* c, int64_t ldc,
                cudaStream_t stream) {
  using namespace gemm;
  static std::mutex mu;
  static bool attr_set[64] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev.device < 0 || dev.device >= 64) return NVFP4_ERR_CUDA;
    if (!attr_set[dev.device]) {
      if (cudaFuncSetAttribute(nvfp4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
          cudaSuccess)
        return NVFP4_ERR_CUDA;
      attr_set[dev.device] = true;
    }
  }
  CUtensorMap ta, tb;
  if (!make_code_map(&ta, A.codes, A.rows, A.cols / 2, BM)) return NVFP4_ERR_CUDA;
  if (!make_code_map(&tb, B.codes, B.rows, B.cols / 2, BN)) return NVFP4_ERR_CUDA;
  Params p;
  p.sfa = A.scales;
  p.sfb = B.scales;
  p.sga = A.global_scale;
  p.sgb = B.global_scale;
  p.c = static_cast<uint16_t*>(c);
  p.ldc = ldc;
  p.M = (int)A.rows;
  p.N = (int)B.rows;
  p.K = (int)A.cols;
  p.tiles_m = (p.M + BM - 1) / BM;
  p.tiles_n = (p.N + BN - 1) / BN;
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.status = dev.status;
  const int grid = p.num_tiles < dev.sm_count ? p.num_tiles : dev.sm_count;
  nvfp4_gemm_kernel<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(ta, tb, p);
  return cudaPeekAtLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace nvfp4
