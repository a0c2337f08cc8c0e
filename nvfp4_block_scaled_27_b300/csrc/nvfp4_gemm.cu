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
// Design: clusters of two CTAs (one per SM) work as a pair on 256 x 256
// output tiles, persistently.  A launch may hold two independent problems
// (the backward pass's dgrad and wgrad): their tiles form one list, longer
// contraction first, and each warp looks up its tile's problem.  CTA r of
// the pair owns output rows
// [128 r, 128 r + 128) of the tile.  Per 256-wide K step each CTA loads 128
// rows of A and 128 of the 256 rows of B (so each SM streams half the B bytes
// a single-SM 128 x 256 tile would need), its own A scales and all of B's
// scales.  Warp roles, in both CTAs:
//   warp 0      operand producer: A and B boxes (128 rows x 128 B, 128-byte
//               swizzle) into a 5-stage ring; the copies of both CTAs
//               complete on the leader's `full` barrier (CTA-pair TMA form).
//   warp 1      allocates the pair's tensor memory.  In CTA 0 (the leader)
//               the whole warp waits and one elected lane issues
//               tcgen05.mma.cta_group::2 kind::mxf4nvf4 block_scale
//               .scale_vec::4X (M = 256, N = 256, K = 64), four per stage,
//               into a 128 x 256 fp32 accumulator in each CTA's tensor
//               memory; tcgen05.commit multicasts stage release (`empty`)
//               and tile completion (`tmem_full`) to both CTAs.
//   warp 2      scale producer: the stage's scale atoms (A: one bulk copy;
//               B: both bands in one 3-D TMA box) into a ring of its own,
//               refilled as soon as the scale writers have read a slot, so
//               scales are in shared memory well before the stage's
//               operands.
//   warps 3-6   scale writers, one per 32-lane tensor-memory quadrant: once
//               the stage's scale columns are free (its previous MMAs done),
//               copy the scale atoms from shared memory into them with
//               tcgen05.st (each quadrant holds the whole set the MMA reads)
//               and arrive on the leader's `sf_done`.  (tcgen05.cp of the
//               same data stalls the MMA stream.)
//   warps 7-14  epilogue: two warps per lane quadrant each pull 128 fp32
//               columns out of tensor memory in two halves, scale by
//               s_gA * s_gB (packed pairs) and round to packed BF16 in
//               registers; the accumulator is released to the leader as soon
//               as the second half is in registers (the next tile's MMAs
//               start while it is converted), then 32 x 32 BF16 boxes go out
//               through swizzled shared memory with TMA stores.
// The refill of a stage thus waits only on the operand copies; scales are
// written off that path.  Tensor memory (512 columns, same addresses in both
// CTAs): accumulator [0, 256) + per-stage scale columns (SFA 4 x 4, SFB 4 x 8).
// Every mbarrier wait is bounded (2 s); on expiry the kernel raises the
// timeout bit, winds down, and the two CTAs still meet in a bounded exit
// handshake before the tensor memory is freed.
#include <cuda_bf16.h>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

#include <cstring>
#include <mutex>

namespace nvfp4 {
namespace gemm {

constexpr int BM = 128;            // output rows per CTA (A rows)
constexpr int BM_PAIR = 2 * BM;    // output rows per pair tile
constexpr int BN = 256;            // output cols per pair tile (B rows)
constexpr int BN_CTA = BN / 2;     // B rows loaded by each CTA
constexpr int BK = 256;            // K elements per stage
constexpr int BKB = BK / 2;        // bytes per row per stage (128: one swizzle row)
constexpr int MMA_K = 64;          // K per tcgen05.mma for kind::mxf4nvf4
constexpr int KSTEPS = BK / MMA_K; // 4 MMAs per stage
constexpr int STAGES = 5;
constexpr int A_BYTES = BM * BKB;          // 16 KiB
constexpr int B_BYTES = BN_CTA * BKB;      // 16 KiB
constexpr int SF_BAND_BYTES = KSTEPS * 512;  // one 128-row band, one stage: 2 KiB
constexpr int SFA_BYTES = SF_BAND_BYTES;
constexpr int SFB_BYTES = 2 * SF_BAND_BYTES;
constexpr int NUM_THREADS = 480;
constexpr int NUM_SF_WARPS = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr int SF_PRODUCER_WARP = 2;
constexpr int FIRST_SF_WARP = 3;
constexpr int FIRST_EPI_WARP = FIRST_SF_WARP + NUM_SF_WARPS;
constexpr int TMEM_COLS = 512;
constexpr int SF_COLS_PER_STAGE = KSTEPS * 4 + KSTEPS * 8;  // 48
constexpr int EPI_BOX = 32;                                  // 32 x 32 BF16 store boxes
constexpr int EPI_BUF_BYTES = EPI_BOX * EPI_BOX * 2;         // 2 KiB
constexpr int TILE_GROUP = 16;                               // pair tiles along M per raster group

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
constexpr int OFF_EPI = OFF_SFB + STAGES * SFB_BYTES;
constexpr int OFF_BAR = OFF_EPI + NUM_EPI_WARPS * 2 * EPI_BUF_BYTES;
constexpr int NUM_BARS = 5 * STAGES + 4;
constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
constexpr int SMEM_USED = OFF_ABORT + 4;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_EPI % 1024 == 0, "store staging must keep the swizzle pattern aligned");
static_assert(256 + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "tensor memory budget");

// Instruction descriptor for kind::mxf4nvf4 (dense, K-major A and B, E2M1
// operands, UE4M3 scales, scale-factor ids 0):
//   [7,10) A format = E2M1 (1), [10,13) B format = E2M1 (1),
//   [17,23) N >> 3, [23] scale type UE4M3 = 0, [24,29) M >> 4.
constexpr uint32_t make_idesc(int m, int n) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
constexpr uint32_t IDESC = make_idesc(BM_PAIR, BN);

// Shared-memory matrix descriptor: start address, leading/stride byte
// offsets (in 16-byte units), descriptor version 1 (bit 46), swizzle mode in
// bits [61,64) (2 = 128-byte swizzle, 0 = none).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swz << 61);
}

// Two accumulator values (fp32 bit patterns) scaled by alpha and rounded to
// BF16 (nearest even), packed with `lo` in the low half-word.  The packed
// multiply rounds each lane like the scalar one; the product is rounded to
// fp32 first, and the result differs from rounding the exact product only
// when that fp32 value sits exactly on a BF16 tie.
__device__ __forceinline__ uint32_t scale_pack2(uint32_t lo, uint32_t hi, uint64_t alpha2) {
  float a, b;
  f2_unpack(f2_mul(f2_pack(__uint_as_float(lo), __uint_as_float(hi)), alpha2), a, b);
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// One launch runs up to MAX_PROBS independent GEMMs (a group): their pair
// tiles form one list, problem 0's first, shared out to the persistent pairs.
constexpr int MAX_PROBS = 2;

struct Prob {
  const uint8_t* sfa;  // A scales, MMA layout
  const uint8_t* sfb;  // B scales, MMA layout
  const float* sga;
  const float* sgb;
  int M, N, K;
  int bands_a, bands_b;  // 128-row scale bands present in the scale buffers
  int tiles_m, tiles_n;
  int tile0;             // index of the problem's first tile in the launch's list
};

struct Params {
  Prob prob[MAX_PROBS];
  int nprob;
  int num_tiles;  // all problems
  uint32_t* status;
};

// Tensor maps of every problem (grid constants, addressed per tile).
struct Maps {
  CUtensorMap a[MAX_PROBS], b[MAX_PROBS], c[MAX_PROBS], sfb[MAX_PROBS];
};

// Tile t of the launch: its problem (returned) and pair-tile coordinates.
// Within a problem: groups of TILE_GROUP tiles along M, M fastest inside a
// group, so the tiles in flight across the GPU share A and B panels in L2.
__device__ __forceinline__ int tile_coords(const Params& p, int t, int& tm, int& tn) {
  const int q = (p.nprob > 1 && t >= p.prob[1].tile0) ? 1 : 0;
  const Prob& g = p.prob[q];
  t -= g.tile0;
  const int group_span = TILE_GROUP * g.tiles_n;
  const int grp = t / group_span;
  const int first_m = grp * TILE_GROUP;
  const int gm = min(TILE_GROUP, g.tiles_m - first_m);
  const int r = t - grp * group_span;
  tm = first_m + r % gm;
  tn = r / gm;
  return q;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
nvfp4_gemm_kernel(const __grid_constant__ Maps maps, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + OFF_BAR;             // STAGES: both CTAs' A/B landed (leader)
  const uint32_t bar_empty = bar_full + STAGES * 8;      // STAGES: pair MMAs done with the stage
  const uint32_t bar_sf = bar_empty + STAGES * 8;        // STAGES: scales in tensor memory (leader)
  const uint32_t bar_sf_full = bar_sf + STAGES * 8;      // STAGES: scale atoms in shared memory
  const uint32_t bar_sf_free = bar_sf_full + STAGES * 8; // STAGES: scale slot read by the writers
  const uint32_t bar_tmem_full = bar_sf_free + STAGES * 8;  // accumulator ready for the epilogue
  const uint32_t bar_tmem_empty = bar_tmem_full + 8;     // accumulator drained (leader)
  const uint32_t bar_exit = bar_tmem_empty + 8;          // peer CTA finished
  const uint32_t bar_mma_done = bar_exit + 8;            // every pair MMA issued has completed
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM_SLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = (int)cluster_id_x();
  const int num_pairs = (int)cluster_count_x();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_sf + 8 * s, 2 * NUM_SF_WARPS);
      mbar_init(bar_sf_full + 8 * s, 1);
      mbar_init(bar_sf_free + 8 * s, NUM_SF_WARPS);
    }
    mbar_init(bar_tmem_full, 1);
    mbar_init(bar_tmem_empty, 2 * NUM_EPI_WARPS);
    mbar_init(bar_exit, 1);
    mbar_init(bar_mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
    for (int q = 0; q < p.nprob; ++q) {
      prefetch_tensormap(&maps.a[q]);
      prefetch_tensormap(&maps.b[q]);
      prefetch_tensormap(&maps.c[q]);
      prefetch_tensormap(&maps.sfb[q]);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(sbase + OFF_TMEM_SLOT, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  // Both CTAs' barriers must be initialised before either signals the other.
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int prod_stage = 0;      // operand producer's ring position (thread 0)
  uint32_t prod_phase = 0;
  if (warp == 0) {
    // ------------------------------------------------- operand producer --
    if (lane == 0) {
      const uint32_t leader_full = mapa_shared(bar_full, 0);
      int& stage = prod_stage;
      uint32_t& phase = prod_phase;
      for (int t = pair; t < p.num_tiles && !*abort_flag; t += num_pairs) {
        int tm, tn;
        const int q = tile_coords(p, t, tm, tn);
        const CUtensorMap* tmap_a = &maps.a[q];
        const CUtensorMap* tmap_b = &maps.b[q];
        const int num_kb = p.prob[q].K / BK;
        const int band_a = 2 * tm + (int)rank;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait_cluster(bar_empty + 8 * stage, phase ^ 1u, p.status)) { *abort_flag = 1; break; }
          // The leader arms its barrier for both CTAs' bytes; the peer's
          // copies may land before or after that, either is fine.
          if (rank == 0) mbar_arrive_expect_tx(bar_full + 8 * stage, 2 * (A_BYTES + B_BYTES));
          tma_load_2d_pair(sbase + OFF_A + stage * A_BYTES, tmap_a, kb * BKB, band_a * BM, leader_full + 8 * stage);
          tma_load_2d_pair(sbase + OFF_B + stage * B_BYTES, tmap_b, kb * BKB, tn * BN + (int)rank * BN_CTA,
                           leader_full + 8 * stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------- MMA issuer (leader CTA) --
    // The whole warp runs the loop and waits (bounded spins inside single asm
    // blocks, decisions made warp-uniform by a vote); one elected lane issues
    // the MMAs.  A single-lane issue loop with two waits per stage held the
    // tensor pipe to ~180 cycles per 128-cycle MMA.
    if (rank == 0) {
      const bool leader = elect_one();
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = pair; t < p.num_tiles && ok; t += num_pairs, ++it) {
        int tm, tn;
        const int num_kb = p.prob[tile_coords(p, t, tm, tn)].K / BK;
        // one vote keeps every lane's decision identical (waits and the
        // abort flag are read per lane)
        ok = __all_sync(0xFFFFFFFFu,
                        mbar_wait_spin(bar_tmem_empty, (uint32_t)(it & 1) ^ 1u, p.status) && !*abort_flag);
        if (!ok) break;
        tc_fence_after();
        for (int kb = 0; kb < num_kb; ++kb) {
          ok = __all_sync(0xFFFFFFFFu, mbar_wait_spin(bar_full + 8 * stage, phase, p.status) &&
                                           mbar_wait_spin(bar_sf + 8 * stage, phase, p.status));
          if (!ok) break;
          tc_fence_after();
          if (leader) {
            const uint32_t sf_col = tmem_base + 256u + (uint32_t)(stage * SF_COLS_PER_STAGE);
            const uint32_t a_s = sbase + OFF_A + stage * A_BYTES;
            const uint32_t b_s = sbase + OFF_B + stage * B_BYTES;
#pragma unroll
            for (int j = 0; j < KSTEPS; ++j) {
              // K-major, 128-byte swizzle: 8-row groups 1024 B apart; the K
              // offset inside the swizzle row advances the start address.
              const uint64_t ad = smem_desc(a_s + 32 * j, 16, 1024, 2);
              const uint64_t bd = smem_desc(b_s + 32 * j, 16, 1024, 2);
              tc_mma_nvf4_pair(tmem_base, ad, bd, IDESC, sf_col + 4 * j, sf_col + 16 + 8 * j,
                               (kb > 0 || j > 0) ? 1u : 0u);
            }
            tc_commit_pair(bar_empty + 8 * stage, 0x3);
          }
          __syncwarp();
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (leader) tc_commit_pair(bar_tmem_full, 0x3);
        __syncwarp();
      }
      if (!ok && leader) *abort_flag = 1;
      // Also on the abort paths: tell both CTAs when the last MMA issued has
      // finished reading their shared memory and writing their tensor memory.
      if (leader) tc_commit_pair(bar_mma_done, 0x3);
      __syncwarp();
    }
  } else if (warp == SF_PRODUCER_WARP) {
    // --------------------------------------------------- scale producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = pair; t < p.num_tiles && !*abort_flag; t += num_pairs) {
        int tm, tn;
        const int q = tile_coords(p, t, tm, tn);
        const Prob& g = p.prob[q];
        const int num_kb = g.K / BK;
        const int64_t atoms_per_band = g.K / 64;
        const int band_a = 2 * tm + (int)rank;
        const bool a_ok = band_a < g.bands_a;
        // both bands of B scales come in one box (a missing second band reads as zeros)
        const uint32_t tx = (a_ok ? SFA_BYTES : 0) + SFB_BYTES;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(bar_sf_free + 8 * stage, phase ^ 1u, p.status)) { *abort_flag = 1; break; }
          const uint32_t full = bar_sf_full + 8 * stage;
          mbar_arrive_expect_tx(full, tx);
          if (a_ok)
            bulk_load(sbase + OFF_SFA + stage * SFA_BYTES,
                      g.sfa + ((int64_t)band_a * atoms_per_band + (int64_t)kb * KSTEPS) * 512, SFA_BYTES, full);
          tma_load_3d(sbase + OFF_SFB + stage * SFB_BYTES, &maps.sfb[q], 0, kb * (SF_BAND_BYTES / 256), 2 * tn, full);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // Let in-flight scale copies land before the CTA can exit.
      for (int s = 0; s < STAGES; ++s) {
        const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
        mbar_wait(bar_sf_full + 8 * s, par, p.status, 100000000ull);
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
    const uint32_t leader_sf = mapa_shared(bar_sf, 0);
    int stage = 0;
    uint32_t phase = 0;
    for (int t = pair; t < p.num_tiles && !*abort_flag; t += num_pairs) {
      int tm, tn;
      const Prob& g = p.prob[tile_coords(p, t, tm, tn)];
      const int num_kb = g.K / BK;
      const bool a_ok = 2 * tm + (int)rank < g.bands_a;
      const bool b1_ok = 2 * tn + 1 < g.bands_b;
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb) {
        // the stage's scale atoms are in shared memory, and its scale
        // columns are free (the MMAs that last used them have completed)
        if (!mbar_wait(bar_sf_full + 8 * stage, phase, p.status) ||
            !mbar_wait_cluster(bar_empty + 8 * stage, phase ^ 1u, p.status)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* sfa_s = smem + OFF_SFA + stage * SFA_BYTES + lane * 16;
        const uint8_t* sfb_s = smem + OFF_SFB + stage * SFB_BYTES + lane * 16;
        uint32_t va[16], vb[32];
#pragma unroll
        for (int j = 0; j < KSTEPS; ++j) {
          uint4 a = *reinterpret_cast<const uint4*>(sfa_s + 512 * j);
          const uint4 b0 = *reinterpret_cast<const uint4*>(sfb_s + 512 * j);
          uint4 b1 = *reinterpret_cast<const uint4*>(sfb_s + SF_BAND_BYTES + 512 * j);
          if (!a_ok) a = make_uint4(0u, 0u, 0u, 0u);    // rows past the operand: zero scales
          if (!b1_ok) b1 = make_uint4(0u, 0u, 0u, 0u);
          va[4 * j + 0] = a.x; va[4 * j + 1] = a.y; va[4 * j + 2] = a.z; va[4 * j + 3] = a.w;
          vb[8 * j + 0] = b0.x; vb[8 * j + 1] = b0.y; vb[8 * j + 2] = b0.z; vb[8 * j + 3] = b0.w;
          vb[8 * j + 4] = b1.x; vb[8 * j + 5] = b1.y; vb[8 * j + 6] = b1.z; vb[8 * j + 7] = b1.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sf_free + 8 * stage);  // the slot's shared memory may be refilled
        const uint32_t col = tmem_base + lane_off + 256u + (uint32_t)(stage * SF_COLS_PER_STAGE);
        tmem_st_32x32b_x16(col, va);
        tmem_st_32x32b_x16(col + 16, vb);
        tmem_st_32x32b_x16(col + 32, vb + 16);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(leader_sf + 8 * stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
    }
  } else {
    // --------------------------------------------------------- epilogue --
    const int quad = warp & 3;                     // lane quadrant this warp may access
    const int half = (warp - FIRST_EPI_WARP) >> 2;  // which 128 accumulator columns
    static_assert(MAX_PROBS == 2, "one alpha per problem below");
    const float alpha_0 = __fmul_rn(*p.prob[0].sga, *p.prob[0].sgb);
    const float alpha_1 = p.nprob > 1 ? __fmul_rn(*p.prob[1].sga, *p.prob[1].sgb) : 0.0f;
    const uint32_t leader_tmem_empty = mapa_shared(bar_tmem_empty, 0);
    const uint32_t stage_buf = sbase + OFF_EPI + (uint32_t)((warp - FIRST_EPI_WARP) * 2 * EPI_BUF_BYTES);
    const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(half * 128);
    // Lane = row of the 32 x 32 box; its four 16-byte pieces go to swizzled
    // positions (64-byte swizzle: piece c of row r at c ^ ((r >> 1) & 3)).
    const uint32_t row_off = (uint32_t)lane * 64u;
    const uint32_t swz = (uint32_t)((lane >> 1) & 3);
    int it = 0;
    for (int t = pair; t < p.num_tiles; t += num_pairs, ++it) {
      if (!mbar_wait_cluster(bar_tmem_full, (uint32_t)(it & 1), p.status)) { *abort_flag = 1; break; }
      if (*abort_flag) break;
      tc_fence_after();
      int tm, tn;
      const int q = tile_coords(p, t, tm, tn);
      const Prob& g = p.prob[q];
      const float alpha = q == 0 ? alpha_0 : alpha_1;
      const uint64_t alpha2 = f2_pack(alpha, alpha);
      // Pull this warp's 32 x 128 accumulator block out of tensor memory
      // (two 32-column loads per wait), scaling and rounding into 64 packed
      // bf16x2 words; release the accumulator as soon as the last chunk is
      // in registers so the next tile's MMAs overlap the stores.
      uint32_t w[64];
      {
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(taddr, v0);
        tmem_ld_32x32b_x32(taddr + 32, v1);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          w[j] = scale_pack2(v0[2 * j], v0[2 * j + 1], alpha2);
          w[16 + j] = scale_pack2(v1[2 * j], v1[2 * j + 1], alpha2);
        }
        tmem_ld_32x32b_x32(taddr + 64, v0);
        tmem_ld_32x32b_x32(taddr + 96, v1);
        tc_wait_ld();
        // every accumulator column this warp reads is in registers: release
        // the accumulator before converting the second half
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(leader_tmem_empty);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          w[32 + j] = scale_pack2(v0[2 * j], v0[2 * j + 1], alpha2);
          w[48 + j] = scale_pack2(v1[2 * j], v1[2 * j + 1], alpha2);
        }
      }
      const int row0 = tm * BM_PAIR + (int)rank * BM + quad * 32;
      const int col0 = tn * BN + half * 128;
      if (row0 >= g.M) continue;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        if (col0 + EPI_BOX * ch >= g.N) break;
        const uint32_t buf = stage_buf + (uint32_t)((ch & 1) * EPI_BUF_BYTES);
        // the store that last used this buffer must have read it
        if (lane == 0) {
          if (ch == 0)
            bulk_wait_group_read<0>();
          else
            bulk_wait_group_read<1>();
        }
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 4; ++c)
          st_shared_v4(buf + row_off + (((uint32_t)c ^ swz) << 4), w[16 * ch + 4 * c], w[16 * ch + 4 * c + 1],
                       w[16 * ch + 4 * c + 2], w[16 * ch + 4 * c + 3]);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&maps.c[q], buf, col0 + EPI_BOX * ch, row0);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group<0>();
  }

  // ----------------------------------------------------------- teardown --
  // Neither CTA may leave while the leader's MMAs can still use its shared
  // and tensor memory, or while the other CTA can still signal its barriers.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_wait_cluster(bar_mma_done, 0, p.status, 10000000000ull);
    // Both CTAs' operand copies complete on the leader's `full` barriers.
    // The leader waits (bounded) for the last phase it armed on every stage,
    // so neither CTA releases its shared memory while a copy it armed can
    // still land; in a run without an abort every such phase has completed
    // (the MMA warp consumed it) and these waits return at once.  A stage
    // never armed passes at once too (parity of the phase before the first).
    if (rank == 0) {
      for (int s = 0; s < STAGES; ++s) {
        const uint32_t par = (s < prod_stage) ? prod_phase : (prod_phase ^ 1u);
        mbar_wait(bar_full + 8 * s, par, p.status, 100000000ull);
      }
    }
    // After an abort the peer may also have issued copies for a stage the
    // leader never armed, which no barrier here can observe: give those time
    // to land before either CTA can exit.
    if (*abort_flag) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 200000ull) {}
    }
    mbar_arrive_cluster(mapa_shared(bar_exit, rank ^ 1u));
    mbar_wait_cluster(bar_exit, 0, p.status, 10000000000ull);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------- MMA-rate probe --
// Measures the issue-to-completion time of a run of back-to-back pair MMAs of
// the GEMM's kind (kind::mxf4nvf4 block_scale scale_vec::4X, M = 256 over the
// pair, the given N, K = 64) with no data movement: thread 0 of the leader
// CTA issues n_mma MMAs on fixed shared-memory operands and fixed scale
// columns (their contents do not matter for the timing), commits them to an
// mbarrier in both CTAs and waits for it.  out[2 p] = SM cycles (clock64)
// and out[2 p + 1] = nanoseconds (globaltimer) of pair p, from before the
// first issue to the commit's arrival.  Every wait is bounded.
constexpr int PROBE_THREADS = 128;
constexpr int PROBE_OFF_BAR = A_BYTES + B_BYTES;  // operands at 0 and A_BYTES
constexpr int PROBE_SMEM = PROBE_OFF_BAR + 16 + 1024;

__global__ void __launch_bounds__(PROBE_THREADS, 1)
mma_rate_kernel(int n_mma, uint32_t idesc, unsigned long long* out, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar = sbase + PROBE_OFF_BAR;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + PROBE_OFF_BAR + 8);
  const int warp = threadIdx.x >> 5;
  const uint32_t rank = cluster_ctarank();
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc_pair(sbase + PROBE_OFF_BAR + 8, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) {
    if (rank == 0) {
      const unsigned long long c0 = clock64();
      const uint64_t t0 = globaltimer_ns();
      const uint64_t ad = smem_desc(sbase, 16, 1024, 2);
      const uint64_t bd = smem_desc(sbase + A_BYTES, 16, 1024, 2);
      for (int i = 0; i < n_mma; ++i) {
        const uint32_t j = (uint32_t)(i & 3);
        tc_mma_nvf4_pair(tmem_base, ad + 2 * j, bd + 2 * j, idesc, tmem_base + 256u + 4u * j,
                         tmem_base + 256u + 16u + 8u * j, i > 0 ? 1u : 0u);
      }
      tc_commit_pair(bar, 0x3);
      const bool ok = mbar_wait_cluster(bar, 0, status);
      const unsigned long long c1 = clock64();
      const uint64_t t1 = globaltimer_ns();
      const int pair = (int)cluster_id_x();
      out[2 * pair] = ok ? c1 - c0 : 0ull;
      out[2 * pair + 1] = ok ? t1 - t0 : 0ull;
    } else {
      (void)mbar_wait_cluster(bar, 0, status);
    }
  }
  tc_fence_before();
  __syncthreads();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
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
// (128 bytes, 128 rows) and 128-byte swizzle; out-of-range rows read as zero.
static bool make_code_map(CUtensorMap* map, const void* base, int64_t rows, int64_t kbytes) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kbytes, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kbytes};
  const cuuint32_t box[2] = {(cuuint32_t)gemm::BKB, (cuuint32_t)gemm::BM};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map over a bf16 matrix [rows, cols] (row stride ld elements) with boxes of
// box_cols x box_rows elements, no swizzle; elements outside the matrix read
// as zero.  The quantisers stage their input tiles through it.
bool make_bf16_tile_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                        int box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over B's scales in the MMA layout, viewed as [bands][K/64 atoms x
// 2][256 bytes]: one box of (256 B, one stage's 8 pieces, 2 bands) is the
// 4 KiB of scales a pair tile needs per K step.  Bands past the operand read
// as zero.
static bool make_sfb_map(CUtensorMap* map, const void* base, int64_t bands, int64_t atoms_per_band) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {256, (cuuint64_t)atoms_per_band * 2, (cuuint64_t)bands};
  const cuuint64_t strides[2] = {256, (cuuint64_t)atoms_per_band * 512};
  const cuuint32_t box[3] = {256, (cuuint32_t)(gemm::SF_BAND_BYTES / 256), 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map over the BF16 output [M, N] (row stride ldc elements) with 32 x 32 boxes
// and 64-byte swizzle; stores outside [M, N] are dropped by the hardware.
static bool make_out_map(CUtensorMap* map, void* base, int64_t M, int64_t N, int64_t ldc) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)ldc * 2};
  const cuuint32_t box[2] = {(cuuint32_t)gemm::EPI_BOX, (cuuint32_t)gemm::EPI_BOX};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// Launch the GEMMs of a group (1 .. MAX_PROBS problems, each with M, N, K
// > 0, validated by the caller) as one persistent grid.  Problems with longer
// contractions go first in the tile list, so the pairs' last tiles are the
// short ones.
int gemm_group_launch(const DeviceInfo& dev, int count, const nvfp4_tensor* const* A, const nvfp4_tensor* const* B,
                      void* const* c, const int64_t* ldc, cudaStream_t stream) {
  using namespace gemm;
  if (count < 1 || count > MAX_PROBS) return NVFP4_ERR_INVALID_ARG;
  static std::mutex mu;
  static int max_pairs[64] = {};
  int pairs_cap = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev.device < 0 || dev.device >= 64) return NVFP4_ERR_CUDA;
    if (max_pairs[dev.device] == 0) {
      if (cudaFuncSetAttribute(nvfp4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
          cudaSuccess)
        return NVFP4_ERR_CUDA;
      // How many CTA pairs fit on the device at once (a persistent grid must
      // not exceed it, or the surplus pairs would wait for a second wave).
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = 2;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * (dev.sm_count / 2), 1, 1);
      cfg.blockDim = dim3(NUM_THREADS, 1, 1);
      cfg.dynamicSmemBytes = SMEM_BYTES;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, nvfp4_gemm_kernel, &cfg) != cudaSuccess || n <= 0)
        return NVFP4_ERR_CUDA;
      max_pairs[dev.device] = n;
    }
    pairs_cap = max_pairs[dev.device];
  }
  int order[MAX_PROBS];
  for (int i = 0; i < count; ++i) order[i] = i;
  if (count == 2 && A[1]->cols > A[0]->cols) {
    order[0] = 1;
    order[1] = 0;
  }
  Maps maps;
  memset(&maps, 0, sizeof(maps));
  Params p;
  memset(&p, 0, sizeof(p));
  int tiles = 0;
  for (int k = 0; k < count; ++k) {
    const nvfp4_tensor& a = *A[order[k]];
    const nvfp4_tensor& b = *B[order[k]];
    if (!make_code_map(&maps.a[k], a.codes, a.rows, a.cols / 2)) return NVFP4_ERR_CUDA;
    if (!make_code_map(&maps.b[k], b.codes, b.rows, b.cols / 2)) return NVFP4_ERR_CUDA;
    if (!make_out_map(&maps.c[k], c[order[k]], a.rows, b.rows, ldc[order[k]])) return NVFP4_ERR_CUDA;
    if (!make_sfb_map(&maps.sfb[k], b.scales, (b.rows + BM - 1) / BM, a.cols / 64)) return NVFP4_ERR_CUDA;
    Prob& g = p.prob[k];
    g.sfa = a.scales;
    g.sfb = b.scales;
    g.sga = a.global_scale;
    g.sgb = b.global_scale;
    g.M = (int)a.rows;
    g.N = (int)b.rows;
    g.K = (int)a.cols;
    g.bands_a = (g.M + BM - 1) / BM;
    g.bands_b = (g.N + BM - 1) / BM;
    g.tiles_m = (g.M + BM_PAIR - 1) / BM_PAIR;
    g.tiles_n = (g.N + BN - 1) / BN;
    g.tile0 = tiles;
    tiles += g.tiles_m * g.tiles_n;
  }
  p.nprob = count;
  p.num_tiles = tiles;
  p.status = dev.status;
  const int pairs = tiles < pairs_cap ? tiles : pairs_cap;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, nvfp4_gemm_kernel, maps, p) != cudaSuccess) return NVFP4_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

int gemm_launch(const DeviceInfo& dev, const nvfp4_tensor& A, const nvfp4_tensor& B, void* c, int64_t ldc,
                cudaStream_t stream) {
  const nvfp4_tensor* a = &A;
  const nvfp4_tensor* b = &B;
  return gemm_group_launch(dev, 1, &a, &b, &c, &ldc, stream);
}

}  // namespace nvfp4

namespace nvfp4 {

int mma_rate_launch(const DeviceInfo& dev, int n_mma, int mma_n, unsigned long long* out, int* pairs_out,
                    cudaStream_t stream) {
  using namespace gemm;
  static std::mutex mu;
  static int max_pairs[64] = {};
  int pairs = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev.device < 0 || dev.device >= 64) return NVFP4_ERR_CUDA;
    if (max_pairs[dev.device] == 0) {
      if (cudaFuncSetAttribute(mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PROBE_SMEM) !=
          cudaSuccess)
        return NVFP4_ERR_CUDA;
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = 2;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * (dev.sm_count / 2), 1, 1);
      cfg.blockDim = dim3(PROBE_THREADS, 1, 1);
      cfg.dynamicSmemBytes = PROBE_SMEM;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, mma_rate_kernel, &cfg) != cudaSuccess || n <= 0) return NVFP4_ERR_CUDA;
      // one pair per two SMs (a pair per SM pair, as the GEMM runs)
      max_pairs[dev.device] = n < dev.sm_count / 2 ? n : dev.sm_count / 2;
    }
    pairs = max_pairs[dev.device];
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(PROBE_THREADS, 1, 1);
  cfg.dynamicSmemBytes = PROBE_SMEM;
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, mma_rate_kernel, n_mma, make_idesc(BM_PAIR, mma_n), out, dev.status) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  *pairs_out = pairs;
  return cudaPeekAtLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace nvfp4

// --------------------------------------------------- delivery-rate probe --
// How fast asynchronous copies fill one multiprocessor's shared memory, the
// path every operand and scale byte of the GEMM takes.  Thread 0 of each CTA
// keeps COPY_SLOTS copies of COPY_CHUNK bytes in flight, reusing a slot as
// soon as its previous copy has landed; the data is never read.  kBoxes:
// the GEMM's operand boxes (128 rows x 128 B, 128-byte swizzle) through a
// tensor map; otherwise plain bulk copies of consecutive chunks.  Every wait
// is bounded.
namespace nvfp4 {
namespace gemm {

constexpr int COPY_CHUNK = 16384;
constexpr int COPY_SLOTS = 12;
constexpr int COPY_SMEM = COPY_CHUNK * COPY_SLOTS + COPY_SLOTS * 8 + 1024;
constexpr int COPY_ROW_BYTES = 2048;  // box mode: src rows of an operand with K = 4096
constexpr int COPY_BOXES_PER_BAND = COPY_ROW_BYTES / BKB;

template <bool kBoxes>
__global__ void __launch_bounds__(32, 1)
copy_rate_kernel(const __grid_constant__ CUtensorMap map, const uint8_t* src, int64_t nchunks, int iters,
                 unsigned long long* out, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  if (threadIdx.x != 0) return;
  const uint32_t ring = smem_u32(smem);
  const uint32_t bars = ring + COPY_CHUNK * COPY_SLOTS;
  for (int s = 0; s < COPY_SLOTS; ++s) mbar_init(bars + 8 * s, 1);
  fence_barrier_init();
  if (kBoxes) prefetch_tensormap(&map);
  int64_t chunk = ((int64_t)blockIdx.x * 7919) % nchunks;  // CTAs start far apart in src
  const uint64_t t0 = globaltimer_ns();
  const unsigned long long c0 = clock64();
  bool ok = true;
  int issued = 0;
  for (; issued < iters; ++issued) {
    const int s = issued % COPY_SLOTS;
    const uint32_t bar = bars + 8 * s;
    if (issued >= COPY_SLOTS && !mbar_wait(bar, (uint32_t)((issued / COPY_SLOTS - 1) & 1), status)) {
      ok = false;
      break;
    }
    mbar_arrive_expect_tx(bar, COPY_CHUNK);
    if (kBoxes) {
      const int64_t band = chunk / COPY_BOXES_PER_BAND, kb = chunk - band * COPY_BOXES_PER_BAND;
      tma_load_2d(ring + s * COPY_CHUNK, &map, (int32_t)(kb * BKB), (int32_t)(band * BM), bar);
    } else {
      bulk_load(ring + s * COPY_CHUNK, src + chunk * COPY_CHUNK, COPY_CHUNK, bar);
    }
    chunk += gridDim.x;
    if (chunk >= nchunks) chunk %= nchunks;
  }
  // every copy issued must land before the CTA exits, also after a timeout
  for (int i = issued > COPY_SLOTS ? issued - COPY_SLOTS : 0; i < issued; ++i)
    ok = mbar_wait(bars + 8 * (i % COPY_SLOTS), (uint32_t)((i / COPY_SLOTS) & 1), status) && ok;
  const uint64_t t1 = globaltimer_ns();
  const unsigned long long c1 = clock64();
  out[3 * blockIdx.x] = ok ? t1 - t0 : 0ull;
  out[3 * blockIdx.x + 1] = ok ? (unsigned long long)iters * COPY_CHUNK : 0ull;
  out[3 * blockIdx.x + 2] = ok ? c1 - c0 : 0ull;
}

}  // namespace gemm

int copy_rate_launch(const DeviceInfo& dev, const void* src, int64_t src_bytes, int mode, int ctas, int iters,
                     unsigned long long* out, cudaStream_t stream) {
  using namespace gemm;
  CUtensorMap map;
  memset(&map, 0, sizeof(map));
  int64_t nchunks = src_bytes / COPY_CHUNK;
  if (mode == 1) {
    const int64_t bands = src_bytes / ((int64_t)COPY_ROW_BYTES * BM);
    if (!make_code_map(&map, src, bands * BM, COPY_ROW_BYTES)) return NVFP4_ERR_CUDA;
    nchunks = bands * COPY_BOXES_PER_BAND;
  }
  auto kernel = mode == 1 ? copy_rate_kernel<true> : copy_rate_kernel<false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, COPY_SMEM) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  kernel<<<ctas, 32, COPY_SMEM, stream>>>(map, static_cast<const uint8_t*>(src), nchunks, iters, out, dev.status);
  return cudaPeekAtLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace nvfp4
