// nvfp4_internal.h -- host-side interfaces between the library's translation
// units (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/nvfp4.h"

namespace nvfp4 {

// Per-device state owned by the API layer.
struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  uint32_t* status = nullptr;  // device address of the status word
};

// Current device's info (filled once per device); nullptr on failure.
const DeviceInfo* device_info();

// TMA map over a bf16 matrix [rows, cols] (row stride ld elements) with
// box_cols x box_rows boxes, zero fill outside; false on failure.
bool make_bf16_tile_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                        int box_rows);

// Quantiser entry used by both public quantise calls.  Arguments have been
// validated by the caller.
int quantize_launch(const DeviceInfo& dev, const void* x, int64_t rows, int64_t cols, int64_t ld,
                    uint32_t flags, bool rht, uint64_t rht_seed, uint64_t sr_seed,
                    const float* amax_in, const nvfp4_tensor& out, cudaStream_t stream);

// Dual-orientation quantiser entry (arguments validated by the caller).
int quantize_dual_launch(const DeviceInfo& dev, const void* x, int64_t rows, int64_t cols, int64_t ld,
                         bool row_sr, uint64_t row_sr_seed, uint64_t rht_seed, uint64_t col_sr_seed,
                         const float* amax_row_in, const float* amax_col_in, const nvfp4_tensor& out_row,
                         const nvfp4_tensor& out_col, cudaStream_t stream);

// MXFP4 quantiser entry (arguments validated by the caller).
int quantize_mx_launch(const DeviceInfo& dev, const void* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* codes,
                       uint8_t* scales, cudaStream_t stream);

// GEMM entries (arguments validated by the caller): one GEMM, or a group of
// independent GEMMs (count 1 or 2, every M, N, K > 0) in one launch.
int gemm_launch(const DeviceInfo& dev, const nvfp4_tensor& A, const nvfp4_tensor& B, void* c,
                int64_t ldc, cudaStream_t stream);
int gemm_group_launch(const DeviceInfo& dev, int count, const nvfp4_tensor* const* A, const nvfp4_tensor* const* B,
                      void* const* c, const int64_t* ldc, cudaStream_t stream);

// FP4 MMA-rate probe (arguments validated by the caller).
int mma_rate_launch(const DeviceInfo& dev, int n_mma, int mma_n, unsigned long long* out, int* pairs_out,
                    cudaStream_t stream);

// Operand delivery-rate probe (arguments validated by the caller).
int copy_rate_launch(const DeviceInfo& dev, const void* src, int64_t src_bytes, int mode, int ctas, int iters,
                     unsigned long long* out, cudaStream_t stream);

// Bounded-wait self-test.
int selftest_wait_launch(const DeviceInfo& dev, uint64_t limit_ns, cudaStream_t stream);

// Codec diagnostics.
int encode_e2m1_rne_launch(const float* v, int64_t n, uint8_t* out, cudaStream_t stream);
int encode_e2m1_sr_launch(const float* v, const uint16_t* u, int64_t n, uint8_t* out,
                          cudaStream_t stream);
int encode_e4m3_launch(const float* t, int64_t n, uint8_t* out, cudaStream_t stream);

}  // namespace nvfp4
