// nvfp4_api.cu -- the C ABI declared in include/nvfp4.h: argument checks,
// per-device state (SM count, status word) and dispatch to the kernels.
#include <mutex>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

// One status word per device (bits kStatusTimeout / kStatusNonFinite).
__device__ uint32_t g_status_word;

// Clears exactly the bits the host has read, so a bit that a kernel on
// another stream raises between the read and the clear survives.
__global__ void status_clear_kernel(uint32_t* status, uint32_t bits) { atomicAnd(status, ~bits); }

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_info[kMaxDevices];
bool g_ready[kMaxDevices] = {};
}  // namespace

const DeviceInfo* device_info() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ready[dev]) {
    DeviceInfo d;
    d.device = dev;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
    if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return nullptr;
    if (cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return nullptr;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return nullptr;
    d.status = static_cast<uint32_t*>(ptr);
    g_info[dev] = d;
    g_ready[dev] = true;
  }
  return &g_info[dev];
}

}  // namespace nvfp4

using nvfp4::DeviceInfo;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Resolve the device and check that it runs sm_103a code (compute 10.3).
int check_device(const DeviceInfo** out) {
  const DeviceInfo* d = nvfp4::device_info();
  if (!d) return NVFP4_ERR_CUDA;
  if (!(d->cc_major == 10 && d->cc_minor == 3)) return NVFP4_ERR_UNSUPPORTED;
  *out = d;
  return NVFP4_OK;
}

// amax and global_scale are always required; codes and scales only when the
// operand holds elements (an empty torch tensor has a null data pointer).
int check_tensor_buffers(const nvfp4_tensor* t) {
  if (!t || !t->amax || !t->global_scale) return NVFP4_ERR_INVALID_ARG;
  if (t->reserved != 0) return NVFP4_ERR_INVALID_ARG;
  if (t->scale_layout != NVFP4_SCALES_CANONICAL && t->scale_layout != NVFP4_SCALES_MMA) return NVFP4_ERR_INVALID_ARG;
  if (t->rows < 0 || t->cols < 0) return NVFP4_ERR_INVALID_ARG;
  if (t->rows > 0 && t->cols > 0 && (!t->codes || !t->scales)) return NVFP4_ERR_INVALID_ARG;
  return NVFP4_OK;
}

int quantize_common(const void* x, int64_t rows, int64_t cols, int64_t ld, uint32_t flags, bool rht,
                    uint64_t rht_seed, uint64_t sr_seed, const float* amax_in, const nvfp4_tensor* out,
                    nvfp4_stream_t stream) {
  const uint32_t known = NVFP4_BLOCK_2D | NVFP4_ROUND_SR | NVFP4_TRANSPOSE_OUT;
  if (flags & ~known) return NVFP4_ERR_INVALID_ARG;
  if (rht && (flags & NVFP4_BLOCK_2D)) return NVFP4_ERR_INVALID_ARG;
  int rc = check_tensor_buffers(out);
  if (rc) return rc;
  if (rows < 0 || cols < 0 || ld < cols) return NVFP4_ERR_INVALID_ARG;
  const bool tr = (flags & NVFP4_TRANSPOSE_OUT) != 0;
  const int64_t orows = tr ? cols : rows, ocols = tr ? rows : cols;
  if (out->rows != orows || out->cols != ocols) return NVFP4_ERR_INVALID_ARG;
  if (ocols % 16 != 0) return NVFP4_ERR_INVALID_ARG;
  if ((flags & NVFP4_BLOCK_2D) && orows % 16 != 0) return NVFP4_ERR_INVALID_ARG;
  if (out->scale_layout == NVFP4_SCALES_MMA && ocols % 64 != 0) return NVFP4_ERR_INVALID_ARG;
  if (cols % 8 != 0 || ld % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  // block and tile indices are 32-bit inside the kernels
  if (rows > 0 && cols > 0 && (rows * (cols / 8)) >= (int64_t)1 << 31) return NVFP4_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  rc = check_device(&dev);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (rows == 0 || cols == 0) {
    // empty tensor: amax = s_g = 0 (or the supplied amax), nothing else to write
    if (amax_in == out->amax) {
      // supplied in place: already holds the amax
    } else if (amax_in) {
      if (cudaMemcpyAsync(out->amax, amax_in, sizeof(float), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    } else if (cudaMemsetAsync(out->amax, 0, sizeof(float), s) != cudaSuccess) {
      return NVFP4_ERR_CUDA;
    }
    if (cudaMemsetAsync(out->global_scale, 0, sizeof(float), s) != cudaSuccess) return NVFP4_ERR_CUDA;
    const size_t sb = nvfp4_scales_bytes(orows, ocols, out->scale_layout);
    if (sb && cudaMemsetAsync(out->scales, 0, sb, s) != cudaSuccess) return NVFP4_ERR_CUDA;
    return NVFP4_OK;
  }
  if (!x || !aligned16(x)) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(out->codes) && orows > 0) {
    // codes rows are written 8 bytes at a time
    if ((reinterpret_cast<uintptr_t>(out->codes) & 7u) != 0) return NVFP4_ERR_INVALID_ARG;
  }
  return nvfp4::quantize_launch(*dev, x, rows, cols, ld, flags, rht, rht_seed, sr_seed, amax_in, *out, s);
}

// Host-side checks of one GEMM: C[M, N] = A[M, K] * B[N, K]^T.
int check_gemm(const nvfp4_tensor* A, const nvfp4_tensor* B, const void* c, int64_t ldc) {
  int rc = check_tensor_buffers(A);
  if (rc) return rc;
  rc = check_tensor_buffers(B);
  if (rc) return rc;
  if (A->scale_layout != NVFP4_SCALES_MMA || B->scale_layout != NVFP4_SCALES_MMA) return NVFP4_ERR_INVALID_ARG;
  const int64_t M = A->rows, N = B->rows, K = A->cols;
  if (B->cols != K) return NVFP4_ERR_INVALID_ARG;
  if (K % 256 != 0) return NVFP4_ERR_INVALID_ARG;
  if (M >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 31)) return NVFP4_ERR_INVALID_ARG;
  if (ldc < N || ldc % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (M > 0 && N > 0 && (!c || !aligned16(c))) return NVFP4_ERR_INVALID_ARG;
  if (M > 0 && N > 0 && K > 0 &&
      (!aligned16(A->codes) || !aligned16(B->codes) || !aligned16(A->scales) || !aligned16(B->scales)))
    return NVFP4_ERR_INVALID_ARG;
  return NVFP4_OK;
}

}  // namespace

extern "C" {

size_t nvfp4_scales_bytes(int64_t rows, int64_t cols, int32_t layout) {
  if (rows < 0 || cols < 0 || cols % 16 != 0) return 0;
  if (layout == NVFP4_SCALES_CANONICAL) return (size_t)(rows * (cols / 16));
  if (layout == NVFP4_SCALES_MMA) {
    if (cols % 64 != 0) return 0;
    return (size_t)(((rows + 127) / 128) * 128 * (cols / 16));
  }
  return 0;
}

int nvfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, uint32_t flags, uint64_t sr_seed,
                   const float* amax_in, const nvfp4_tensor* out, nvfp4_stream_t stream) {
  return quantize_common(x, rows, cols, ld, flags, false, 0, sr_seed, amax_in, out, stream);
}

int nvfp4_quantize_rht_sr(const void* x, int64_t rows, int64_t cols, int64_t ld, uint32_t flags,
                          uint64_t rht_seed, uint64_t sr_seed, const float* amax_in, const nvfp4_tensor* out,
                          nvfp4_stream_t stream) {
  return quantize_common(x, rows, cols, ld, flags | NVFP4_ROUND_SR, true, rht_seed, sr_seed, amax_in, out,
                         stream);
}

int nvfp4_quantize_dual(const void* x, int64_t rows, int64_t cols, int64_t ld, uint32_t row_flags,
                        uint64_t row_sr_seed, uint64_t rht_seed, uint64_t col_sr_seed, const float* amax_row_in,
                        const float* amax_col_in, const nvfp4_tensor* out_row, const nvfp4_tensor* out_col,
                        nvfp4_stream_t stream) {
  if (row_flags & ~NVFP4_ROUND_SR) return NVFP4_ERR_INVALID_ARG;  // 1D blocks, no transpose
  int rc = check_tensor_buffers(out_row);
  if (rc) return rc;
  rc = check_tensor_buffers(out_col);
  if (rc) return rc;
  if (out_row->scale_layout != out_col->scale_layout) return NVFP4_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || ld < cols) return NVFP4_ERR_INVALID_ARG;
  if (out_row->rows != rows || out_row->cols != cols || out_col->rows != cols || out_col->cols != rows)
    return NVFP4_ERR_INVALID_ARG;
  if (cols % 16 != 0 || rows % 16 != 0) return NVFP4_ERR_INVALID_ARG;
  if (out_row->scale_layout == NVFP4_SCALES_MMA && (cols % 64 != 0 || rows % 64 != 0)) return NVFP4_ERR_INVALID_ARG;
  if (ld % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (rows > 0 && cols > 0 && (rows * (cols / 8)) >= (int64_t)1 << 31) return NVFP4_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  rc = check_device(&dev);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (rows == 0 || cols == 0) {
    // empty tensor: both operands as the separate calls leave them
    for (int k = 0; k < 2; ++k) {
      const nvfp4_tensor* o = k ? out_col : out_row;
      const float* ain = k ? amax_col_in : amax_row_in;
      if (ain == o->amax) {
        // supplied in place: already holds the amax
      } else if (ain) {
        if (cudaMemcpyAsync(o->amax, ain, sizeof(float), cudaMemcpyDeviceToDevice, s) != cudaSuccess) return NVFP4_ERR_CUDA;
      } else if (cudaMemsetAsync(o->amax, 0, sizeof(float), s) != cudaSuccess) {
        return NVFP4_ERR_CUDA;
      }
      if (cudaMemsetAsync(o->global_scale, 0, sizeof(float), s) != cudaSuccess) return NVFP4_ERR_CUDA;
      const size_t sb = nvfp4_scales_bytes(o->rows, o->cols, o->scale_layout);
      if (sb && cudaMemsetAsync(o->scales, 0, sb, s) != cudaSuccess) return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
  }
  if (!x || !aligned16(x)) return NVFP4_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(out_row->codes) & 7u) != 0 || (reinterpret_cast<uintptr_t>(out_col->codes) & 7u) != 0)
    return NVFP4_ERR_INVALID_ARG;
  return nvfp4::quantize_dual_launch(*dev, x, rows, cols, ld, (row_flags & NVFP4_ROUND_SR) != 0, row_sr_seed, rht_seed,
                                     col_sr_seed, amax_row_in, amax_col_in, *out_row, *out_col, s);
}

int nvfp4_quantize_mxfp4(const void* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* codes, uint8_t* scales_e8m0,
                         nvfp4_stream_t stream) {
  if (rows < 0 || cols < 0 || ld < cols || cols % 32 != 0 || ld % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (rows > 0 && cols > 0 && (rows * (cols / 32)) >= (int64_t)1 << 31) return NVFP4_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  int rc = check_device(&dev);
  if (rc) return rc;
  if (rows == 0 || cols == 0) return NVFP4_OK;
  if (!x || !codes || !scales_e8m0 || !aligned16(x) || !aligned16(codes)) return NVFP4_ERR_INVALID_ARG;
  return nvfp4::quantize_mx_launch(*dev, x, rows, cols, ld, codes, scales_e8m0, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_gemm(const nvfp4_tensor* A, const nvfp4_tensor* B, void* c, int64_t ldc, nvfp4_stream_t stream) {
  return nvfp4_gemm_group(1, &A, &B, &c, &ldc, stream);
}

int nvfp4_gemm_group(int32_t count, const nvfp4_tensor* const* A, const nvfp4_tensor* const* B, void* const* c,
                     const int64_t* ldc, nvfp4_stream_t stream) {
  if (count < 1 || count > NVFP4_GEMM_GROUP_MAX || !A || !B || !c || !ldc) return NVFP4_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {
    int rc = check_gemm(A[i], B[i], c[i], ldc[i]);
    if (rc) return rc;
  }
  const DeviceInfo* dev = nullptr;
  int rc = check_device(&dev);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const nvfp4_tensor* ga[NVFP4_GEMM_GROUP_MAX];
  const nvfp4_tensor* gb[NVFP4_GEMM_GROUP_MAX];
  void* gc[NVFP4_GEMM_GROUP_MAX];
  int64_t gl[NVFP4_GEMM_GROUP_MAX];
  int n = 0;
  for (int i = 0; i < count; ++i) {
    const int64_t M = A[i]->rows, N = B[i]->rows, K = A[i]->cols;
    if (M == 0 || N == 0) continue;
    if (K == 0) {
      // empty contraction: C = 0
      if (cudaMemset2DAsync(c[i], (size_t)ldc[i] * 2, 0, (size_t)N * 2, (size_t)M, s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
      continue;
    }
    ga[n] = A[i];
    gb[n] = B[i];
    gc[n] = c[i];
    gl[n] = ldc[i];
    ++n;
  }
  if (n == 0) return NVFP4_OK;
  return nvfp4::gemm_group_launch(*dev, n, ga, gb, gc, gl, s);
}

int nvfp4_check_status(nvfp4_stream_t stream) {
  const DeviceInfo* d = nvfp4::device_info();
  if (!d) return NVFP4_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return NVFP4_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, d->status, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  if (word) {
    nvfp4::status_clear_kernel<<<1, 1, 0, s>>>(d->status, word);
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  if (word & nvfp4::kStatusTimeout) return NVFP4_ERR_TIMEOUT;
  if (word & nvfp4::kStatusNonFinite) return NVFP4_ERR_NONFINITE;
  return NVFP4_OK;
}

const char* nvfp4_status_string(int status) {
  switch (status) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument (null pointer, shape, alignment or flags)";
    case NVFP4_ERR_UNSUPPORTED: return "unsupported device (needs compute capability 10.3, sm_103a)";
    case NVFP4_ERR_CUDA: return "CUDA runtime or launch error";
    case NVFP4_ERR_TIMEOUT: return "a bounded device-side wait expired";
    case NVFP4_ERR_NONFINITE: return "input tensor holds NaN or Inf";
    default: return "unknown status";
  }
}

int nvfp4_version(void) { return 100; }

int nvfp4_selftest_wait_timeout(uint32_t limit_us, nvfp4_stream_t stream) {
  if (limit_us == 0 || limit_us > 2000000u) return NVFP4_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  int rc = check_device(&dev);
  if (rc) return rc;
  return nvfp4::selftest_wait_launch(*dev, (uint64_t)limit_us * 1000ull, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_mma_rate_probe(int32_t n_mma, int32_t mma_n, uint64_t* out, int32_t* pairs_launched,
                         nvfp4_stream_t stream) {
  if (n_mma < 1 || n_mma > (1 << 20) || (mma_n != 128 && mma_n != 256) || !out || !pairs_launched)
    return NVFP4_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(out) & 7u) != 0) return NVFP4_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  int rc = check_device(&dev);
  if (rc) return rc;
  int pairs = 0;
  rc = nvfp4::mma_rate_launch(*dev, n_mma, mma_n, reinterpret_cast<unsigned long long*>(out), &pairs,
                              reinterpret_cast<cudaStream_t>(stream));
  if (rc == NVFP4_OK) *pairs_launched = pairs;
  return rc;
}

int nvfp4_copy_rate_probe(const void* src, int64_t src_bytes, int32_t mode, int32_t ctas, int32_t iters,
                          uint64_t* out, nvfp4_stream_t stream) {
  if (!src || !out || (mode != 0 && mode != 1) || iters < 1 || iters > (1 << 20) || ctas < 1)
    return NVFP4_ERR_INVALID_ARG;
  if (src_bytes < (mode == 0 ? 16384 : 262144)) return NVFP4_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) & 15u) != 0 || (reinterpret_cast<uintptr_t>(out) & 7u) != 0)
    return NVFP4_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  int rc = check_device(&dev);
  if (rc) return rc;
  if (ctas > dev->sm_count) return NVFP4_ERR_INVALID_ARG;
  return nvfp4::copy_rate_launch(*dev, src, src_bytes, mode, ctas, iters, reinterpret_cast<unsigned long long*>(out),
                                 reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_encode_e2m1_rne(const float* v, int64_t n, uint8_t* out, nvfp4_stream_t stream) {
  if (n < 0 || (n > 0 && (!v || !out))) return NVFP4_ERR_INVALID_ARG;
  if (n == 0) return NVFP4_OK;
  const DeviceInfo* dev = nullptr;
  int rc = check_device(&dev);
  if (rc) return rc;
  return nvfp4::encode_e2m1_rne_launch(v, n, out, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_encode_e2m1_sr(const float* v, const uint16_t* u16, int64_t n, uint8_t* out, nvfp4_stream_t stream) {
  if (n < 0 || (n > 0 && (!v || !u16 || !out))) return NVFP4_ERR_INVALID_ARG;
  if (n == 0) return NVFP4_OK;
  const DeviceInfo* dev = nullptr;
  int rc = check_device(&dev);
  if (rc) return rc;
  return nvfp4::encode_e2m1_sr_launch(v, u16, n, out, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_encode_e4m3(const float* t, int64_t n, uint8_t* out, nvfp4_stream_t stream) {
  if (n < 0 || (n > 0 && (!t || !out))) return NVFP4_ERR_INVALID_ARG;
  if (n == 0) return NVFP4_OK;
  const DeviceInfo* dev = nullptr;
  int rc = check_device(&dev);
  if (rc) return rc;
  return nvfp4::encode_e4m3_launch(t, n, out, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
