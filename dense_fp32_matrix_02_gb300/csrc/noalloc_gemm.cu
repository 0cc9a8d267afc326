// gemm_f32_noalloc: the split-K product with its scratch in a static device
// array owned by the library, for callers that must not allocate device
// memory (see include/gemm_f32.h).  No cudaMalloc, cudaFree or allocating
// library routine runs on this path.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "gemm_f32.h"
#include "kernels.h"

namespace {

constexpr int64_t kScratchBytes = 16ll << 20;  // 16 MiB per device
constexpr int kMaxDevices = 64;

// The scratch itself.  Each GPU that loads the library holds it until the
// process exits.  Host code must not use this name as an address: it is a
// host-side stand-in; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) float g_noalloc_scratch[kScratchBytes / 4];

std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices];  // device address, per device
bool g_scratch_ready[kMaxDevices];

// Device address of the scratch on the current device, looked up once per
// device with that device current.
int scratch_on_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return GEMM_F32_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GEMM_F32_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ready[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) return GEMM_F32_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<float*>(ptr);
    g_scratch_ready[dev] = true;
  }
  *out = g_scratch_ptr[dev];
  return GEMM_F32_OK;
}

}  // namespace

extern "C" {

int gemm_f32_noalloc(int64_t M, int64_t N, int64_t K, const float* A,
                     int64_t lda, const float* B, int64_t ldb, float* C,
                     int64_t ldc, gemm_f32_stream_t stream) {
  const long long need = gemm_f32_impl::auto_plan_scratch_bytes(
      M, N, K, A, lda, B, ldb, C, ldc);
  if (need < 0) return static_cast<int>(-need);
  if (need > kScratchBytes) return GEMM_F32_ERR_SCRATCH_LIMIT;
  float* scratch = nullptr;
  if (need > 0) {
    const int st = scratch_on_current_device(&scratch);
    if (st != GEMM_F32_OK) return st;
  }
  return gemm_f32_impl::run_auto_with_scratch(
      M, N, K, A, lda, B, ldb, C, ldc, scratch, need > 0 ? kScratchBytes : 0,
      stream);
}

int64_t gemm_f32_noalloc_scratch_bytes(void) { return kScratchBytes; }

}  // extern "C"
