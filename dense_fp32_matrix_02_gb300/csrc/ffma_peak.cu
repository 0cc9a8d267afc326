// FP32 FMA throughput probe: the measured denominator of the FFMA-bound
// kernels' roofline.  "3 · La mémoire partagée" bounds the tiled product by
// the FP32 FMA pipe once shared-memory reuse removes the memory bound; this
// kernel runs nothing but independent FMA chains on every SM so the pipe's
// achievable rate on this GPU, at its clocks, can be timed.
//
// Each thread keeps kChains independent accumulators and applies
// a <- a·s + t to each, kUnroll times per loop iteration, so every warp has
// kChains FMAs in flight per dependency step.  s and t keep the values in
// [1/2, 2] (no overflow, no subnormals).  A result that no input can produce
// guards the only store, so the compiler keeps every FMA.
#include <cuda_runtime.h>

#include "gemm_f32.h"
#include "kernels.h"

namespace gemm_f32_impl {
namespace {

constexpr int kChains = 8;
constexpr int kUnroll = 16;
constexpr int kThreads = 256;
constexpr int kBlocksPerSm = 8;  // 2048 threads: full residency

__global__ void __launch_bounds__(kThreads)
    ffma_peak_kernel(long long iters, float s, float t, float* sink) {
  float a[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c)
    a[c] = 1.0f + 0.0625f * (float)((threadIdx.x + c) & 7);
#pragma unroll 1
  for (long long i = 0; i < iters; ++i) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int c = 0; c < kChains; ++c) a[c] = fmaf(a[c], s, t);
  }
  float sum = 0.f;
#pragma unroll
  for (int c = 0; c < kChains; ++c) sum += a[c];
  if (sum == -1.0f) sink[threadIdx.x] = sum;  // never true for s, t > 0
}

}  // namespace
}  // namespace gemm_f32_impl

extern "C" {

int64_t gemm_f32_ffma_peak_flops(int64_t iters) {
  int dev = 0, sms = 0;
  if (iters < 0 || cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
          cudaSuccess)
    return -GEMM_F32_ERR_INVALID_ARG;
  using namespace gemm_f32_impl;
  return 2LL * kChains * kUnroll * iters * kThreads * kBlocksPerSm * sms;
}

int gemm_f32_ffma_peak_launch(int64_t iters, float* sink,
                              gemm_f32_stream_t stream) {
  using namespace gemm_f32_impl;
  if (iters < 0 || !sink) return GEMM_F32_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return record_cuda_error(e);
  // fixed point of a <- a·s + t is t / (1 - s) = 1
  ffma_peak_kernel<<<sms * kBlocksPerSm, kThreads, 0,
                     reinterpret_cast<cudaStream_t>(stream)>>>(
      iters, 0.999f, 0.001f, sink);
  e = cudaGetLastError();
  return e == cudaSuccess ? GEMM_F32_OK : record_cuda_error(e);
}

}  // extern "C"
