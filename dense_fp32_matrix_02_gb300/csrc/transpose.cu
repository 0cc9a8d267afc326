// Out-of-place transpose of a strided batch of fp32 matrices,
// dst_b = src_bᵀ: the copy that lets Aᵀ·B run as a plain product.  It is
// HBM-bound: tiles go through shared memory (one padding column, so that
// reading a column of the tile spreads over the banks), so that both the
// reads of src and the writes of dst are whole row segments.  Where rows,
// strides and pointers allow, 64×64 tiles move as float4 (each thread
// keeps four 16-byte loads in flight); otherwise 32×32 tiles move as
// single floats.  One resident wave of 256-thread blocks walks the tiles
// grid-stride; edges are guarded.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace gemm_f32_impl {
namespace {

__global__ void __launch_bounds__(256)
    transpose_kernel(const float* __restrict__ src, long long lds,
                     long long ss, float* __restrict__ dst, long long ldd,
                     long long sd, int rows, int cols, int batch) {
  griddep_wait();  // src may belong to the kernel before
  griddep_launch_dependents();
  __shared__ float tile[32][33];
  const int tiles_c = (cols + 31) / 32;
  const long long per = (long long)((rows + 31) / 32) * tiles_c;
  const long long total = per * batch;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (long long t = blockIdx.x; t < total; t += gridDim.x) {
    const long long b = t / per;
    const int rem = (int)(t - b * per);
    const int r0 = (rem / tiles_c) * 32, c0 = (rem % tiles_c) * 32;
    const float* s = src + b * ss;
    float* d = dst + b * sd;
#pragma unroll
    for (int i = ty; i < 32; i += 8) {
      const int r = r0 + i, c = c0 + tx;
      if (r < rows && c < cols) tile[i][tx] = s[(long long)r * lds + c];
    }
    __syncthreads();
#pragma unroll
    for (int i = ty; i < 32; i += 8) {
      const int c = c0 + i, r = r0 + tx;  // dst row c, column r
      if (c < cols && r < rows) d[(long long)c * ldd + r] = tile[tx][i];
    }
    __syncthreads();
  }
}

// float4 form: cols, lds, ss multiples of 4, src and dst 16-byte aligned,
// ldd and sd multiples of 4 and ldd >= rows rounded up to 4.  dst columns
// from rows up to that rounding (row padding of dst) are written as zeros.
__global__ void __launch_bounds__(256)
    transpose4_kernel(const float* __restrict__ src, long long lds,
                      long long ss, float* __restrict__ dst, long long ldd,
                      long long sd, int rows, int cols, int batch) {
  griddep_wait();  // src may belong to the kernel before
  griddep_launch_dependents();
  __shared__ float tile[64][65];
  const int tiles_c = (cols + 63) / 64;
  const long long per = (long long)((rows + 63) / 64) * tiles_c;
  const long long total = per * batch;
  const int rows4 = (rows + 3) & ~3;
  for (long long t = blockIdx.x; t < total; t += gridDim.x) {
    const long long b = t / per;
    const int rem = (int)(t - b * per);
    const int r0 = (rem / tiles_c) * 64, c0 = (rem % tiles_c) * 64;
    const float* s = src + b * ss;
    float* d = dst + b * sd;
    float4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // row r0 + i, columns c0 + 4q .. + 3
      const int idx = threadIdx.x + 256 * j, i = idx >> 4, q = idx & 15;
      const int r = r0 + i, c = c0 + 4 * q;
      v[j] = (r < rows && c < cols)
                 ? *reinterpret_cast<const float4*>(s + (long long)r * lds + c)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int idx = threadIdx.x + 256 * j, i = idx >> 4, q = idx & 15;
      tile[i][4 * q] = v[j].x;
      tile[i][4 * q + 1] = v[j].y;
      tile[i][4 * q + 2] = v[j].z;
      tile[i][4 * q + 3] = v[j].w;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // dst row c0 + i, columns r0 + 4q .. + 3
      const int idx = threadIdx.x + 256 * j, i = idx >> 4, q = idx & 15;
      const int c = c0 + i, r = r0 + 4 * q;
      if (c < cols && r < rows4)
        *reinterpret_cast<float4*>(d + (long long)c * ldd + r) =
            make_float4(tile[4 * q][i], tile[4 * q + 1][i],
                        tile[4 * q + 2][i], tile[4 * q + 3][i]);
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_transpose(const float* src, long long lds, long long ss,
                             float* dst, long long ldd, long long sd,
                             long long rows, long long cols, long long batch,
                             int sm_count, cudaStream_t stream) {
  if (rows <= 0 || cols <= 0 || batch <= 0) return cudaSuccess;
  if (rows > 0x7fffffffLL || cols > 0x7fffffffLL || batch > 0x7fffffffLL)
    return cudaErrorInvalidValue;
  const bool vec = cols % 4 == 0 && lds % 4 == 0 && ss % 4 == 0 &&
                   ldd % 4 == 0 && sd % 4 == 0 && ldd >= ((rows + 3) & ~3LL) &&
                   (reinterpret_cast<uintptr_t>(src) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
  const int t = vec ? 64 : 32;
  const long long tiles = ((rows + t - 1) / t) * ((cols + t - 1) / t) * batch;
  const long long wave = 8LL * (sm_count > 0 ? sm_count : 1);
  const int grid = (int)(tiles < wave ? tiles : wave);
  if (vec)
    return launch_pdl(transpose4_kernel, dim3(grid), dim3(256), 0, stream,
                      src, lds, ss, dst, ldd, sd, (int)rows, (int)cols,
                      (int)batch);
  return launch_pdl(transpose_kernel, dim3(grid), dim3(256), 0, stream, src,
                    lds, ss, dst, ldd, sd, (int)rows, (int)cols, (int)batch);
}

}  // namespace gemm_f32_impl
