// gemm_f32_host: C = A·B for matrices in host memory, with the copies to and
// from the GPU overlapped with the multiply (see include/gemm_f32.h).
//
// Schedule on one device, for P row chunks of A and C (the first and last
// small when M is large, see chunk_bounds):
//   copy-in stream   B (whole) | A_0 | A_1 | ... | A_{P-1}
//   caller's stream          wait B, A_c -> C_c = A_c·B   (one gemm per chunk)
//   copy-out stream                        wait C_c -> C_c to the host
// and the caller's stream finally waits for the last copy out, so the call
// is complete when `stream` is.  The two copy streams and the events are
// created once per device and kept; no device memory is allocated.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "gemm_f32.h"
#include "kernels.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 16;

struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start, b_ready, a_ready[kMaxChunks], c_ready[kMaxChunks],
      done;
};

std::mutex g_pipe_mu;
HostPipe g_pipes[kMaxDevices];

cudaError_t pipe_for_current_device(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  HostPipe& p = g_pipes[dev];
  if (!p.ready) {
    if ((e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking)) !=
        cudaSuccess)
      return e;
    if ((e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking)) !=
        cudaSuccess)
      return e;
    cudaEvent_t* all[] = {&p.start, &p.b_ready, &p.done};
    for (cudaEvent_t* ev : all)
      if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) !=
          cudaSuccess)
        return e;
    for (int c = 0; c < kMaxChunks; ++c) {
      if ((e = cudaEventCreateWithFlags(&p.a_ready[c],
                                        cudaEventDisableTiming)) != cudaSuccess)
        return e;
      if ((e = cudaEventCreateWithFlags(&p.c_ready[c],
                                        cudaEventDisableTiming)) != cudaSuccess)
        return e;
    }
    p.ready = true;
  }
  *out = &p;
  return cudaSuccess;
}

// Row chunks: enough to overlap copies with the multiply, few enough that
// every chunk still fills the GPU with tiles.
int chunk_count(int64_t M, int64_t N) {
  const int64_t tiles_per_row_block = (N + 127) / 128;  // tiles per 128 rows
  int p = 4;
  while (p > 1 && ((M + p - 1) / p + 127) / 128 * tiles_per_row_block < 256)
    --p;
  return (int)std::max<int64_t>(1, std::min<int64_t>(p, M));
}

// First row of each chunk (bounds[c] .. bounds[c+1]); returns the count.
// The pipeline's ends are serial: nothing is multiplied before B and the
// first A chunk are in, and the last chunk's product and copy back follow
// everything else.  So when M holds at least two waves of 128-row tiles
// (a wave: two CTAs per SM), the first and last chunks are half a wave and
// the chunks between at most one wave each, so that no chunk leaves a
// nearly empty round of tiles behind; otherwise up to four chunks of
// equal whole 128-row tiles (the last one shorter) that each still fill
// the GPU, so every chunk starts on a tile row and its A and C rows keep
// the 16-byte alignment of the whole matrices.
int chunk_bounds(int64_t M, int64_t N, int sm_count, int64_t* bounds) {
  const int64_t tiles_per_rb = (N + 127) / 128;  // tiles per 128 rows
  const int64_t rbs = (M + 127) / 128;
  const int64_t wave_rb =
      std::max<int64_t>(1, 2 * (int64_t)sm_count / tiles_per_rb);
  if (rbs >= 2 * wave_rb && wave_rb >= 2) {
    const int64_t edge = wave_rb / 2;
    const int64_t rest = rbs - 2 * edge;
    int64_t n_mid = (rest + wave_rb - 1) / wave_rb;
    n_mid = std::min<int64_t>(n_mid, kMaxChunks - 2);
    const int64_t mid = (rest + n_mid - 1) / n_mid;
    int n = 0;
    int64_t rb = 0;
    bounds[n++] = 0;
    rb += edge;
    bounds[n++] = rb * 128;
    for (int64_t c = 0; c < n_mid; ++c) {
      rb = std::min<int64_t>(rb + mid, rbs - edge);
      if (rb * 128 > bounds[n - 1]) bounds[n++] = rb * 128;
    }
    bounds[n] = M;  // the last chunk: the final edge rows
    return n;
  }
  const int chunks = chunk_count(M, N);
  const int64_t rows = ((M + chunks - 1) / chunks + 127) / 128 * 128;
  int n = 0;
  for (int c = 0; c < chunks; ++c) {
    const int64_t r0 = c * rows;
    if (r0 >= M) break;
    bounds[n++] = r0;
  }
  bounds[n] = M;
  return n;
}

// rows × cols floats between a host matrix (row stride ld) and a dense
// device block; one linear copy when the host rows are contiguous.
cudaError_t copy_rows(float* dst, int64_t dst_ld, const float* src,
                      int64_t src_ld, int64_t rows, int64_t cols,
                      cudaMemcpyKind kind, cudaStream_t s) {
  if (dst_ld == cols && src_ld == cols)
    return cudaMemcpyAsync(dst, src, rows * cols * 4, kind, s);
  return cudaMemcpy2DAsync(dst, dst_ld * 4, src, src_ld * 4, cols * 4, rows,
                           kind, s);
}

}  // namespace

extern "C" {

int gemm_f32_host_chunks(int64_t M, int64_t N, int sm_count,
                         int64_t bounds[17]) {
  if (M < 1 || N < 1 || sm_count < 1 || !bounds)
    return -GEMM_F32_ERR_INVALID_ARG;
  return chunk_bounds(M, N, sm_count, bounds);
}

int gemm_f32_host(int64_t M, int64_t N, int64_t K, const float* hA,
                  int64_t lda, const float* hB, int64_t ldb, float* hC,
                  int64_t ldc, float* dA, float* dB, float* dC,
                  void* workspace, int64_t workspace_bytes,
                  gemm_f32_stream_t stream) {
  if (M < 0 || N < 0 || K < 0 || lda < K || ldb < N || ldc < N)
    return GEMM_F32_ERR_INVALID_ARG;
  if (workspace_bytes < 0 || (workspace_bytes > 0 && !workspace))
    return GEMM_F32_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_F32_OK;
  if (!hC || !dC || (K > 0 && (!hA || !hB || !dA || !dB)))
    return GEMM_F32_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe* pp = nullptr;
  cudaError_t e = pipe_for_current_device(&pp);
  if (e != cudaSuccess) return gemm_f32_impl::record_cuda_error(e);
  HostPipe& p = *pp;

  // everything starts after the work already queued on the caller's stream
  if ((e = cudaEventRecord(p.start, s)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(p.in, p.start, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(p.out, p.start, 0)) != cudaSuccess)
    return gemm_f32_impl::record_cuda_error(e);

  if (K > 0) {
    if ((e = copy_rows(dB, N, hB, ldb, K, N, cudaMemcpyHostToDevice,
                       p.in)) != cudaSuccess ||
        (e = cudaEventRecord(p.b_ready, p.in)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s, p.b_ready, 0)) != cudaSuccess)
      return gemm_f32_impl::record_cuda_error(e);
  }
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount,
                                  dev)) != cudaSuccess)
    return gemm_f32_impl::record_cuda_error(e);
  int64_t bounds[kMaxChunks + 1];
  const int chunks = chunk_bounds(M, N, sms, bounds);
  for (int c = 0; c < chunks; ++c) {
    const int64_t r0 = bounds[c], r1 = bounds[c + 1];
    if (r0 >= r1) continue;
    if (K > 0) {
      if ((e = copy_rows(dA + r0 * K, K, hA + r0 * lda, lda, r1 - r0, K,
                         cudaMemcpyHostToDevice, p.in)) != cudaSuccess ||
          (e = cudaEventRecord(p.a_ready[c], p.in)) != cudaSuccess ||
          (e = cudaStreamWaitEvent(s, p.a_ready[c], 0)) != cudaSuccess)
        return gemm_f32_impl::record_cuda_error(e);
    }
    const int st = gemm_f32_impl::run_auto_with_scratch(
        r1 - r0, N, K, dA + r0 * K, K, dB, N, dC + r0 * N, N, workspace,
        workspace_bytes, stream);
    if (st != GEMM_F32_OK) return st;
    if ((e = cudaEventRecord(p.c_ready[c], s)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(p.out, p.c_ready[c], 0)) != cudaSuccess ||
        (e = copy_rows(hC + r0 * ldc, ldc, dC + r0 * N, N, r1 - r0, N,
                       cudaMemcpyDeviceToHost, p.out)) != cudaSuccess)
      return gemm_f32_impl::record_cuda_error(e);
  }
  if ((e = cudaEventRecord(p.done, p.out)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(s, p.done, 0)) != cudaSuccess)
    return gemm_f32_impl::record_cuda_error(e);
  return GEMM_F32_OK;
}

}  // extern "C"
