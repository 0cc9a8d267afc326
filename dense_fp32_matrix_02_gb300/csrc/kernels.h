// Internal interface between the C-ABI dispatcher (gemm_f32_api.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "common.cuh"
#include "gemm_f32.h"

namespace gemm_f32_impl {

// Launches `kernel` with programmatic stream serialization: its CTAs may be
// scheduled while the previous kernel in the stream finishes; the kernel
// calls griddep_wait before it touches global memory.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block,
                       size_t smem, cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same with thread-block clusters of `cluster_x` consecutive CTAs
// (along x).
template <typename... Params, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(Params...), dim3 grid,
                               dim3 block, size_t smem, cudaStream_t stream,
                               unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// SIMT tile configurations (BM x BN x BK).  "Occ1" variants let a thread
// use up to 255 registers at one 256-thread CTA per SM; the 128 x 64 and
// 64 x 64 tiles run 128-thread CTAs, three and four per SM.  Every one
// compiles without register spills (128 x 128 tiles at two CTAs per SM,
// capped at 128 registers a thread, spilled and are not offered).
enum SimtCfg {
  kSimt128x64x16 = 0,
  kSimt64x64x16 = 1,
  kSimt128x128x16Occ1 = 2,
  kSimt128x128x32Occ1 = 3,
  kSimt128x128x16Occ1S6 = 4,
  kSimtKm128x128x32Occ1 = 5,  // A kept K-major (16-byte copies)
  // warp-specialised: a ninth warp issues every copy (16-byte operands
  // only; otherwise the same as kSimt128x128x32Occ1)
  kSimtWs128x128x32 = 6,
  kSimtCfgCount = 7
};

// The driver's cuTensorMapEncodeTiled, looked up once (thread-safe); null
// if the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Sets cudaFuncAttributeMaxDynamicSharedMemorySize for `fn` on the current
// device once (a launch asking for more than 48 KB fails without it).
cudaError_t ensure_smem_attr(const void* fn, int bytes);

cudaError_t launch_simt(const Problem& p, int cfg, bool vec, bool c_vec,
                        const WaitCfg& wc,
                        cudaStream_t stream);

// 3xTF32 tcgen05 kernel configurations: 256 x 128 tiles at one CTA per SM,
// or 128 x 128 tiles at two; "Raw" variants let the tensor core truncate the
// raw fp32 operands to TF32 for the big part instead of rounding them first.
enum TcCfg {
  kTc256 = 0,
  kTc128 = 1,
  kTc128Raw = 2,
  kTc256Raw = 3,
  kTcCfgCount = 4
};

int tf32x3_tile_m(int cfg);

// Bytes of the partial tiles a launch that splits `split_tiles` tiles of
// tile_m × 128 over `splits` > 1 CTAs each writes (and the reduction reads).
long long tf32x3_partials_bytes(int tile_m, long long split_tiles,
                                int splits);

// 3xTF32 tcgen05 kernel.  Needs A, B 16-byte aligned, lda and ldb multiples
// of 4, K >= 1 and an sm_100-family device.  Batched problems (p.batch > 1,
// strides multiples of 4 and either 0 or at least one whole matrix) and,
// with configuration kTc128Raw or kTc256Raw, one of p.transB (B stored
// N×K), p.transA (A stored K×M; always 128-row tiles) or p.storeT (C stored
// transposed: the caller swapped the operands, op(A)ᵀ·op(B)ᵀ computed as
// B·A).  With splits > 1 and a
// `partials` buffer of tf32x3_partials_bytes for the tiles past the first
// full_tiles (grouped order), each of those tiles' K range is split over
// `splits` CTAs and a second kernel sums the partial tiles into C in split
// order (deterministic); full_tiles = 0 splits every tile.  With `cluster`
// (full_tiles = 0, 2 <= splits <= kMaxClusterSplits, no buffer needed) the
// splits of a tile form a thread-block cluster instead and add their
// partial tiles through distributed shared memory, in the same split order
// (bit-identical results), with no second kernel.  splits is reduced so no
// split is empty.  Single products only.
constexpr int kMaxClusterSplits = 8;  // the portable cluster size
cudaError_t launch_tf32x3(const Problem& p, int cfg, int full_tiles,
                          int splits, float* partials, bool cluster,
                          const WaitCfg& wc, cudaStream_t stream);

// Whether the streaming 3xTF32 kernel takes an N × K B (N <= 128,
// K <= 128: B lives in TMEM).
bool tf32x3_stream_fits(long long N, long long K);

// Persistent 3xTF32 kernel for narrow, shallow B and many rows: single
// plain products (no batch, transposes or split-K), A and B 16-byte aligned
// with lda and ldb multiples of 4; C any alignment (TMA stores when it is
// 16-byte aligned with ldc a multiple of 4); fused bias / GELU.
cudaError_t launch_tf32x3_stream(const Problem& p, int sm_count,
                                 const WaitCfg& wc, cudaStream_t stream);

// Scratch bytes the automatic plan wants for these arguments on the current
// device (0 = none), or minus a gemm_f32_status.
long long auto_plan_scratch_bytes(int64_t M, int64_t N, int64_t K,
                                  const float* A, int64_t lda, const float* B,
                                  int64_t ldb, const float* C, int64_t ldc);

// FFMA kernel fed by TMA under mbarrier phases (128x128x32 tiles, 4
// stages).  Needs A, B 16-byte aligned, lda and ldb multiples of 4, K >= 1.
cudaError_t launch_tma_ffma(const Problem& p, bool c_vec, const WaitCfg& wc,
                            cudaStream_t stream);

// Records a CUDA error for gemm_f32_last_cuda_error; returns
// GEMM_F32_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// gemm_f32_ws's path: automatic plan with the given scratch.
int run_auto_with_scratch(int64_t M, int64_t N, int64_t K, const float* A,
                          int64_t lda, const float* B, int64_t ldb, float* C,
                          int64_t ldc, void* scratch, int64_t scratch_bytes,
                          gemm_f32_stream_t stream);

// One mixed-precision product: 16-bit A (M×K) and B (K×N), row-major.
struct Problem16 {
  int M, N, K;
  int type;  // gemm_f32_mixed_type
  const void* A;
  long long lda;
  const void* B;
  long long ldb;
  float* C;
  long long ldc;
};

// How the 16-bit kernel cuts C into work units, one per CTA at a time:
// tiles of 128 rows by `wn` columns (256, or 128 / 64 when N is that
// narrow, so no MMA computes columns that all lie past N), walked in the
// grouped order; the first `full` tiles whole, in whole rounds of the
// grid, and each tile of the last, partly filled round (every tile, when
// there are fewer tiles than SMs) cut into `parts` strips of wn / parts
// columns, so that the last round spreads over the GPU instead of leaving
// most SMs idle while one tile per busy SM runs its whole length.
struct Plan16 {
  int bm;  // rows per tile: 128, or 256 (two MMAs of M = 128 per k-step)
  int wn;
  long long tiles_m, tiles_n;
  long long full;  // whole tiles; the rest are split
  int parts;       // strips per split tile: 1, 2 or 4
  long long units;
  int grid;        // persistent CTAs: min(units, sm_count)
};

// narrow = false keeps every tile whole and 256 wide.
Plan16 plan_mixed16(long long M, long long N, int sm_count, bool narrow,
                    int bm = 128);

// tcgen05 kind::f16 kernel, persistent over plan.grid CTAs.
// Needs A, B 16-byte aligned, lda and ldb multiples of 8, K >= 1.
cudaError_t launch_mixed16(const Problem16& p, const Plan16& plan, bool c_vec,
                           const WaitCfg& wc, cudaStream_t stream);

// dst = round16(src) (type gemm_f32_mixed_type) for a rows×cols block.
cudaError_t launch_round16(int type, long long rows, long long cols,
                           const float* src, long long lds, uint16_t* dst,
                           long long ldd, int sm_count, cudaStream_t stream);

// dst_b = src_bᵀ for b < batch: src_b = src + b·ss is rows×cols (row
// stride lds), dst_b = dst + b·sd is cols×rows (row stride ldd).
cudaError_t launch_transpose(const float* src, long long lds, long long ss,
                             float* dst, long long ldd, long long sd,
                             long long rows, long long cols, long long batch,
                             int sm_count, cudaStream_t stream);

// C[0:M, 0:N] = 0.
cudaError_t launch_fill_zero(float* C, long long ldc, long long M, long long N,
                             int sm_count, cudaStream_t stream);

}  // namespace gemm_f32_impl
