// FP32 GEMM on the FFMA pipe, operands staged by TMA under mbarrier phases.
//
// The same 8×8 register outer product as the cp.async kernel ("3 · La
// mémoire partagée", §3.4), with A kept K-major (FfmaTile).  The two
// __syncthreads of the page's tiled loop (§3.2-§3.3) become a pair of
// mbarrier phases per ring slot:
//   full[s]   completes when TMA has written stage s (transaction bytes);
//             every warp waits on it before reading the stage;
//   empty[s]  completes when all eight warps have finished reading stage s
//             (one arrival per warp); the copy of the stage STAGES ahead may
//             only then overwrite the slot.
// Thread 0 issues the copies: before computing stage kt it waits for
// empty[] of the slot read at kt−1 and loads stage kt+STAGES−1 into it.
// TMA writes A (BK = 32 fp32 = 128-byte rows) in the 128-byte swizzle that
// FfmaTile reads and B (BK × 128) unswizzled; copies that fall past M, N or
// K are zero-filled by TMA, and the epilogue guards the stores.  Every wait
// is bounded by a %globaltimer deadline that sets the status word; a CTA
// that gives up waits for its copies in flight and ends without storing.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "ffma_tile.cuh"
#include "kernels.h"

namespace gemm_f32_impl {
namespace tma_ffma {

constexpr int kBM = 128, kBN = 128;
constexpr int kThreads = FfmaTile<kBM, kBN, 32>::kThreads;  // 256: 8 warps
constexpr long long kDrainNs = 2000000000LL;

// BK = 32 (128-byte A rows, 128-byte swizzle) or 16 (64-byte, 64-byte).
template <int BK, int STAGES>
struct TCfg {
  static constexpr int kBK = BK;
  static constexpr int kStages = STAGES;
  using Tile = FfmaTile<kBM, kBN, BK>;
  static constexpr int kStageBytesA = kBM * BK * 4;
  static constexpr int kStageBytesB = BK * kBN * 4;
  static constexpr int kOffB = STAGES * kStageBytesA;
  static constexpr int kOffBar = kOffB + STAGES * kStageBytesB;
  static constexpr int kSmemBytes = kOffBar + 2 * STAGES * 8 + 16 + 1024;
};

// Bounded wait (polling); false when `limit_ns` passes or the CTA abort
// flag is set.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity,
                                           long long limit_ns,
                                           volatile int* abort) {
  return bounded_wait(bar, parity, limit_ns, abort, 0u);
}

template <class Cf>
__global__ void __launch_bounds__(kThreads, 1)
    tma_ffma_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b, Problem p,
                    int tiles_m, int tiles_n, int c_vec, WaitCfg wc) {
  griddep_wait();  // A, B and C may belong to the kernel before
  constexpr int kBK = Cf::kBK, kStages = Cf::kStages;
  constexpr int kStageBytesA = Cf::kStageBytesA;
  constexpr int kStageBytesB = Cf::kStageBytesB;
  constexpr int kOffB = Cf::kOffB, kOffBar = Cf::kOffBar;
  using Tile = typename Cf::Tile;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  volatile int* abort = reinterpret_cast<volatile int*>(bars + 2 * kStages);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[kStages + s]); };

  const int tid = threadIdx.x, lane = tid & 31;
  int tm, tn;
  tile_coords<8>(blockIdx.x, tiles_m, tiles_n, tm, tn);
  const int bm = tm * kBM, bn = tn * kBN;
  const int nk = (p.K + kBK - 1) / kBK;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kThreads / 32);
    }
    *abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
  }
  __syncthreads();

  int issued = 0;  // copies issued by thread 0
  auto issue = [&](int kt) {
    const int s = kt % kStages;
    mbar_arrive_expect_tx(full(s), kStageBytesA + kStageBytesB);
    tma_load_2d(sbase + s * kStageBytesA, &tmap_a, full(s), kt * kBK, bm);
    tma_load_2d(sbase + kOffB + s * kStageBytesB, &tmap_b, full(s), bn,
                kt * kBK);
    ++issued;
  };
  if (tid == 0 && !(wc.debug & kDebugStallProducer)) {
    for (int kt = 0; kt < kStages - 1 && kt < nk; ++kt) issue(kt);
  }

  Tile tile;
  tile.init(tid);
  typename Tile::Acc acc;
  Tile::zero(acc);

  bool ok = true;
  for (int kt = 0; kt < nk; ++kt) {
    const int s = kt % kStages;
    if (tid == 0 && !(wc.debug & kDebugStallProducer)) {
      const int next = kt + kStages - 1;
      if (next < nk) {
        // the slot `next` lands in was last read at kt - 1
        if (kt >= 1 && !wait_phase(empty((kt - 1) % kStages),
                                   ((kt - 1) / kStages) & 1, wc.limit,
                                   abort)) {
          *abort = 1;
          record_status(wc.status, kStatusTimeoutEmpty);
        } else {
          issue(next);
        }
      }
    }
    if (!wait_phase(full(s), (kt / kStages) & 1, wc.limit, abort)) {
      *abort = 1;
      record_status(wc.status, kStatusTimeoutFull);
      ok = false;
      break;
    }
    tile.compute(reinterpret_cast<const float*>(smem + s * kStageBytesA),
                 reinterpret_cast<const float*>(smem + kOffB +
                                                s * kStageBytesB),
                 acc, p.status);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
  }
  if (tid == 0 && *abort) {  // let the copies still in flight land
    for (int kt = issued > kStages ? issued - kStages : 0; kt < issued; ++kt)
      if (!wait_phase(full(kt % kStages), (kt / kStages) & 1, kDrainNs,
                      nullptr))
        record_status(wc.status, kStatusTimeoutDrain);
  }
  __syncwarp();  // warp 0 reconverges after thread 0's drain
  __syncthreads();
  if (ok && !*abort) tile.store(p, bm, bn, c_vec != 0, acc);
}

}  // namespace tma_ffma

namespace {

template <class Cf>
cudaError_t launch_cfg(const Problem& p, bool c_vec, const WaitCfg& wc,
                       cudaStream_t stream) {
  using namespace tma_ffma;
  const auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap ta, tb;
  const cuuint32_t estr[2] = {1, 1};
  {
    const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)p.lda * 4};
    const cuuint32_t box[2] = {(cuuint32_t)Cf::kBK, (cuuint32_t)kBM};
    if (encode(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
               const_cast<float*>(p.A), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE,
               Cf::kBK == 32 ? CU_TENSOR_MAP_SWIZZLE_128B
                             : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)p.K};
    const cuuint64_t strides[1] = {(cuuint64_t)p.ldb * 4};
    const cuuint32_t box[2] = {(cuuint32_t)kBN, (cuuint32_t)Cf::kBK};
    if (encode(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
               const_cast<float*>(p.B), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto fn = tma_ffma_kernel<Cf>;
  cudaError_t e =
      ensure_smem_attr(reinterpret_cast<const void*>(fn), Cf::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int tiles_m = (p.M + kBM - 1) / kBM, tiles_n = (p.N + kBN - 1) / kBN;
  const long long grid = (long long)tiles_m * tiles_n;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(fn, dim3((unsigned)grid), dim3(kThreads), Cf::kSmemBytes,
                    stream, ta, tb, p, tiles_m, tiles_n, c_vec ? 1 : 0, wc);
}

}  // namespace

// 128x128 tiles, BK = 32, 4 stages: measured best at 4096^3 among BK 16/32
// and 4-8 stages.
cudaError_t launch_tma_ffma(const Problem& p, bool c_vec, const WaitCfg& wc,
                            cudaStream_t stream) {
  return launch_cfg<tma_ffma::TCfg<32, 4>>(p, c_vec, wc, stream);
}

}  // namespace gemm_f32_impl
