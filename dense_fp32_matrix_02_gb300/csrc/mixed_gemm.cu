// Mixed-precision matrix product on the 5th-generation tensor cores:
// C (fp32) = A·B with A and B 16-bit floats (bfloat16 or IEEE binary16)
// and fp32 accumulation: the arithmetic of "Rendre le GPU rapide", "Les
// Tensor Cores" (only the operands are 16-bit; sums and tensors stay fp32).
//
// One persistent CTA per SM walks the work units: 128-row output tiles
// 256 columns wide (128 or 64 when N is that narrow), and, in the last,
// partly filled round, strips of 128 or 64 columns cut from its tiles
// (Plan16).  The walk is grid-stride over a grouped tile order, so CTAs
// running at the same time share A row-panels and B column-panels in L2:
//   warp 0      TMA producer.  Per k-block of 64: the A tile (128 rows of
//               64 k, K-major, 128-byte swizzle) and the unit's B columns
//               (64 k rows of up to 256 n, N-major, as 64×64 boxes,
//               128-byte swizzle) into a 4-stage ring.
//   warp 1      MMA issuer.  Four tcgen05.mma kind::f16 (M 128, N = the
//               unit's width, K 16) per stage into one of two TMEM
//               accumulators of 256 columns; tcgen05.commit releases the
//               stage and, after the last k-block, publishes the
//               accumulator.
//   warps 2-9   Epilogue.  tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32·(w mod 4) + 0..31, i.e. those rows of the tile, and
//               one half of the unit's columns, 32 columns at a time).  Each 32×32
//               block goes through a 4 KB shared-memory staging buffer of the
//               warp (128-byte swizzle) and out by a TMA bulk tensor store,
//               which writes whole 128-byte row segments and skips what lies
//               past M or N.  The accumulator is released once read, so the
//               tile after next accumulates into it while this one is still
//               being written; storing one tile overlaps the MMAs of the
//               next.  Where C cannot be described by a tensor map (not
//               16-byte aligned, or ldc not a multiple of 4) each lane
//               stores its row directly instead.
// Launched with programmatic stream serialization (the prologue overlaps
// the end of the kernel before it; griddepcontrol.wait precedes every
// global access).
// Every mbarrier wait is bounded by %globaltimer.  A CTA that gives up sets
// the status word, lets its copies and MMAs in flight land, frees TMEM and
// returns without storing further tiles.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "kernels.h"
#include "tcgen05.cuh"

namespace gemm_f32_impl {
namespace mixed16 {

constexpr int kBN = 256, kBK = 64;  // kBK: 128-byte rows
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;  // 320
constexpr int kBoxBytesB = 64 * kBK * 2;       // 8 KB: 64 n × 64 k
constexpr int kStageBytesB = kBN * kBK * 2;    // 32 KB
constexpr int kStagingBytes = 32 * 32 * 4;     // one warp's 32×32 fp32 block
constexpr int kTmemCols = 512;                 // the whole TMEM
constexpr long long kDrainNs = 2000000000LL;
constexpr uint32_t kSleepNs = 100000;

// Tile rows BM: 128 (4 stages of 48 KB; two 128 × 256 accumulators, so
// one tile accumulates while the other is stored) or 256 (3 stages of
// 64 KB; two MMAs of M = 128 per k-step into the halves of one 256 × 256
// accumulator that fills TMEM: each B stage feeds twice the MMAs).
template <int BM>
struct Shape {
  static constexpr int kBM = BM;
  static constexpr int kStages = BM == 128 ? 4 : 3;
  static constexpr int kStageBytesA = BM * kBK * 2;  // 16 or 32 KB
  static constexpr int kOffB = kStages * kStageBytesA;
  static constexpr int kOffStaging = kOffB + kStages * kStageBytesB;
  static constexpr int kOffCtl = kOffStaging + kEpiWarps * kStagingBytes;
  static constexpr int kHalves = BM / 128;         // M = 128 MMAs per k-step
  static constexpr int kBufs = BM == 128 ? 2 : 1;  // accumulators
  static constexpr int kAccCols = 256 * kHalves;   // TMEM columns of one
  struct __align__(8) Control {
    uint64_t full[kStages];   // TMA -> MMA (transaction bytes)
    uint64_t empty[kStages];  // MMA completion -> producer
    uint64_t acc_full[2];     // last MMA of a tile -> epilogue
    uint64_t acc_empty[2];    // epilogue warps -> MMA (one arrival per warp)
    uint64_t mma_done;        // every MMA issued has completed
    uint32_t tmem_base;
    int abort;
  };
  static constexpr int kSmemBytes = kOffCtl + (int)sizeof(Control) + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kBufs * kAccCols <= kTmemCols, "TMEM budget");
};

// sleep: the epilogue warps, idle while a tile accumulates; the producer
// and the MMA issuer poll.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity,
                                           long long limit_ns,
                                           volatile int* abort, bool sleep) {
  return bounded_wait(bar, parity, limit_ns, abort, sleep ? kSleepNs : 0u);
}

// Work unit u of a Plan16: tile row tm, first column n0, width columns.
struct Unit {
  int tm, n0, width;
};

__device__ __forceinline__ Unit unit_of(int u, int tiles_m, int tiles_n,
                                        int wn, int full, int parts) {
  int t = u, part = 0, width = wn;
  if (u >= full) {
    const int v = u - full;
    t = full + v / parts;
    part = v - (v / parts) * parts;
    width = wn / parts;
  }
  int tm, tn;
  tile_coords<8>(t, tiles_m, tiles_n, tm, tn);
  return Unit{tm, tn * wn + part * width, width};
}

// ab_type: 0 binary16, 1 bfloat16 (the kind::f16 operand format code).
template <int AB_TYPE, int BM>
__global__ void __launch_bounds__(kThreads, 1)
    mixed16_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b,
                   const __grid_constant__ CUtensorMap tmap_c, float* C,
                   long long ldc, int M, int N, int K, int tiles_m,
                   int tiles_n, int wn, int whole, int parts, int units,
                   int c_mode, WaitCfg wc) {
  // c_mode: 2 = TMA stores through staging, 1 = direct 16-byte stores,
  // 0 = direct scalar stores
  using Sh = Shape<BM>;
  constexpr int kBM = Sh::kBM, kStages = Sh::kStages;
  constexpr int kStageBytesA = Sh::kStageBytesA, kOffB = Sh::kOffB;
  constexpr int kOffStaging = Sh::kOffStaging, kOffCtl = Sh::kOffCtl;
  constexpr int kHalves = Sh::kHalves, kBufs = Sh::kBufs;
  constexpr int kAccCols = Sh::kAccCols;
  using Control = typename Sh::Control;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  Control* ctl = reinterpret_cast<Control*>(smem + kOffCtl);
  volatile int* abort = &ctl->abort;
  auto full = [&](int s) { return smem_u32(&ctl->full[s]); };
  auto empty = [&](int s) { return smem_u32(&ctl->empty[s]); };
  auto acc_full = [&](int b) { return smem_u32(&ctl->acc_full[b]); };
  auto acc_empty = [&](int b) { return smem_u32(&ctl->acc_empty[b]); };
  const uint32_t mma_done = smem_u32(&ctl->mma_done);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (K + kBK - 1) / kBK;  // >= 1 (host)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < kBufs; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), kEpiWarps);
    }
    mbar_init(mma_done, 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
    if (c_mode == 2) prefetch_tmap(&tmap_c);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;
  griddep_wait();  // A, B and C may belong to the kernel before

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;  // k-blocks issued, over all tiles of this CTA
      if (!(wc.debug & kDebugStallProducer)) {
        for (int u = blockIdx.x; u < units && !*abort; u += gridDim.x) {
          const Unit w = unit_of(u, tiles_m, tiles_n, wn, whole, parts);
          const int boxes = w.width / 64;
          for (int kb = 0; kb < nk; ++kb) {
            const int s = it % kStages;
            if (it >= kStages &&
                !wait_phase(empty(s), ((it / kStages) - 1) & 1, wc.limit,
                            abort, false)) {
              *abort = 1;
              record_status(wc.status, kStatusTimeoutEmpty);
              break;
            }
            mbar_arrive_expect_tx(full(s),
                                  kStageBytesA + boxes * kBoxBytesB);
            tma_load_2d(sbase + s * kStageBytesA, &tmap_a, full(s), kb * kBK,
                        w.tm * kBM);
            const uint32_t bdst = sbase + kOffB + s * kStageBytesB;
            for (int c = 0; c < boxes; ++c)
              tma_load_2d(bdst + c * kBoxBytesB, &tmap_b, full(s),
                          w.n0 + 64 * c, kb * kBK);
            ++it;
          }
        }
      }
      if (*abort) {  // let the copies still in flight land before leaving
        for (int k = it > kStages ? it - kStages : 0; k < it; ++k)
          if (!wait_phase(full(k % kStages), (k / kStages) & 1, kDrainNs,
                          nullptr, false))
            record_status(wc.status, kStatusTimeoutDrain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x, i = 0; ok && u < units; u += gridDim.x, ++i) {
        const int b = i % kBufs;
        const uint32_t idesc = idesc_f16(
            128, unit_of(u, tiles_m, tiles_n, wn, whole, parts).width,
            AB_TYPE, true);
        if (i >= kBufs &&
            !wait_phase(acc_empty(b), ((i / kBufs) - 1) & 1, wc.limit, abort,
                        false)) {
          *abort = 1;
          record_status(wc.status, kStatusTimeoutMma);
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem + b * kAccCols;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          if (!wait_phase(full(s), (it / kStages) & 1, wc.limit, abort,
                          false)) {
            *abort = 1;
            record_status(wc.status, kStatusTimeoutFull);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a0 = sbase + s * kStageBytesA;
          const uint32_t b0 = sbase + kOffB + s * kStageBytesB;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // A: 16 k = 32 bytes along the swizzled row (rows 128·hm..
            // from 16 KB·hm); B: 16 k rows
            const uint64_t bd =
                smem_desc_sw128(b0 + 2048 * kk, kBoxBytesB, 1024);
#pragma unroll
            for (int hm = 0; hm < kHalves; ++hm) {
              const uint64_t ad =
                  smem_desc_sw128(a0 + hm * 16384 + 32 * kk, 16, 1024);
              mma_f16_ss(d_tmem + hm * 256, ad, bd, idesc, (kb | kk) != 0);
            }
          }
          tc_commit(empty(s));
        }
        if (ok) tc_commit(acc_full(b));
      }
      // no MMA may still run when TMEM is freed at the end
      tc_commit(mma_done);
      if (!wait_phase(mma_done, 0, kDrainNs, nullptr, false))
        record_status(wc.status, kStatusTimeoutDrain);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;         // TMEM lane quarter = rows 32q..32q+31
    const int h = (warp - 2) >> 2;  // column half
    const uint32_t lane_bits = (uint32_t)(q * 32) << 16;
    // staging: row r (this lane) is 128 bytes at r·128, its 16-byte chunk j
    // at slot j ^ (r mod 8), the layout a 128-byte-swizzle TMA store reads
    unsigned char* stg = smem + kOffStaging + (warp - 2) * kStagingBytes;
    const uint32_t stg_s = sbase + kOffStaging + (warp - 2) * kStagingBytes;
    for (int u = blockIdx.x, i = 0; u < units; u += gridDim.x, ++i) {
      const int b = i % kBufs;
      const bool ok =
          wait_phase(acc_full(b), (i / kBufs) & 1, wc.limit, abort, true);
      if (!__all_sync(0xffffffffu, ok)) {
        *abort = 1;
        if (lane == 0) record_status(wc.status, kStatusTimeoutMma);
        break;
      }
      tc_fence_after_sync();
      const Unit w = unit_of(u, tiles_m, tiles_n, wn, whole, parts);
      const int half = w.width / 2;  // 32, 64 or 128 columns per warp
      const int n0 = w.n0 + h * half;
#pragma unroll 1
      for (int hm = 0; hm < kHalves; ++hm)
#pragma unroll 1
      for (int c0 = 0; c0 < half; c0 += 32) {
        const int m0 = w.tm * kBM + hm * 128 + q * 32;
        const int m = m0 + lane;
        float* crow = C + (long long)m * ldc;
        uint32_t v[32];
        tmem_ld32(tmem + lane_bits + b * kAccCols + hm * 256 + h * half + c0,
                  v);
        tmem_ld_wait();
        if (hm == kHalves - 1 && c0 + 32 == half) {
          // all of this warp's part of the accumulator is in registers
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty(b));
        }
        const int n = n0 + c0;
        if (c_mode == 2) {
          if (lane == 0) bulk_wait_group_read<0>();  // staging free again
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(stg + lane * 128 +
                                       ((j ^ (lane & 7)) << 4)) =
                make_float4(__uint_as_float(v[4 * j]),
                            __uint_as_float(v[4 * j + 1]),
                            __uint_as_float(v[4 * j + 2]),
                            __uint_as_float(v[4 * j + 3]));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && m0 < M && n < N) {  // else nothing to write
            tma_store_2d(&tmap_c, stg_s, n, m0);
            bulk_commit_group();
          }
        } else if (m < M) {
          if (c_mode == 1 && n + 32 <= N) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(crow + n + j) = make_float4(
                  __uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                  __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n + j < N) crow[n + j] = __uint_as_float(v[j]);
          }
        }
      }
    }
    if (c_mode == 2 && lane == 0) bulk_wait_group<0>();  // C written
  }

  griddep_launch_dependents();
  tc_fence_before_sync();
  // the roles ran on one lane of warps 0 and 1: reconverge each warp before
  // the CTA barrier (a barrier reached by part of a warp does not hold it)
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// dst = src rounded to 16 bits (nearest, ties to even) for a rows×cols
// block.  vec: cols, lds and ldd multiples of 4, src 16-byte and dst 8-byte
// aligned, so each thread converts four consecutive elements.
template <int AB_TYPE>
__global__ void __launch_bounds__(256)
    round16_kernel(long long rows, long long cols,
                   const float* __restrict__ src, long long lds,
                   uint16_t* __restrict__ dst, long long ldd, int vec) {
  griddep_wait();  // src may belong to the kernel before
  griddep_launch_dependents();
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long first = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (vec) {
    const long long groups = cols / 4;
    const long long total = rows * groups;
    for (long long g = first; g < total; g += stride) {
      const long long i = g / groups, j = (g % groups) * 4;
      const float4 x = *reinterpret_cast<const float4*>(src + i * lds + j);
      uint2 o;
      if constexpr (AB_TYPE == 1) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
        o.x = *reinterpret_cast<const uint32_t*>(&lo);
        o.y = *reinterpret_cast<const uint32_t*>(&hi);
      } else {
        const __half2 lo = __floats2half2_rn(x.x, x.y);
        const __half2 hi = __floats2half2_rn(x.z, x.w);
        o.x = *reinterpret_cast<const uint32_t*>(&lo);
        o.y = *reinterpret_cast<const uint32_t*>(&hi);
      }
      *reinterpret_cast<uint2*>(dst + i * ldd + j) = o;
    }
  } else {
    const long long total = rows * cols;
    for (long long g = first; g < total; g += stride) {
      const long long i = g / cols, j = g % cols;
      const float x = src[i * lds + j];
      uint16_t o;
      if constexpr (AB_TYPE == 1) {
        const __nv_bfloat16 r = __float2bfloat16_rn(x);
        o = *reinterpret_cast<const uint16_t*>(&r);
      } else {
        const __half r = __float2half_rn(x);
        o = *reinterpret_cast<const uint16_t*>(&r);
      }
      dst[i * ldd + j] = o;
    }
  }
}

// C[0:M, 0:N] = 0 (the empty sum of a K = 0 product).
__global__ void __launch_bounds__(256)
    fill_zero_kernel(float* C, long long ldc, long long M, long long N) {
  griddep_wait();
  griddep_launch_dependents();
  const long long total = M * N;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x;
       g < total; g += (long long)gridDim.x * blockDim.x)
    C[(g / N) * ldc + g % N] = 0.f;
}

// 2-D map of a row-major 16-bit matrix (x contiguous) with a 64 × by box in
// the 128-byte swizzle; out-of-range elements read as zeros.
bool encode_16(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* m,
               int type, const void* base, long long x, long long y,
               long long ld, int by) {
  const cuuint64_t dims[2] = {(cuuint64_t)x, (cuuint64_t)y};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)by};
  const cuuint32_t estr[2] = {1, 1};
  return encode(m,
                type == GEMM_F32_MIXED_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                2, const_cast<void*>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mixed16

Plan16 plan_mixed16(long long M, long long N, int sm_count, bool narrow,
                    int bm) {
  Plan16 p;
  p.bm = bm == 256 ? 256 : 128;
  p.wn = (!narrow || N > 128) ? 256 : (N > 64 ? 128 : 64);
  p.tiles_m = (M + p.bm - 1) / p.bm;
  p.tiles_n = (N + p.wn - 1) / p.wn;
  const long long total = p.tiles_m * p.tiles_n;
  const long long g = sm_count > 0 ? sm_count : 1;
  p.full = total;
  p.parts = 1;
  if (narrow) {
    // the tiles of the last, partly filled round: all of them when there
    // are fewer tiles than SMs
    const long long tail = total % g;
    int parts = 1;
    while (tail > 0 && parts * 2 <= p.wn / 64 && tail * parts * 2 <= g)
      parts *= 2;
    if (parts > 1) {
      p.full = total - tail;
      p.parts = parts;
    }
  }
  p.units = p.full + (total - p.full) * p.parts;
  p.grid = (int)(p.units < g ? p.units : g);
  return p;
}

namespace {

template <int BM>
cudaError_t launch_bm(const Problem16& p, const Plan16& plan, bool c_vec,
                      const WaitCfg& wc, cudaStream_t stream) {
  using namespace mixed16;
  using Sh = Shape<BM>;
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap ta, tb;
  if (!encode_16(encode, &ta, p.type, p.A, p.K, p.M, p.lda, BM) ||
      !encode_16(encode, &tb, p.type, p.B, p.N, p.K, p.ldb, kBK))
    return cudaErrorInvalidValue;
  // C: fp32 M×N, 32×32 boxes in the 128-byte swizzle (rows of 128 bytes)
  CUtensorMap tc;
  std::memset(&tc, 0, sizeof(tc));
  int c_mode = c_vec ? 1 : 0;
  if (c_vec) {
    const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)p.ldc * 4};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.C, dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
      c_mode = 2;
  }
  auto fn = p.type == GEMM_F32_MIXED_BF16 ? mixed16_kernel<1, BM>
                                          : mixed16_kernel<0, BM>;
  cudaError_t e =
      ensure_smem_attr(reinterpret_cast<const void*>(fn), Sh::kSmemBytes);
  if (e != cudaSuccess) return e;
  if (plan.units > 0x7fffffffLL || plan.units < 1 || plan.grid < 1 ||
      (plan.wn != 64 && plan.wn != 128 && plan.wn != 256) ||
      (plan.parts != 1 && plan.parts != 2 && plan.parts != 4) ||
      plan.wn / plan.parts < 64 ||
      plan.bm != BM || plan.tiles_m != (p.M + BM - 1) / BM ||
      plan.tiles_n != (p.N + plan.wn - 1) / plan.wn)
    return cudaErrorInvalidConfiguration;
  return launch_pdl(fn, dim3(plan.grid), dim3(kThreads), Sh::kSmemBytes,
                    stream,
                    ta, tb, tc, p.C, p.ldc, p.M, p.N, p.K, (int)plan.tiles_m,
                    (int)plan.tiles_n, plan.wn, (int)plan.full, plan.parts,
                    (int)plan.units, c_mode, wc);
}

}  // namespace

cudaError_t launch_mixed16(const Problem16& p, const Plan16& plan, bool c_vec,
                           const WaitCfg& wc, cudaStream_t stream) {
  return plan.bm == 256 ? launch_bm<256>(p, plan, c_vec, wc, stream)
                        : launch_bm<128>(p, plan, c_vec, wc, stream);
}

cudaError_t launch_round16(int type, long long rows, long long cols,
                           const float* src, long long lds, uint16_t* dst,
                           long long ldd, int sm_count, cudaStream_t stream) {
  using namespace mixed16;
  if (rows == 0 || cols == 0) return cudaSuccess;
  const bool vec = cols % 4 == 0 && lds % 4 == 0 && ldd % 4 == 0 &&
                   (reinterpret_cast<uintptr_t>(src) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(dst) & 7u) == 0;
  const long long work = vec ? rows * (cols / 4) : rows * cols;
  long long blocks = (work + 255) / 256;
  const long long cap = 8LL * sm_count;
  if (blocks > cap) blocks = cap;
  if (type == GEMM_F32_MIXED_BF16)
    return launch_pdl(round16_kernel<1>, dim3((unsigned)blocks), dim3(256), 0,
                      stream, rows, cols, src, lds, dst, ldd, vec ? 1 : 0);
  return launch_pdl(round16_kernel<0>, dim3((unsigned)blocks), dim3(256), 0,
                    stream, rows, cols, src, lds, dst, ldd, vec ? 1 : 0);
}

cudaError_t launch_fill_zero(float* C, long long ldc, long long M, long long N,
                             int sm_count, cudaStream_t stream) {
  using namespace mixed16;
  if (M == 0 || N == 0) return cudaSuccess;
  long long blocks = (M * N + 255) / 256;
  const long long cap = 8LL * sm_count;
  if (blocks > cap) blocks = cap;
  return launch_pdl(fill_zero_kernel, dim3((unsigned)blocks), dim3(256), 0,
                    stream, C, ldc, M, N);
}

}  // namespace gemm_f32_impl
