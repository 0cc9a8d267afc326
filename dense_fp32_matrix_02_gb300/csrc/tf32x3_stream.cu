// FP32 GEMM for narrow, shallow B (N <= 128, K <= 128) and many rows of A:
// the tall-skinny, memory-bound regime, where the whole of B fits in Tensor
// Memory and the work is streaming A in and C out.  The arithmetic is the
// 3xTF32 split of the tensor kernel in tf32x3_gemm.cu (raw operands as the
// big part, truncated by the tensor core; small = x − trunc(x) exact in
// fp32; a·b ≈ a_big·b_big + a_big·b_small + a_small·b_big), computed as
// Cᵀ = Bᵀ·Aᵀ tile by tile: TMEM lane n holds column n of C.
//
// One persistent CTA per SM (608 threads) walks 128-row tiles of C:
//   warp 0       TMA producer: A in 16-deep k stages (128 rows × 64 bytes,
//                64-byte swizzle) into an 8- or 10-stage ring that runs on
//                across tiles, so the loads of the next tiles are in flight
//                while this one is multiplied and stored;
//   warps 1-2    MMA issuers (warp 1 also allocates all 512 TMEM columns),
//                taking the tiles in turn, each into its own accumulator:
//                per stage 2 k-steps × 3 tcgen05.mma kind::tf32 (M 128 =
//                columns of C, N 128 = rows, K 8).  One issuing thread gets
//                through about one such instruction per 80 ns, under half
//                the tensor core's rate for this shape, so one issuer alone
//                left the tensor core idle more than half the time and
//                bounded the kernel (a second issuer: 106.7 -> 83.5 us at
//                1048576 × 64 × 64, 12.8 -> 11.1 us at 65536 × 64 × 64);
//   warps 3-10   converters: once, Bᵀ (raw and small parts, zero past N and
//                K) into TMEM from B, which the producer's first copy puts
//                in the epilogue's staging buffers (free until the first
//                tile is stored); then per stage the small part of the A
//                tile into its own shared buffer, signalling the barrier of
//                the tile's issuer;
//   warps 11-18  epilogue: two per TMEM lane quarter, each reading half of
//                the accumulator's columns (64 rows of C) in one go and
//                releasing it at once, so the tile after next accumulates
//                into it while this one is stored.  With the fused bias /
//                GELU applied, each 32-row × 32-column block goes through
//                one of the warp's two 4 KB staging buffers (128-byte
//                swizzle) and out by a TMA bulk tensor store, which skips
//                what lies past M or N; per-lane row stores only where C
//                cannot be described by a tensor map.
// TMEM columns: accumulators [0, 256), Bᵀ raw [256, 256 + Kp), Bᵀ small
// [256 + Kp, 256 + 2·Kp), Kp = K rounded up to 16.
// Launched with programmatic stream serialization: the prologue (barriers,
// TMEM, tensor-map prefetch) overlaps the end of the kernel before it, and
// every thread waits for that kernel (griddepcontrol.wait) before touching
// global memory.
// Every mbarrier wait is bounded by %globaltimer; a role that gives up sets
// the status word and the CTA's abort flag, copies and MMAs in flight are
// waited for, TMEM is freed and the CTA ends.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "kernels.h"
#include "tcgen05.cuh"

namespace gemm_f32_impl {
namespace tf32x3_stream {

constexpr int kTileM = 128;  // rows of C per tile (the MMA's N)
constexpr int kTileN = 128;  // columns of C (the MMA's M, TMEM lanes)
constexpr int kBK = 16;      // k per stage: 64-byte rows
// A stages in the ring: 10, or 8 when a CTA has few tiles (the first
// copies of every SM then ask less of DRAM at once, and the first tiles
// start sooner: 65536 × 64 × 64 11.7 -> 10.9 µs; 1048576 rows lose 5 %
// with 8, so larger problems keep 10)
constexpr int kMaxStages = 10;
constexpr int kConvWarps = 8, kEpiWarps = 8;
// MMA issuers: warps 1 .. kIssuers; issuer w takes the tiles i (this CTA's
// count) with i mod kIssuers = w, accumulator i mod 2
constexpr int kIssuers = 2;
constexpr int kConvBase = 1 + kIssuers;                // first converter warp
constexpr int kEpiBase = kConvBase + kConvWarps;       // first epilogue warp
constexpr int kThreads = 32 * (kEpiBase + kEpiWarps);  // 608
constexpr int kStageBytes = kTileM * kBK * 4;                  // 8 KB
constexpr int kStagingBytes = 32 * 32 * 4;  // one 32×32 fp32 block
// shared memory: raw A stages, small-part stages, epilogue staging, control
__host__ __device__ constexpr int off_small(int stages) {
  return stages * kStageBytes;
}
__host__ __device__ constexpr int off_staging(int stages) {
  return 2 * stages * kStageBytes;
}
__host__ __device__ constexpr int off_ctl(int stages) {
  return off_staging(stages) + kEpiWarps * 2 * kStagingBytes;
}
constexpr int kAccCols = kTileM;
constexpr int kTmemCols = 512;
constexpr int kMaxK = (kTmemCols - 2 * kAccCols) / 2;  // 128
constexpr uint32_t kIdesc = idesc_tf32(kTileN, kTileM);
constexpr long long kDrainNs = 2000000000LL;
constexpr uint32_t kSleepNs = 100000;

struct __align__(8) Control {
  uint64_t full[kMaxStages];   // TMA -> converters (transaction bytes)
  uint64_t conv[kIssuers][kMaxStages];  // converters -> the tile's issuer
  uint64_t empty[kMaxStages];  // MMA completion -> producer
  uint64_t acc_full[2];     // last MMA of a tile -> epilogue
  uint64_t acc_empty[2];    // epilogue warps -> MMA (one arrival per warp)
  uint64_t b_full;          // TMA -> converters: B in shared memory
  uint64_t b_ready;         // Bᵀ in TMEM (one arrival per converter warp)
  uint64_t mma_done;        // every MMA issued has completed
  uint32_t tmem_base;
  int abort;
};

constexpr int smem_bytes(int stages) {
  return off_ctl(stages) + (int)sizeof(Control) + 1024;
}
static_assert(smem_bytes(kMaxStages) <= 227 * 1024, "shared memory budget");

// Tiles of A per CTA prefetched into L2 before the wait for the kernel
// before (see the prologue).
constexpr int kPrefetchTiles = 2;

// Asks the TMA unit to bring the box at (x, y) of a tensor map into L2
// (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_2d(const void* tmap, int x,
                                                   int y) {
  asm volatile(
      "cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];\n" ::
          "l"(tmap),
      "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity,
                                           long long limit_ns,
                                           volatile int* abort, bool sleep) {
  return bounded_wait(bar, parity, limit_ns, abort, sleep ? kSleepNs : 0u);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity,
                                          long long limit_ns,
                                          volatile int* abort) {
  return __all_sync(0xffffffffu, wait_phase(bar, parity, limit_ns, abort,
                                            true));
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
}

// Recomputes, in IEEE arithmetic (see ieee_dot), every NaN in column n of C,
// rows [m_lo, m_hi) (the split product gives NaN where an operand is
// infinite), with the fused bias / activation.  Kept out of line so the
// epilogue's usual path carries none of it.
__device__ __noinline__ void repair_nan_rows(float* C, long long ldc, int M,
                                             int N, int K, int m_lo,
                                             int m_hi, int n, float bias_n,
                                             int act, bool epi,
                                             RawOperands raw,
                                             unsigned int* status) {
  const long long c_ext = matrix_extent_bytes(M, N, ldc);
  for (int m = m_lo; m < m_hi && m < M; ++m) {
    float* d = C + (long long)m * ldc + n;
    if (!span_ok(d, 4, C, c_ext, status) || *d == *d) continue;
    float y = ieee_dot(raw, m, n, 0, K);
    if (epi) y = epilogue_act(y + bias_n, act);
    *d = y;
  }
}

template <int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    tf32x3_stream_kernel(const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ CUtensorMap tmap_c, float* C,
                         long long ldc, int M, int N, int K, int nb,
                         int tiles, int c_tma, const float* bias, int act,
                         RawOperands raw, WaitCfg wc) {
  static_assert(STAGES >= 2 && STAGES <= kMaxStages, "ring depth");
  constexpr int kStages = STAGES;
  constexpr int kOffSmall = off_small(STAGES);
  constexpr int kOffStaging = off_staging(STAGES);
  constexpr int kOffCtl = off_ctl(STAGES);
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  Control* ctl = reinterpret_cast<Control*>(smem + kOffCtl);
  volatile int* abort = &ctl->abort;
  auto full = [&](int s) { return smem_u32(&ctl->full[s]); };
  auto conv = [&](int w, int s) { return smem_u32(&ctl->conv[w][s]); };
  auto empty = [&](int s) { return smem_u32(&ctl->empty[s]); };
  auto acc_full = [&](int b) { return smem_u32(&ctl->acc_full[b]); };
  auto acc_empty = [&](int b) { return smem_u32(&ctl->acc_empty[b]); };
  const uint32_t b_full = smem_u32(&ctl->b_full);
  const uint32_t b_ready = smem_u32(&ctl->b_ready);
  const uint32_t mma_done = smem_u32(&ctl->mma_done);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nks = (K + kBK - 1) / kBK;  // stages per tile, 1..8 (host)
  const int kp = nks * kBK;             // K rounded up to 16

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      for (int w = 0; w < kIssuers; ++w) mbar_init(conv(w, s), kConvWarps);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), kEpiWarps);
    }
    mbar_init(b_full, 1);
    mbar_init(b_ready, kConvWarps);
    mbar_init(mma_done, kIssuers);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
    if (c_tma) prefetch_tmap(&tmap_c);
    // While the kernel before ends, bring this CTA's first tiles of A and
    // all of B into L2.  A prefetch only warms L2 (the point of coherence,
    // so nothing stale can be read later): the copies that use the data
    // still wait for that kernel first.
    for (int t = blockIdx.x, j = 0; j < kPrefetchTiles && t < tiles;
         t += gridDim.x, ++j)
      for (int kb = 0; kb < nks; ++kb)
        tma_prefetch_l2_2d(&tmap_a, kb * kBK, t * kTileM);
    tma_prefetch_l2_2d(&tmap_b, 0, 0);
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
  const uint32_t bt_raw = tmem + 2 * kAccCols;
  const uint32_t bt_small = bt_raw + kp;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;  // stages issued, over all tiles of this CTA
      bool b_sent = false;
      if (!(wc.debug & kDebugStallProducer)) {
        // B first (nb × kp box: rows k, columns n, zero past K and N)
        mbar_arrive_expect_tx(b_full, nb * kp * 4);
        tma_load_2d(sbase + kOffStaging, &tmap_b, b_full, 0, 0);
        b_sent = true;
        for (int t = blockIdx.x; t < tiles && !*abort; t += gridDim.x) {
          for (int kb = 0; kb < nks; ++kb) {
            const int s = it % kStages;
            if (it >= kStages &&
                !wait_phase(empty(s), ((it / kStages) - 1) & 1, wc.limit,
                            abort, false)) {
              *abort = 1;
              record_status(wc.status, kStatusTimeoutEmpty);
              break;
            }
            mbar_arrive_expect_tx(full(s), kStageBytes);
            tma_load_2d(sbase + s * kStageBytes, &tmap_a, full(s), kb * kBK,
                        t * kTileM);
            ++it;
          }
        }
      }
      if (*abort) {  // let the copies still in flight land before leaving
        for (int k = it > kStages ? it - kStages : 0; k < it; ++k)
          if (!wait_phase(full(k % kStages), (k / kStages) & 1, kDrainNs,
                          nullptr, false))
            record_status(wc.status, kStatusTimeoutDrain);
        if (b_sent && !wait_phase(b_full, 0, kDrainNs, nullptr, false))
          record_status(wc.status, kStatusTimeoutDrain);
      }
    }
  } else if (warp < kConvBase) {
    // ----------------------------------------------------------- MMA issuers
    if (lane == 0) {
      const int w = warp - 1;
      bool ok = wait_phase(b_ready, 0, wc.limit, abort, false);
      if (!ok) {
        *abort = 1;
        record_status(wc.status, kStatusTimeoutFull);
      }
      // bit s: parity of this issuer's next wait on conv(w, s); its own
      // uses of ring slot s complete that barrier's phases in order
      uint32_t conv_par = 0;
      for (int t = blockIdx.x, i = 0; ok && t < tiles; t += gridDim.x, ++i) {
        if (i % kIssuers != w) continue;
        int it = i * nks;  // the tile's first stage, over all tiles
        const int b = i & 1;
        if (i >= 2 && !wait_phase(acc_empty(b), ((i >> 1) - 1) & 1, wc.limit,
                                  abort, false)) {
          *abort = 1;
          record_status(wc.status, kStatusTimeoutMma);
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem + b * kAccCols;
        for (int kb = 0; kb < nks; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t par = (conv_par >> s) & 1u;
          conv_par ^= 1u << s;
          if (!wait_phase(conv(w, s), par, wc.limit, abort, false)) {
            *abort = 1;
            record_status(wc.status, kStatusTimeoutFull);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_big = sbase + s * kStageBytes;
          const uint32_t a_small = sbase + kOffSmall + s * kStageBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 8; ++kk) {
            const uint32_t col = (uint32_t)(kb * kBK + 8 * kk);
            const uint64_t d_big = smem_desc_kmajor_sw64(a_big + 32 * kk);
            const uint64_t d_small = smem_desc_kmajor_sw64(a_small + 32 * kk);
            mma_tf32_ts(d_tmem, bt_small + col, d_big, kIdesc,
                        (kb | kk) != 0);
            mma_tf32_ts(d_tmem, bt_raw + col, d_small, kIdesc, 1);
            mma_tf32_ts(d_tmem, bt_raw + col, d_big, kIdesc, 1);
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
  } else if (warp < kEpiBase) {
    // ------------------------------------------------------------ converters
    const int q = warp & 3;         // TMEM lane quarter
    const int h = (warp - kConvBase) >> 2;  // half of Bᵀ's k range
    const int n = q * 32 + lane;    // column of C = TMEM lane
    const uint32_t lane_bits = (uint32_t)(q * 32) << 16;
    // Bᵀ, k in [h·kp/2, (h+1)·kp/2) (a multiple of 8 wide): column n of
    // the staged B (rows of nb floats), contiguous across the warp
    bool ok = warp_wait(b_full, 0, wc.limit, abort);
    if (!ok) {
      *abort = 1;
      if (lane == 0) record_status(wc.status, kStatusTimeoutFull);
    } else {
      const float* bs = reinterpret_cast<const float*>(smem + kOffStaging);
      for (int k0 = h * (kp / 2); k0 < (h + 1) * (kp / 2); k0 += 8) {
        uint32_t raw[8], small[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          // B's box (nb × kp floats) in the epilogue staging
          const float* bp = bs + (k0 + j) * nb + n;
          const float x =
              n < nb && span_ok(bp, 4, bs, 4LL * nb * kp, wc.status) ? *bp
                                                                    : 0.f;
          raw[j] = __float_as_uint(x);
          small[j] = tf32_small_of_truncated(x);
        }
        if (tmem_span_ok(bt_raw + lane_bits + k0, 8, tmem, kTmemCols, q,
                         wc.status) &&
            tmem_span_ok(bt_small + lane_bits + k0, 8, tmem, kTmemCols, q,
                         wc.status)) {
          tmem_st8(bt_raw + lane_bits + k0, raw);
          tmem_st8(bt_small + lane_bits + k0, small);
        }
      }
    }
    tmem_st_wait();
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(b_ready);

    const int t32 = threadIdx.x - 32 * kConvBase;  // 0..255
    int it = 0;
    for (int t = blockIdx.x, i = 0; ok && t < tiles; t += gridDim.x, ++i) {
      for (int kb = 0; kb < nks; ++kb, ++it) {
        const int s = it % kStages;
        if (!warp_wait(full(s), (it / kStages) & 1, wc.limit, abort)) {
          *abort = 1;
          if (lane == 0) record_status(wc.status, kStatusTimeoutFull);
          ok = false;
          break;
        }
        // small part of the raw A tile, position for position (the
        // swizzle is the same in both buffers)
        const float4* araw =
            reinterpret_cast<const float4*>(smem + s * kStageBytes);
        float4* asml =
            reinterpret_cast<float4*>(smem + kOffSmall + s * kStageBytes);
#pragma unroll
        for (int j = 0; j < kStageBytes / 16 / (32 * kConvWarps); ++j) {
          const int c = t32 + 32 * kConvWarps * j;
          if (!span_ok(araw + c, 16, araw, kStageBytes, wc.status)) continue;
          const float4 v = araw[c];
          asml[c] = make_float4(
              __uint_as_float(tf32_small_of_truncated(v.x)),
              __uint_as_float(tf32_small_of_truncated(v.y)),
              __uint_as_float(tf32_small_of_truncated(v.z)),
              __uint_as_float(tf32_small_of_truncated(v.w)));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(conv(i % kIssuers, s));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - kEpiBase;        // 0..7
    const int q = warp & 3;               // TMEM lane quarter
    const int hh = e >> 2;                // half of the accumulator columns
    const int n = q * 32 + lane;
    const uint32_t lane_bits = (uint32_t)(q * 32) << 16;
    const bool active = q * 32 < N;       // this quarter holds columns of C
    const float bias_n = (bias != nullptr && n < N) ? bias[n] : 0.f;
    const bool epi = bias != nullptr || act != 0;
    unsigned char* stg0 = smem + kOffStaging + e * 2 * kStagingBytes;
    const uint32_t stg0_s = sbase + kOffStaging + e * 2 * kStagingBytes;
    int chunk = 0;  // staged blocks so far (alternating buffers)
    for (int t = blockIdx.x, i = 0; t < tiles; t += gridDim.x, ++i) {
      const int b = i & 1;
      if (!warp_wait(acc_full(b), (i >> 1) & 1, wc.limit, abort)) {
        *abort = 1;
        if (lane == 0) record_status(wc.status, kStatusTimeoutMma);
        break;
      }
      tc_fence_after_sync();
      if (!active) {
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty(b));
        continue;
      }
      // this warp's 64 accumulator columns (rows of C) in four loads
      // issued together, then the accumulator goes back to the MMA
      const int c_begin = hh * (kAccCols / 2);
      uint32_t v[kAccCols / 2];
      if (tmem_span_ok(tmem + lane_bits + b * kAccCols + c_begin,
                       kAccCols / 2, tmem, kTmemCols, q, wc.status)) {
#pragma unroll
        for (int c = 0; c < kAccCols / 2; c += 16)
          tmem_ld16(tmem + lane_bits + b * kAccCols + c_begin + c, v + c);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int c = 0; c < kAccCols / 2; ++c) v[c] = 0u;
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(b));
      const int m0 = t * kTileM + c_begin;
      const bool nan_here = any_nan(v);
      if (epi) {
#pragma unroll
        for (int r = 0; r < kAccCols / 2; ++r)
          v[r] = __float_as_uint(
              epilogue_act(__uint_as_float(v[r]) + bias_n, act));
      }
      if (c_tma) {
#pragma unroll
        for (int j = 0; j < kAccCols / 2 / 32; ++j, ++chunk) {
          // staging row r (32 floats, 128 bytes): element (r, lane) in
          // 16-byte chunk (lane / 4) ^ (r mod 8), the layout a 128-byte
          // swizzle TMA store reads
          const int sb = chunk & 1;
          if (lane == 0) bulk_wait_group_read<1>();  // buffer sb free
          __syncwarp();
          unsigned char* stg = stg0 + sb * kStagingBytes;
#pragma unroll
          for (int r = 0; r < 32; ++r) {
            unsigned char* sp =
                stg + r * 128 + ((((lane >> 2) ^ (r & 7)) << 4) |
                                 ((lane & 3) << 2));
            if (span_ok(sp, 4, stg0, 2 * kStagingBytes, wc.status))
              *reinterpret_cast<uint32_t*>(sp) = v[32 * j + r];
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && m0 + 32 * j < M) {
            tma_store_2d(&tmap_c, stg0_s + sb * kStagingBytes, q * 32,
                         m0 + 32 * j);
            bulk_commit_group();
          }
        }
      } else if (n < N) {
        const long long c_ext = matrix_extent_bytes(M, N, ldc);
#pragma unroll
        for (int r = 0; r < kAccCols / 2; ++r) {
          float* d = C + (long long)(m0 + r) * ldc + n;
          if (m0 + r < M && span_ok(d, 4, C, c_ext, wc.status))
            *d = __uint_as_float(v[r]);
        }
      }
      // NaN outputs (an infinite operand) are recomputed in IEEE arithmetic
      // once this warp's stores of the tile have landed; out of line, so
      // the common case pays only for the test
      if (__any_sync(0xffffffffu, nan_here)) {
        if (c_tma) {
          if (lane == 0) bulk_wait_group<0>();
          __syncwarp();
          fence_proxy_async_global();
        }
        if (nan_here && n < N)
          repair_nan_rows(C, ldc, M, N, K, m0, m0 + kAccCols / 2, n, bias_n,
                          act, epi, raw, wc.status);
        __syncwarp();
      }
    }
    if (c_tma && lane == 0) bulk_wait_group<0>();  // C written
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

}  // namespace tf32x3_stream

bool tf32x3_stream_fits(long long N, long long K) {
  return N >= 1 && N <= tf32x3_stream::kTileN && K >= 1 &&
         K <= tf32x3_stream::kMaxK;
}

cudaError_t launch_tf32x3_stream(const Problem& p, int sm_count,
                                 const WaitCfg& wc, cudaStream_t stream) {
  using namespace tf32x3_stream;
  if (!tf32x3_stream_fits(p.N, p.K) || p.M < 1 || p.batch != 1 ||
      p.transA || p.transB || p.storeT)
    return cudaErrorInvalidValue;
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  // A: K × M elements (x = k), rows lda apart; 16 × 128 boxes, 64-byte
  // swizzle; out-of-range elements read as zeros
  CUtensorMap ta;
  const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)p.M};
  const cuuint64_t strides[1] = {(cuuint64_t)p.lda * 4};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kTileM};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
             const_cast<float*>(p.A), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // B: N × K elements (x = n); one nb × kp box, nb = N rounded up to 4 (the
  // box's rows are whole 16-byte units), zero past N and K
  const int nks = (p.K + kBK - 1) / kBK, kp = nks * kBK;
  const int nb = (p.N + 3) / 4 * 4;
  CUtensorMap tb;
  const cuuint64_t bdims[2] = {(cuuint64_t)p.N, (cuuint64_t)p.K};
  const cuuint64_t bstrides[1] = {(cuuint64_t)p.ldb * 4};
  const cuuint32_t bbox[2] = {(cuuint32_t)nb, (cuuint32_t)kp};
  if (encode(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(p.B),
             bdims, bstrides, bbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // C: N × M elements (x = n), 32 × 32 boxes in the 128-byte swizzle, when
  // C is 16-byte aligned with ldc a multiple of 4; else lane stores
  CUtensorMap tc;
  std::memset(&tc, 0, sizeof(tc));
  int c_tma = 0;
  if ((reinterpret_cast<uintptr_t>(p.C) & 15u) == 0 && p.ldc % 4 == 0) {
    const cuuint64_t cdims[2] = {(cuuint64_t)p.N, (cuuint64_t)p.M};
    const cuuint64_t cstrides[1] = {(cuuint64_t)p.ldc * 4};
    const cuuint32_t cbox[2] = {32, 32};
    if (encode(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.C, cdims, cstrides,
               cbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
      c_tma = 1;
  }
  const long long tiles = ((long long)p.M + kTileM - 1) / kTileM;
  const int grid = (int)(tiles < sm_count ? tiles : sm_count);
  const bool few = tiles <= 8LL * grid;  // at most 8 tiles a CTA
  auto fn = few ? tf32x3_stream_kernel<8> : tf32x3_stream_kernel<kMaxStages>;
  const int smem = few ? smem_bytes(8) : smem_bytes(kMaxStages);
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(fn), smem);
  if (e != cudaSuccess) return e;
  RawOperands raw;
  raw.A = p.A;
  raw.lda = p.lda;
  raw.sA = 0;
  raw.B = p.B;
  raw.ldb = p.ldb;
  raw.sB = 0;
  raw.transA = 0;
  raw.transB = 0;
  return launch_pdl(fn, dim3(grid), dim3(kThreads), smem, stream, ta, tb, tc,
                    p.C, p.ldc, p.M, p.N, p.K, nb, (int)tiles, c_tma, p.bias,
                    p.act, raw, wc);
}

}  // namespace gemm_f32_impl
