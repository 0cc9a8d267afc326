// FP32 GEMM on the tcgen05 tensor cores by three TF32 products per term.
//
// The pages' own tensor-core path ("Rendre le GPU rapide", section "Les
// Tensor Cores") rounds operands to 16 bits and keeps the sums in f32; that
// cannot hold single-precision accuracy.  Here every fp32 value x is split
// into a TF32 part big and small = x − big, which fp32 holds exactly.  Then
//     a·b ≈ a_big·b_big + a_big·b_small + a_small·b_big
// drops only a_small·b_small and the TF32 truncation of small, and the sums
// run in the tensor core's fp32 accumulator in Tensor Memory (TMEM).  Two
// splits are built:
//   * rounded: big = x rounded to the nearest TF32 value (ties to even, the
//     integer add-and-cut that the same section uses for bf16), written out
//     explicitly; per-term error ≈ 2^-21 |a b|;
//   * raw (the default): the MMAs read x itself and the tensor core keeps
//     its top 19 bits, so big = x truncated to TF32 and the converters only
//     write small = x − trunc(x); per-term error ≤ 3·2^-20 |a b|.  A test
//     (A·I = A bit for bit) pins the truncation this relies on.
// Both are far inside the single-precision tolerance.
//
// The kernel computes the tile of C transposed, Cᵀ = Bᵀ·Aᵀ, so that neither
// operand needs a transpose in shared memory:
//   * the MMA's A operand is Bᵀ (128 columns of C × k), written into TMEM by
//     converter threads: TMEM lane n takes column n of the B tile, which the
//     32 threads of a warp read as contiguous rows of B in shared memory;
//   * the MMA's B operand is the A tile (TILE_M rows of C × k), K-major as
//     TMA copies it from row-major A, 64-byte swizzled.
// The fp32 accumulator D (TMEM lane = column n of C, TMEM column = row m of
// C) is read back by the same converter warps once every MMA has completed:
// each 32-row block of a warp's 32 columns is staged in the (now idle) ring
// in the 128-byte swizzle and written by a TMA bulk tensor store (to C, or
// to the split-K scratch); for the transposed store, or a C no tensor map
// can describe, the 32 lanes store 32 consecutive columns of one row.
//
// Tiles: TILE_M rows × 128 columns of C.  For K >= 2048 the dispatcher
// takes TILE_M = 256 (5 stages of 40 KB, 512 TMEM columns, one CTA per SM:
// each B stage converted into TMEM feeds twice the MMAs); below that,
// 128 × 128 with a 4-stage ring of 16-deep k stages (24 KB each) and 256
// TMEM columns, so two CTAs share each SM and one CTA's epilogue overlaps
// the other's main loop.
// Warp roles (320 threads):
//   warp 0     TMA producer (one thread): the A tile TILE_M×16 and the B
//              tile 16×128 of each stage, completion counted on full[s];
//   warp 1     TMEM allocator and MMA issuer (one thread): waits conv[s],
//              issues 2 k-steps × 3 TF32 MMAs (M = 128, N = TILE_M, K = 8),
//              commits the stage's release to empty[s];
//   warps 2-9  converters, two per TMEM lane quarter (a warp may only touch
//              the 32 lanes of quarter warp % 4): each splits half of the
//              stage's k range of Bᵀ into TMEM and its share of the A tile
//              in shared memory (the small part into its own buffer; with
//              the rounded split also big, written back in place), then
//              stores half of its quarter's columns of D in the epilogue.
// Operand forms: B stored N×K (TB), C stored transposed (TSTORE) for the
// swapped form of op(A)ᵀ·op(B)ᵀ (both at either tile size), and A stored
// K×M (TA, 128-row tiles: transposed by the converters from a staging
// buffer); strided
// batches run as gridDim.z; split-K writes partial tiles that a second
// kernel adds in split order.
// Launched with programmatic stream serialization: the prologue overlaps
// the end of the kernel before it (every thread waits for it with
// griddepcontrol.wait before touching global memory), and the converters
// let the next kernel be scheduled once the main loop is over.
// Every mbarrier wait is bounded by a %globaltimer deadline; a wait that
// runs out sets the status word and a CTA-wide abort flag, the roles drain
// their copies and MMAs in flight, TMEM is freed, and the CTA ends without
// writing C.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "tcgen05.cuh"

namespace gemm_f32_impl {
namespace tf32x3 {

// Tile configuration.  TILE_M rows of C per CTA (the MMA's N), always 128
// columns (the MMA's M = TMEM lanes), STAGES-deep ring of 16-deep k stages.
// TB: B is stored transposed (N×K, K-contiguous); its tile arrives as
// 128 rows n of 16 k (64-byte swizzle) and a converter lane reads its own
// row instead of a column.  TSTORE: the product computed is Cᵀ and is
// stored transposed (used for op(A)ᵀ·op(B)ᵀ = (B·A)ᵀ with A, B swapped).
// TA: A is stored transposed (K×M, M-contiguous); its tile lands as 16 rows
// k of 128 m in a staging buffer, and each converter lane takes one m (a
// column of the staged tile, contiguous across the warp) and writes the
// raw value and the small part K-major, in the 64-byte swizzle TMA would
// have used, into the stage's A buffers.
template <int TILE_M, int STAGES, bool RAW_BIG, bool TB = false,
          bool TSTORE = false, bool TA = false>
struct Cfg {
  static constexpr bool kTB = TB;
  static constexpr bool kTStore = TSTORE;
  static constexpr bool kTA = TA;
  // RAW_BIG: the MMAs read the raw fp32 operands as their "big" part and the
  // tensor core keeps their top 19 bits (TF32 truncation); converters then
  // write only small = x - trunc(x).  Otherwise big is rounded to the
  // nearest TF32 value explicitly and written out as well.
  static constexpr bool kRawBig = RAW_BIG;
  static constexpr int kTileM = TILE_M;
  static constexpr int kTileN = 128;
  static constexpr int kBK = 16;  // k per stage: 64-byte rows
  static constexpr int kStages = STAGES;
  static constexpr int kThreads = 320;
  static constexpr int kConvWarps = 8;
  static constexpr int kAccCols = kTileM;  // TMEM columns of the accumulator
  static constexpr int kTmemNeed = kAccCols + kStages * 2 * kBK;
  static constexpr int kTmemCols = kTmemNeed <= 256 ? 256 : 512;
  static constexpr int kStageBytesA = kTileM * kBK * 4;
  static constexpr int kStageBytesB = kBK * kTileN * 4;
  static constexpr uint32_t kIdesc = idesc_tf32(kTileN, kTileM);
  static constexpr int kOffASmall = kStages * kStageBytesA;
  static constexpr int kOffB = 2 * kStages * kStageBytesA;
  // TA: the staging buffers of the stored (transposed) A tiles
  static constexpr int kOffAT = kOffB + kStages * kStageBytesB;
  static constexpr int kOffCtl = kOffAT + (TA ? kStages * kStageBytesA : 0);
  static constexpr int kMinBlocks = kTmemCols == 256 ? 2 : 1;
  static_assert(kTmemNeed <= kTmemCols, "TMEM budget");
  static_assert(TILE_M % 16 == 0 && TILE_M >= 64 && TILE_M <= 256,
                "MMA N in [64, 256], multiple of 16");
  static_assert(!TB || RAW_BIG, "transposed B only with the raw split");
  static_assert(!TA || (RAW_BIG && TILE_M == 128 && !TB && !TSTORE),
                "transposed A: raw split, 128-row tiles, plain B and store");
  // the epilogue stages 8 warps × TILE_M / 64 blocks of 4 KB in the ring
  static_assert(8 * (TILE_M / 64) * 4096 <= kOffCtl, "epilogue staging");
  // a cluster-reduced split keeps its whole partial tile in the ring
  static_assert(TILE_M * 128 * 4 <= kOffCtl, "partial tile in the ring");
};

constexpr int kMaxStages = 8;
constexpr long long kDrainNs = 2000000000LL;

struct __align__(8) Control {
  uint64_t full[kMaxStages];   // TMA -> converters (tx bytes)
  uint64_t conv[kMaxStages];   // converters -> MMA (one arrival per warp)
  uint64_t empty[kMaxStages];  // MMA completion -> producer
  uint64_t accum;              // last MMA completion -> epilogue
  uint32_t tmem_base;
  int abort;
};

template <class C>
constexpr int smem_bytes() {
  return C::kOffCtl + (int)sizeof(Control) + 1024;
}

// Rounds x to the nearest TF32 value (ties to even) and returns the exact
// remainder x - big.  Values TF32 holds exactly give small = 0; NaN stays
// NaN; ±Inf gives small = NaN (so an Inf input turns the outputs it reaches
// into NaN, which the epilogue then recomputes in IEEE arithmetic).
__device__ __forceinline__ void tf32_split(float x, uint32_t& big,
                                           uint32_t& small) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t b = (u + 0xFFFu + ((u >> 13) & 1u)) & 0xFFFFE000u;
  big = b;
  small = __float_as_uint(__fsub_rn(x, __uint_as_float(b)));
}

// Bounded wait on one phase of an mbarrier.  Gives up (false) when the CTA
// abort flag is raised or `limit_ns` of %globaltimer time pass.  With
// `sleep`, each probe lets the thread sleep until the phase completes (up to
// kSleepNs) instead of polling shared memory; the single-thread roles that
// feed the pipeline (producer, MMA issuer) poll, to react at once.
constexpr uint32_t kSleepNs = 200000;

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity,
                                           long long limit_ns,
                                           volatile int* abort,
                                           bool sleep = true) {
  return bounded_wait(bar, parity, limit_ns, abort, sleep ? kSleepNs : 0u);
}

// The same for all 32 lanes of a warp: every lane waits, and the warp goes
// on only if all of them saw the phase (tcgen05.ld/st need the whole warp).
__device__ __forceinline__ bool warp_wait_phase(uint32_t bar, uint32_t parity,
                                                long long limit_ns,
                                                volatile int* abort) {
  const bool ok = wait_phase(bar, parity, limit_ns, abort);
  return __all_sync(0xffffffffu, ok);
}

template <class Cf>
__global__ void __launch_bounds__(Cf::kThreads, Cf::kMinBlocks)
    tf32x3_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                       const __grid_constant__ CUtensorMap tmap_b,
                       const __grid_constant__ CUtensorMap tmap_c,
                       const __grid_constant__ CUtensorMap tmap_p, float* C,
                       long long ldc, int M, int N, int K, int tiles_m,
                       int tiles_n, int full_tiles, int tail_splits,
                       int kb_per_split, float* partials, long long sC,
                       int batched_ab, int store_tma, int cluster_reduce,
                       int cta_base, int pdl_flags, const float* bias,
                       int act, RawOperands raw, WaitCfg wc) {
  // batch: matrix blockIdx.z; tensor-map batch coordinates are z for a
  // batched operand and 0 for one shared by every product (batched_ab bits
  // 0 = A, 1 = B); C advances by sC per product.
  constexpr int kTileM = Cf::kTileM, kTileN = Cf::kTileN, kBK = Cf::kBK;
  constexpr int kStages = Cf::kStages, kConvWarps = Cf::kConvWarps;
  constexpr int kAccCols = Cf::kAccCols, kTmemCols = Cf::kTmemCols;
  constexpr int kStageBytesA = Cf::kStageBytesA;
  constexpr int kStageBytesB = Cf::kStageBytesB;
  constexpr int kOffASmall = Cf::kOffASmall, kOffB = Cf::kOffB;
  constexpr uint32_t kIdesc = Cf::kIdesc;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  Control* ctl = reinterpret_cast<Control*>(smem + Cf::kOffCtl);
  volatile int* abort = &ctl->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work of this CTA.  The first full_tiles CTAs each take one whole tile
  // (in the grouped tile order) and store it to C.  Each tile after those
  // (a tail tile: the last, partly filled round of CTAs) is split over
  // tail_splits adjacent CTAs: CTA full_tiles + j·tail_splits + s sums k
  // stages [s·kb_per_split, min(nk, (s+1)·kb_per_split)) of tail tile j and
  // stores that partial tile, TILE_M × 128 row-major, to workspace slot
  // j·tail_splits + s; a second kernel adds the slots in split order.
  // (cta_base: the index of this launch's first CTA in that numbering —
  // a launch of only the split tail tiles starts at full_tiles)
  const int cta = (int)blockIdx.x + cta_base;
  const bool whole = cta < full_tiles;
  const int jt = whole ? 0 : (cta - full_tiles) / tail_splits;
  const int split = whole ? 0 : (cta - full_tiles) % tail_splits;
  int tm, tn;
  tile_coords<8>(whole ? cta : full_tiles + jt, tiles_m, tiles_n, tm, tn);
  const int bm = tm * kTileM, bn = tn * kTileN;
  const int nk_total = (K + kBK - 1) / kBK;
  const int kb0 = split * kb_per_split;
  const int nk = whole ? nk_total
                       : min(nk_total, kb0 + kb_per_split) - kb0;  // >= 1
  const int z = blockIdx.z;
  const int za = (batched_ab & 1) ? z : 0, zb = (batched_ab & 2) ? z : 0;
  // element (m, n) goes to out[(m − mo)·ldo + (n − no)]
  float* out = C + z * sC;
  long long ldo = ldc;
  int mo = 0, no = 0;
  if (!whole) {
    out = partials + (long long)(jt * tail_splits + split) * kTileM * kTileN;
    ldo = kTileN;
    mo = bm;
    no = bn;
  }

  auto full = [&](int s) { return smem_u32(&ctl->full[s]); };
  auto conv = [&](int s) { return smem_u32(&ctl->conv[s]); };
  auto empty = [&](int s) { return smem_u32(&ctl->empty[s]); };
  const uint32_t accum = smem_u32(&ctl->accum);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(conv(s), kConvWarps);
      mbar_init(empty(s), 1);
    }
    mbar_init(accum, 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;
  // pdl_flags bit 1: the launch of the split tail tiles that follows a
  // launch of the whole tiles; it needs nothing from that kernel (other
  // tiles of C), which let it be scheduled once past its own wait (bit 0),
  // so it starts at once and waits for it only before it ends
  if (!(pdl_flags & 2))
    griddep_wait();  // A, B, C and the scratch may belong to the kernel before
  if (pdl_flags & 1) griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      if (!(wc.debug & kDebugStallProducer)) {
        for (int kb = 0; kb < nk; ++kb) {
          const int s = kb % kStages;
          const uint32_t use = kb / kStages;
          if (kb >= kStages &&
              !wait_phase(empty(s), (use - 1) & 1, wc.limit, abort, false)) {
            *abort = 1;
            record_status(wc.status, kStatusTimeoutEmpty);
            break;
          }
          mbar_arrive_expect_tx(full(s), kStageBytesA + kStageBytesB);
          if constexpr (Cf::kTA)  // stored A: x = m, y = k
            tma_load_3d(sbase + Cf::kOffAT + s * kStageBytesA, &tmap_a,
                        full(s), bm, (kb0 + kb) * kBK, za);
          else
            tma_load_3d(sbase + s * kStageBytesA, &tmap_a, full(s),
                        (kb0 + kb) * kBK, bm, za);
          if constexpr (Cf::kTB)
            tma_load_3d(sbase + kOffB + s * kStageBytesB, &tmap_b, full(s),
                        (kb0 + kb) * kBK, bn, zb);
          else
            tma_load_3d(sbase + kOffB + s * kStageBytesB, &tmap_b, full(s),
                        bn, (kb0 + kb) * kBK, zb);
          ++issued;
        }
      }
      if (*abort) {  // let the copies still in flight land before leaving
        for (int kb = issued > kStages ? issued - kStages : 0; kb < issued;
             ++kb) {
          if (!wait_phase(full(kb % kStages), (kb / kStages) & 1, kDrainNs,
                          nullptr))
            record_status(wc.status, kStatusTimeoutDrain);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % kStages;
        if (!wait_phase(conv(s), (kb / kStages) & 1, wc.limit, abort,
                        false)) {
          *abort = 1;
          record_status(wc.status, kStatusTimeoutFull);
          break;
        }
        tc_fence_after_sync();
        const uint32_t bt_big = tmem + kAccCols + s * 2 * kBK;
        const uint32_t bt_small = bt_big + kBK;
        const uint32_t a_big = sbase + s * kStageBytesA;
        const uint32_t a_small = sbase + kOffASmall + s * kStageBytesA;
#pragma unroll
        for (int kk = 0; kk < kBK / 8; ++kk) {
          const uint64_t d_big = smem_desc_kmajor_sw64(a_big + 32 * kk);
          const uint64_t d_small = smem_desc_kmajor_sw64(a_small + 32 * kk);
          mma_tf32_ts(tmem, bt_small + 8 * kk, d_big, kIdesc,
                      (kb | kk) != 0);
          mma_tf32_ts(tmem, bt_big + 8 * kk, d_small, kIdesc, 1);
          mma_tf32_ts(tmem, bt_big + 8 * kk, d_big, kIdesc, 1);
        }
        tc_commit(empty(s));
      }
      tc_commit(accum);
      // no MMA may still run when TMEM is freed at the end
      if (!wait_phase(accum, 0, kDrainNs, nullptr))
        record_status(wc.status, kStatusTimeoutDrain);
    }
  } else {
    // ------------------------------------------------------------ converters
    const int q = warp & 3;           // TMEM lane quarter of this warp
    const int h = (warp - 2) >> 2;    // which half of k (Bᵀ) / of D columns
    const int n_loc = q * 32 + lane;  // column of the C tile = TMEM lane
    const int t = threadIdx.x - 64;   // 0..255
    const uint32_t lane_bits = (uint32_t)(q * 32) << 16;
    bool ok = true;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kStages;
      if (!warp_wait_phase(full(s), (kb / kStages) & 1, wc.limit, abort)) {
        *abort = 1;
        if (lane == 0) record_status(wc.status, kStatusTimeoutFull);
        ok = false;
        break;
      }
      // Bᵀ: column n_loc of the B tile, k in [8h, 8h + 8) -> TMEM lane n_loc
      const float* bcol =
          reinterpret_cast<const float*>(smem + kOffB + s * kStageBytesB) +
          n_loc + 8 * h * kTileN;
      uint32_t big[8], small[8];
      const uint32_t tcol = tmem + lane_bits + kAccCols + s * 2 * kBK + 8 * h;
      float4* araw = reinterpret_cast<float4*>(smem + s * kStageBytesA);
      float4* asml =
          reinterpret_cast<float4*>(smem + kOffASmall + s * kStageBytesA);
      // the stage's buffers, for the checked build
      const unsigned char* bstage = smem + kOffB + s * kStageBytesB;
      unsigned int* const st = wc.status;
      (void)bstage, (void)st;
      constexpr int kChunksPerThread = kStageBytesA / 16 / (32 * kConvWarps);
      if constexpr (Cf::kRawBig) {
        float x[8];
        if constexpr (Cf::kTB) {
          // row n_loc of the stored Bᵀ tile: 64-byte rows, 16-byte chunk c
          // at c ^ ((row >> 1) & 3); this warp's k-slice is chunks 2h, 2h+1
          const unsigned char* brow =
              smem + kOffB + s * kStageBytesB + n_loc * 64;
          const int sw = (n_loc >> 1) & 3;
          const unsigned char* p0 = brow + (((2 * h) ^ sw) << 4);
          const unsigned char* p1 = brow + (((2 * h + 1) ^ sw) << 4);
          const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
          const float4 v0 = span_ok(p0, 16, bstage, kStageBytesB, st)
                                ? *reinterpret_cast<const float4*>(p0)
                                : z4;
          const float4 v1 = span_ok(p1, 16, bstage, kStageBytesB, st)
                                ? *reinterpret_cast<const float4*>(p1)
                                : z4;
          x[0] = v0.x; x[1] = v0.y; x[2] = v0.z; x[3] = v0.w;
          x[4] = v1.x; x[5] = v1.y; x[6] = v1.z; x[7] = v1.w;
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            x[k] = span_ok(bcol + k * kTileN, 4, bstage, kStageBytesB, st)
                       ? bcol[k * kTileN]
                       : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          big[k] = __float_as_uint(x[k]);
          small[k] = tf32_small_of_truncated(x[k]);
        }
        if (tmem_span_ok(tcol, 8, tmem, kTmemCols, q, st) &&
            tmem_span_ok(tcol + kBK, 8, tmem, kTmemCols, q, st)) {
          tmem_st8(tcol, big);
          tmem_st8(tcol + kBK, small);
        }
        if constexpr (Cf::kTA) {
          // A row m = n_loc, k in [8h, 8h + 8): read down column m of the
          // staged [k][m] tile, write two 16-byte chunks of row m, raw and
          // small, at chunk c ^ ((m >> 1) & 3) of the 64-byte rows
          const float* acol = reinterpret_cast<const float*>(
                                  smem + Cf::kOffAT + s * kStageBytesA) +
                              n_loc + 8 * h * kTileM;
          float ax[8];
          const unsigned char* atstage = smem + Cf::kOffAT + s * kStageBytesA;
          (void)atstage;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            ax[k] = span_ok(acol + k * kTileM, 4, atstage, kStageBytesA, st)
                        ? acol[k * kTileM]
                        : 0.f;
          unsigned char* rraw = smem + s * kStageBytesA + n_loc * 64;
          unsigned char* rsml =
              smem + kOffASmall + s * kStageBytesA + n_loc * 64;
          const int sw = (n_loc >> 1) & 3;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int pos = ((2 * h + c) ^ sw) << 4;
            if (span_ok(rraw + pos, 16, araw, kStageBytesA, st))
              *reinterpret_cast<float4*>(rraw + pos) =
                  make_float4(ax[4 * c], ax[4 * c + 1], ax[4 * c + 2],
                              ax[4 * c + 3]);
            if (span_ok(rsml + pos, 16, asml, kStageBytesA, st))
              *reinterpret_cast<float4*>(rsml + pos) = make_float4(
                __uint_as_float(tf32_small_of_truncated(ax[4 * c])),
                __uint_as_float(tf32_small_of_truncated(ax[4 * c + 1])),
                __uint_as_float(tf32_small_of_truncated(ax[4 * c + 2])),
                __uint_as_float(tf32_small_of_truncated(ax[4 * c + 3])));
          }
        } else {
          // A: the raw tile stays the big part; only small is written
#pragma unroll
          for (int j = 0; j < kChunksPerThread; ++j) {
            const int c = t + 32 * kConvWarps * j;
            if (!span_ok(araw + c, 16, araw, kStageBytesA, st)) continue;
            const float4 v = araw[c];
            asml[c] = make_float4(
                __uint_as_float(tf32_small_of_truncated(v.x)),
                __uint_as_float(tf32_small_of_truncated(v.y)),
                __uint_as_float(tf32_small_of_truncated(v.z)),
                __uint_as_float(tf32_small_of_truncated(v.w)));
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tf32_split(span_ok(bcol + k * kTileN, 4, bstage, kStageBytesB, st)
                         ? bcol[k * kTileN]
                         : 0.f,
                     big[k], small[k]);
        if (tmem_span_ok(tcol, 8, tmem, kTmemCols, q, st) &&
            tmem_span_ok(tcol + kBK, 8, tmem, kTmemCols, q, st)) {
          tmem_st8(tcol, big);
          tmem_st8(tcol + kBK, small);
        }
        // A: element-wise, position for position (the swizzle is untouched)
#pragma unroll
        for (int j = 0; j < kChunksPerThread; ++j) {
          const int c = t + 32 * kConvWarps * j;
          if (!span_ok(araw + c, 16, araw, kStageBytesA, st)) continue;
          const float4 v = araw[c];
          uint32_t b0, b1, b2, b3, s0, s1, s2, s3;
          tf32_split(v.x, b0, s0);
          tf32_split(v.y, b1, s1);
          tf32_split(v.z, b2, s2);
          tf32_split(v.w, b3, s3);
          araw[c] = make_float4(__uint_as_float(b0), __uint_as_float(b1),
                                __uint_as_float(b2), __uint_as_float(b3));
          asml[c] = make_float4(__uint_as_float(s0), __uint_as_float(s1),
                                __uint_as_float(s2), __uint_as_float(s3));
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(conv(s));
    }
    // ------------------------------------------------------------ epilogue
    if (__all_sync(0xffffffffu, ok && !*abort)) {
      if (!warp_wait_phase(accum, 0, wc.limit, abort)) {
        *abort = 1;
        if (lane == 0) record_status(wc.status, kStatusTimeoutMma);
      } else {
        tc_fence_after_sync();
        griddep_launch_dependents();  // the main loop is over
        const int n = bn + n_loc;
        const int c_begin = h * (kAccCols / 2);
        // NaN outputs (an infinite operand) are recomputed in IEEE
        // arithmetic over this CTA's k range (see ieee_dot)
        RawOperands ro = raw;
        ro.A += za * raw.sA;
        ro.B += zb * raw.sB;
        const int k0 = kb0 * kBK, k1 = min(K, (kb0 + nk) * kBK);
        // where this CTA's stores may land (for the checked build): its
        // partial-tile slot, or the stored matrix
        const long long out_ext =
            !whole ? 4LL * kTileM * kTileN
            : Cf::kTStore ? matrix_extent_bytes(N, M, ldo)
                          : matrix_extent_bytes(M, N, ldo);
        unsigned int* const st = wc.status;
        (void)out_ext, (void)st;
        // this lane's column n has one bias value; load it once
        const bool epi = whole && (bias != nullptr || act != 0);
        const float bias_n =
            (epi && bias != nullptr && n < N) ? bias[n] : 0.f;
        // TMA stores (store_tma bit 0: whole tiles to C, bit 1: partial
        // tiles to the scratch): each 32-row block of this warp's half of
        // the accumulator (rows c of the tile × the warp's 32 columns) is
        // staged in the ring, idle now that every MMA has completed, row by
        // row in the 128-byte swizzle, and stored by one bulk tensor copy
        // that skips what lies past M or N
        const bool tma = !cluster_reduce && !Cf::kTStore &&
                         ((whole ? store_tma : store_tma >> 1) & 1);
        if (cluster_reduce) {
          // this split's partial tile, row-major TILE_M × 128 fp32 at the
          // start of the idle ring, for the cluster's reduction at the end
          float* part = reinterpret_cast<float*>(smem);
          constexpr long long kPartBytes = 4LL * kTileM * kTileN;
#pragma unroll 1
          for (int j = 0; j < kAccCols / 2 / 32; ++j) {
            uint32_t v[32];
            const uint32_t ta = tmem + lane_bits + c_begin + 32 * j;
            if (tmem_span_ok(ta, 32, tmem, kTmemCols, q, st)) {
              tmem_ld16(ta, v);
              tmem_ld16(ta + 16, v + 16);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int r = 0; r < 32; ++r) v[r] = 0u;
            }
            const bool nan_here = any_nan(v);
            const bool fix = __any_sync(0xffffffffu, nan_here);
#pragma unroll
            for (int r = 0; r < 32; ++r) {
              float* d = part + (c_begin + 32 * j + r) * kTileN + n_loc;
              if (span_ok(d, 4, part, kPartBytes, st))
                *d = __uint_as_float(v[r]);
            }
            if (fix && nan_here && n < N) {
#pragma unroll 1
              for (int r = 0; r < 32; ++r) {
                float* d = part + (c_begin + 32 * j + r) * kTileN + n_loc;
                const int m = bm + c_begin + 32 * j + r;
                if (!span_ok(d, 4, part, kPartBytes, st) || *d == *d ||
                    m >= M)
                  continue;
                *d = ieee_dot(ro, m, n, k0, k1);
              }
            }
          }
        }
        if (tma) {
          constexpr int kBlocks = kAccCols / 2 / 32;
          unsigned char* stg = smem + (warp - 2) * kBlocks * 4096;
          const uint32_t stg_s = sbase + (warp - 2) * kBlocks * 4096;
#pragma unroll 1
          for (int j = 0; j < kBlocks; ++j) {
            uint32_t v[32];
            const uint32_t ta = tmem + lane_bits + c_begin + 32 * j;
            if (tmem_span_ok(ta, 32, tmem, kTmemCols, q, st)) {
              tmem_ld16(ta, v);
              tmem_ld16(ta + 16, v + 16);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int r = 0; r < 32; ++r) v[r] = 0u;
            }
            const bool nan_here = any_nan(v);
            const bool fix = __any_sync(0xffffffffu, nan_here);
            if (epi) {
#pragma unroll
              for (int r = 0; r < 32; ++r) {
                float x = __uint_as_float(v[r]);
                if (bias != nullptr) x += bias_n;
                v[r] = __float_as_uint(epilogue_act(x, act));
              }
            }
#pragma unroll
            for (int r = 0; r < 32; ++r) {
              unsigned char* sp =
                  stg + j * 4096 + r * 128 +
                  ((((lane >> 2) ^ (r & 7)) << 4) | ((lane & 3) << 2));
              if (span_ok(sp, 4, stg, kBlocks * 4096, st))
                *reinterpret_cast<uint32_t*>(sp) = v[r];
            }
            if (fix && nan_here && n < N) {
#pragma unroll 1
              for (int r = 0; r < 32; ++r) {
                uint32_t* slot = reinterpret_cast<uint32_t*>(
                    stg + j * 4096 + r * 128 +
                    ((((lane >> 2) ^ (r & 7)) << 4) | ((lane & 3) << 2)));
                if (!span_ok(slot, 4, stg, kBlocks * 4096, st)) continue;
                const float x = __uint_as_float(*slot);
                const int m = bm + c_begin + 32 * j + r;
                if (x == x || m >= M) continue;
                float y = ieee_dot(ro, m, n, k0, k1);
                if (epi) {
                  if (bias != nullptr) y += bias_n;
                  y = epilogue_act(y, act);
                }
                *slot = __float_as_uint(y);
              }
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int x0 = bn + q * 32;  // first column of this warp
            for (int j = 0; j < kBlocks; ++j) {
              const int y0 = bm + c_begin + 32 * j;  // first row
              if (whole) {
                if (x0 < N && y0 < M)
                  tma_store_3d(&tmap_c, stg_s + j * 4096, x0, y0, z);
              } else {
                tma_store_2d(&tmap_p, stg_s + j * 4096, q * 32,
                             (jt * tail_splits + split) * kTileM + c_begin +
                                 32 * j);
              }
            }
            bulk_commit_group();
            bulk_wait_group<0>();
          }
          __syncwarp();
        }
#pragma unroll 1
        for (int c0 = c_begin; !tma && !cluster_reduce &&
                               c0 < c_begin + kAccCols / 2;
             c0 += 16) {
          uint32_t v[16];
          if (tmem_span_ok(tmem + lane_bits + c0, 16, tmem, kTmemCols, q,
                           st)) {
            tmem_ld16(tmem + lane_bits + c0, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int r = 0; r < 16; ++r) v[r] = 0u;
          }
          const bool nan_here = any_nan(v);
          const bool fix = __any_sync(0xffffffffu, nan_here) && nan_here;
          if constexpr (Cf::kTStore) {
            // this lane holds 16 consecutive rows m of column n: they are
            // 16 consecutive elements of row n of the stored transpose
            if (n < N) {
              float* dst = out + (long long)n * ldo + bm + c0;
              if (bm + c0 + 16 <= M &&
                  ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0)) {
#pragma unroll
                for (int i = 0; i < 16; i += 4)
                  if (span_ok(dst + i, 16, out, out_ext, st))
                    *reinterpret_cast<float4*>(dst + i) = make_float4(
                        __uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                        __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
              } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  if (bm + c0 + i < M && span_ok(dst + i, 4, out, out_ext, st))
                    dst[i] = __uint_as_float(v[i]);
              }
              if (fix) {
#pragma unroll 1
                for (int i = 0; i < 16 && bm + c0 + i < M; ++i)
                  if (span_ok(dst + i, 4, out, out_ext, st) && dst[i] != dst[i])
                    dst[i] = ieee_dot(ro, bm + c0 + i, n, k0, k1);
              }
            }
          } else if (n < N) {
            // fused epilogue (not on partial tiles: the reduction has it)
            if (epi) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float x = __uint_as_float(v[i]);
                if (bias != nullptr) x += bias_n;
                v[i] = __float_as_uint(epilogue_act(x, act));
              }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int m = bm + c0 + i;
              float* d = out + (long long)(m - mo) * ldo + (n - no);
              if (m < M && span_ok(d, 4, out, out_ext, st))
                *d = __uint_as_float(v[i]);
            }
            if (fix) {
#pragma unroll 1
              for (int i = 0; i < 16 && bm + c0 + i < M; ++i) {
                const int m = bm + c0 + i;
                float* d = out + (long long)(m - mo) * ldo + (n - no);
                if (!span_ok(d, 4, out, out_ext, st) || *d == *d) continue;
                float y = ieee_dot(ro, m, n, k0, k1);
                if (epi) {
                  if (bias != nullptr) y += bias_n;
                  y = epilogue_act(y, act);
                }
                *d = y;
              }
            }
          }
        }
      }
    }
  }

  griddep_launch_dependents();
  tc_fence_before_sync();
  // the roles ran on one lane of warps 0 and 1: reconverge each warp before
  // the CTA barrier (a barrier reached by part of a warp does not hold it)
  __syncwarp();
  __syncthreads();
  if (cluster_reduce) {
    // The splits of this tile are the CTAs of this cluster (rank = split).
    // Once every partial tile is in its CTA's shared memory (barrier 1),
    // CTA `split` adds rows [split·TILE_M/S, (split+1)·TILE_M/S) of the S
    // partials, read through distributed shared memory in split order
    // 0, 1, …, S−1 (the order of the reduction kernel: identical results),
    // applies the fused epilogue and stores those rows of C; barrier 2
    // keeps every CTA's partial in place until all have read it.
    cluster_sync_all();
    if (warp >= 2) {
      const int S = tail_splits;
      bool any_abort = false;
      for (int s2 = 0; s2 < S; ++s2)
        any_abort |=
            ld_cluster_s32(cluster_map(smem_u32(&ctl->abort), s2)) != 0;
      if (!any_abort) {
        const int r0 = split * kTileM / S, r1 = (split + 1) * kTileM / S;
        const int t = threadIdx.x - 64;
        const bool cvec = (reinterpret_cast<uintptr_t>(C) & 15u) == 0 &&
                          (ldc & 3) == 0;
        const bool epi = bias != nullptr || act != 0;
        const long long c_ext = matrix_extent_bytes(M, N, ldc);
        unsigned int* const st = wc.status;
        (void)c_ext, (void)st;
        for (int g = t; g < (r1 - r0) * (kTileN / 4); g += 32 * kConvWarps) {
          const int ml = r0 + g / (kTileN / 4), c4 = (g % (kTileN / 4)) * 4;
          const int m = bm + ml, n = bn + c4;
          if (m >= M || n >= N) continue;
          const uint32_t off = sbase + (uint32_t)(ml * kTileN + c4) * 4u;
          if (!smem_span_ok(off, 16, sbase, 4 * kTileM * kTileN, st)) continue;
          // every split's four values in flight at once, then the sum in
          // split order
          float4 v[kMaxClusterSplits];
#pragma unroll
          for (int s2 = 0; s2 < kMaxClusterSplits; ++s2)
            if (s2 < S) v[s2] = ld_cluster_v4(cluster_map(off, s2));
          float4 acc = v[0];
#pragma unroll
          for (int s2 = 1; s2 < kMaxClusterSplits; ++s2) {
            if (s2 >= S) break;
            acc.x += v[s2].x;
            acc.y += v[s2].y;
            acc.z += v[s2].z;
            acc.w += v[s2].w;
          }
          float a[4] = {acc.x, acc.y, acc.z, acc.w};
          if (epi)
            for (int e = 0; e < 4; ++e)
              a[e] = apply_epilogue(a[e], bias, act, n + e);
          float* dst = C + (long long)m * ldc + n;
          if (cvec && n + 3 < N) {
            if (span_ok(dst, 16, C, c_ext, st))
              *reinterpret_cast<float4*>(dst) =
                  make_float4(a[0], a[1], a[2], a[3]);
          } else {
            for (int e = 0; e < 4 && n + e < N; ++e)
              if (span_ok(dst + e, 4, C, c_ext, st)) dst[e] = a[e];
          }
        }
      }
    }
    cluster_sync_all();  // no CTA leaves while another reads its partial
  }
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  // the kernel the next one in the stream waits for must not end before
  // the whole-tile launch it overlapped
  if (pdl_flags & 2) griddep_wait();
}

// Tail tile j (tile full_tiles + j in the grouped order): C = the sum over
// s = 0..tail_splits−1, in that order, of partial slot j·tail_splits + s,
// then the fused epilogue.  Each thread adds four consecutive columns of one
// row of one tile.
__global__ void __launch_bounds__(256)
    tail_reduce_kernel(const float* __restrict__ partials, int tail_splits,
                       int full_tiles, int tail_tiles, int tile_m,
                       int tiles_m, int tiles_n, int M, int N,
                       float* __restrict__ C, long long ldc, int vec,
                       const float* __restrict__ bias, int act) {
  constexpr int kCols = 128, kGroups = kCols / 4;
  griddep_wait();  // the partial tiles of the kernel before
  griddep_launch_dependents();
  const bool epi = bias != nullptr || act != 0;
  const long long slot = (long long)tile_m * kCols;
  const long long per_tile = (long long)tile_m * kGroups;
  const long long total = (long long)tail_tiles * per_tile;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x;
       g < total; g += (long long)gridDim.x * blockDim.x) {
    const int j = (int)(g / per_tile);
    const int rem = (int)(g % per_tile);
    const int r = rem / kGroups, c4 = (rem % kGroups) * 4;
    int tm, tn;
    tile_coords<8>(full_tiles + j, tiles_m, tiles_n, tm, tn);
    const int m = tm * tile_m + r, n = tn * kCols + c4;
    if (m >= M || n >= N) continue;
    const float* src = partials + (long long)j * tail_splits * slot +
                       (long long)r * kCols + c4;
    float4 acc = *reinterpret_cast<const float4*>(src);
    // the loads of several splits in flight at once; the sums still run in
    // split order
#pragma unroll 4
    for (int s = 1; s < tail_splits; ++s) {
      const float4 v = *reinterpret_cast<const float4*>(src + s * slot);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    float a[4] = {acc.x, acc.y, acc.z, acc.w};
    if (epi)
      for (int e = 0; e < 4; ++e) a[e] = apply_epilogue(a[e], bias, act, n + e);
    float* dst = C + (long long)m * ldc + n;
    if (vec && n + 3 < N) {
      *reinterpret_cast<float4*>(dst) = make_float4(a[0], a[1], a[2], a[3]);
    } else {
      for (int e = 0; e < 4 && n + e < N; ++e) dst[e] = a[e];
    }
  }
}

// ---------------------------------------------------------------- host
}  // namespace tf32x3

namespace {

// GEMM_F32_TMA_STORE=0 keeps the epilogue's per-lane stores (comparison).
bool env_store_tma() {
  const char* v = std::getenv("GEMM_F32_TMA_STORE");
  return !(v && v[0] == '0');
}

// 3-D tensor map (x innermost, y rows, z batch) of fp32 with a box of
// bx × by × 1.  A batch stride of 0 (one matrix shared by every product)
// gives a batch extent of 1.
bool encode_3d(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* m,
               const float* base, long long x, long long y, long long ld,
               long long stride, int batch, int bx, int by,
               CUtensorMapSwizzle swz) {
  const cuuint32_t estr[3] = {1, 1, 1};
  const bool batched = batch > 1 && stride != 0;
  const cuuint64_t dims[3] = {(cuuint64_t)x, (cuuint64_t)y,
                              (cuuint64_t)(batched ? batch : 1)};
  const long long zs = batched ? stride : (y * ld + 3) / 4 * 4;
  const cuuint64_t strides[2] = {(cuuint64_t)ld * 4, (cuuint64_t)zs * 4};
  const cuuint32_t box[3] = {(cuuint32_t)bx, (cuuint32_t)by, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                const_cast<float*>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class Cf>
cudaError_t launch_cfg(const Problem& p, int full_tiles, int tail_splits,
                       float* partials, bool cluster, const WaitCfg& wc,
                       cudaStream_t stream) {
  using namespace tf32x3;
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap ta, tb;
  const bool ok_a =
      Cf::kTA ? encode_3d(encode, &ta, p.A, p.M, p.K, p.lda, p.sA, p.batch,
                          Cf::kTileM, Cf::kBK, CU_TENSOR_MAP_SWIZZLE_NONE)
              : encode_3d(encode, &ta, p.A, p.K, p.M, p.lda, p.sA, p.batch,
                          Cf::kBK, Cf::kTileM, CU_TENSOR_MAP_SWIZZLE_64B);
  if (!ok_a) return cudaErrorInvalidValue;
  const bool ok_b =
      Cf::kTB ? encode_3d(encode, &tb, p.B, p.K, p.N, p.ldb, p.sB, p.batch,
                          Cf::kBK, Cf::kTileN, CU_TENSOR_MAP_SWIZZLE_64B)
              : encode_3d(encode, &tb, p.B, p.N, p.K, p.ldb, p.sB, p.batch,
                          Cf::kTileN, Cf::kBK, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!ok_b) return cudaErrorInvalidValue;
  // C (x = n, y = m, z = batch) and the partial tiles (x = n within the
  // tile, y = slot·TILE_M + row): 32 × 32 boxes in the 128-byte swizzle,
  // stored by TMA from the epilogue; C only where a tensor map can describe
  // it (16-byte aligned, ldc and the batch stride multiples of 4), never
  // for the transposed store
  CUtensorMap tc, tp;
  std::memset(&tc, 0, sizeof(tc));
  std::memset(&tp, 0, sizeof(tp));
  int store_tma = 0;
  if (!Cf::kTStore && (reinterpret_cast<uintptr_t>(p.C) & 15u) == 0 &&
      p.ldc % 4 == 0 && (p.batch == 1 || p.sC % 4 == 0) &&
      env_store_tma()) {
    const cuuint64_t dims[3] = {(cuuint64_t)p.N, (cuuint64_t)p.M,
                                (cuuint64_t)p.batch};
    const long long zs = p.batch > 1 ? p.sC : (long long)p.M * p.ldc;
    const cuuint64_t strides[2] = {(cuuint64_t)p.ldc * 4,
                                   (cuuint64_t)((zs + 3) / 4 * 4) * 4};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.C, dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
      store_tma |= 1;
  }
  auto fn = tf32x3_gemm_kernel<Cf>;
  constexpr int kSmem = smem_bytes<Cf>();
  cudaError_t e =
      ensure_smem_attr(reinterpret_cast<const void*>(fn), kSmem);
  if (e != cudaSuccess) return e;
  const int tiles_m = (p.M + Cf::kTileM - 1) / Cf::kTileM;
  const int tiles_n = (p.N + Cf::kTileN - 1) / Cf::kTileN;
  const int nk = (p.K + Cf::kBK - 1) / Cf::kBK;
  const long long tiles = (long long)tiles_m * tiles_n;
  int ts = tail_splits;
  long long full = full_tiles;
  // the split tiles' splits as clusters: no partial-tile buffer
  bool use_cluster = cluster && p.batch == 1 && ts >= 2 &&
                     ts <= kMaxClusterSplits && full >= 0 && full < tiles;
  if (!use_cluster &&
      (ts < 2 || !partials || p.batch > 1 || full < 0 || full >= tiles)) {
    ts = 1;
    full = tiles;
  }
  const int kb_per_split = (nk + ts - 1) / ts;
  ts = (nk + kb_per_split - 1) / kb_per_split;  // no empty split
  if (ts < 2) {
    full = tiles;
    use_cluster = false;
  }
  const long long tail = tiles - full;
  const long long grid = full + tail * ts;
  if (grid > 0x7fffffffLL || p.batch < 1 || p.batch > 65535)
    return cudaErrorInvalidConfiguration;
  const int batched_ab =
      (p.batch > 1 && p.sA != 0 ? 1 : 0) | (p.batch > 1 && p.sB != 0 ? 2 : 0);
  if (tail > 0 && !use_cluster && env_store_tma()) {
    const cuuint64_t dims[2] = {128, (cuuint64_t)(tail * ts * Cf::kTileM)};
    const cuuint64_t strides[1] = {128 * 4};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, partials, dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
      store_tma |= 2;
  }
  RawOperands raw;
  raw.A = p.A;
  raw.lda = p.lda;
  raw.sA = p.sA;
  raw.B = p.B;
  raw.ldb = p.ldb;
  raw.sB = p.sB;
  raw.transA = Cf::kTA ? 1 : 0;
  raw.transB = Cf::kTB ? 1 : 0;
  if (use_cluster) {
    // whole tiles first (if any), in a launch of their own that lets the
    // next one be scheduled once past its wait for the kernel before; then
    // the split tiles, one cluster per tile, which overlap its last round
    // and wait for it only before they end
    if (full > 0) {
      e = launch_pdl(fn, dim3((unsigned)full, 1, 1), dim3(Cf::kThreads),
                     kSmem, stream, ta, tb, tc, tp, p.C, p.ldc, p.M, p.N,
                     p.K, tiles_m, tiles_n, (int)full, ts, kb_per_split,
                     (float*)nullptr, p.sC, batched_ab, store_tma, 0, 0, 1,
                     p.bias, p.act, raw, wc);
      if (e != cudaSuccess) return e;
    }
    return launch_pdl_cluster(
        fn, dim3((unsigned)(tail * ts), 1, 1), dim3(Cf::kThreads), kSmem,
        stream, (unsigned)ts, ta, tb, tc, tp, p.C, p.ldc, p.M, p.N, p.K,
        tiles_m, tiles_n, (int)full, ts, kb_per_split, (float*)nullptr, p.sC,
        batched_ab, store_tma, 1, (int)full, full > 0 ? 2 : 0, p.bias, p.act,
        raw, wc);
  }
  e = launch_pdl(fn, dim3((unsigned)grid, 1, (unsigned)p.batch),
                 dim3(Cf::kThreads), kSmem, stream, ta, tb, tc, tp, p.C,
                 p.ldc, p.M, p.N, p.K, tiles_m, tiles_n, (int)full, ts,
                 kb_per_split, partials, p.sC, batched_ab, store_tma, 0, 0, 0,
                 p.bias, p.act, raw, wc);
  if (e != cudaSuccess || tail == 0) return e;
  const int vec = ((reinterpret_cast<uintptr_t>(p.C) & 15u) == 0 &&
                   p.ldc % 4 == 0)
                      ? 1
                      : 0;
  const long long groups = tail * Cf::kTileM * (128 / 4);
  const int blocks = (int)((groups + 255) / 256 < 4096 ? (groups + 255) / 256
                                                      : 4096);
  return launch_pdl(tail_reduce_kernel, dim3(blocks), dim3(256), 0, stream,
                    (const float*)partials, ts, (int)full, (int)tail,
                    Cf::kTileM, tiles_m, tiles_n, p.M, p.N, p.C, p.ldc, vec,
                    p.bias, p.act);
}

}  // namespace


int tf32x3_tile_m(int cfg) {
  return (cfg == kTc256 || cfg == kTc256Raw) ? 256 : 128;
}

long long tf32x3_partials_bytes(int tile_m, long long split_tiles,
                                int splits) {
  return splits > 1 ? split_tiles * splits * tile_m * 128LL * 4 : 0;
}

cudaError_t launch_tf32x3(const Problem& p, int cfg, int full_tiles,
                          int splits, float* partials, bool cluster,
                          const WaitCfg& wc, cudaStream_t stream) {
  using namespace tf32x3;
  switch (cfg) {
    case kTc256:
      return launch_cfg<Cfg<256, 5, false>>(p, full_tiles, splits, partials,
                                            cluster, wc, stream);
    case kTc128:
      return launch_cfg<Cfg<128, 4, false>>(p, full_tiles, splits, partials,
                                            cluster, wc, stream);
    case kTc128Raw:
      if (p.transB)  // A·Bᵀ with B stored N×K
        return launch_cfg<Cfg<128, 4, true, true>>(p, full_tiles, splits,
                                                   partials, cluster, wc,
                                                   stream);
      if (p.storeT)  // caller passed (B, A) swapped: store the transpose
        return launch_cfg<Cfg<128, 4, true, false, true>>(p, full_tiles, splits,
                                                          partials, cluster,
                                                          wc, stream);
      if (p.transA)  // Aᵀ·B with A stored K×M: A transposed by the converters
        return launch_cfg<Cfg<128, 3, true, false, false, true>>(
            p, full_tiles, splits, partials, cluster, wc, stream);
      return launch_cfg<Cfg<128, 4, true>>(p, full_tiles, splits, partials,
                                           cluster, wc, stream);
    case kTc256Raw:
      if (p.transB)
        return launch_cfg<Cfg<256, 5, true, true>>(p, full_tiles, splits,
                                                   partials, cluster, wc,
                                                   stream);
      if (p.storeT)
        return launch_cfg<Cfg<256, 5, true, false, true>>(
            p, full_tiles, splits, partials, cluster, wc, stream);
      if (p.transA)  // the transposed-A staging exists for 128-row tiles
        return launch_tf32x3(p, kTc128Raw, full_tiles, splits, partials,
                             cluster, wc, stream);
      return launch_cfg<Cfg<256, 5, true>>(p, full_tiles, splits, partials,
                                           cluster, wc, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace gemm_f32_impl
