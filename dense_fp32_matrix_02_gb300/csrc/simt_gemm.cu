// FP32 GEMM on the FFMA pipe, operands staged by cp.async.
//
// One CTA computes a BM×BN tile of C.  The k loop walks BK-deep stages of a
// STAGES-deep shared-memory ring: while the CTA multiplies stage kt, the
// copies for stage kt + STAGES − 1 are already in flight.  This replaces
// the two __syncthreads of "3 · La mémoire partagée", §3.2-§3.3 (one after
// the cooperative load, one before the tile is overwritten) with a single
// barrier per stage: it both publishes stage kt and proves every thread has
// finished reading the stage that the next copies overwrite.
//
// Edges ("3 · La mémoire partagée", §3.3 assumes N % T == 0 and the
// cuda-oxide tiled_sgemm drops the K remainder; here every size is exact):
// copies of chunks that fall past M, N or K read only the bytes that exist
// and fill the rest with zeros, and the epilogue stores only elements inside
// M×N.
//
// With aligned operands (VEC: 16-byte aligned, leading dimensions multiples
// of 4) A is copied in 16-byte chunks and kept K-major (FfmaTile, read along
// K); otherwise it is copied one float at a time and lands transposed
// (As[BK][BM], as in §3.4 of the same page; FfmaTileT).  B is copied in
// 16-byte chunks when VEC holds and one float at a time otherwise, so any
// alignment and any leading dimension work.
#include <type_traits>

#include "ffma_tile.cuh"
#include "kernels.h"

namespace gemm_f32_impl {

// cp.async of `bytes` (0..16, or 0 / 4) from src to the shared dst; the
// checked build first tests dst against its stage buffer [dbase, dbase +
// dfloats) and, when bytes > 0, src against the operand's extent, and
// skips (or zero-fills) what falls outside.
__device__ __forceinline__ void cp16_checked(float* dst, const float* dbase,
                                             int dfloats, const float* src,
                                             int bytes, const float* sbase,
                                             long long sextent,
                                             unsigned int* st) {
  if (!span_ok(dst, 16, dbase, 4LL * dfloats, st)) return;
  if (bytes > 0 && !span_ok(src, bytes, sbase, sextent, st)) {
    src = sbase;
    bytes = 0;
  }
  cp_async16(smem_u32(dst), src, bytes);
}

__device__ __forceinline__ void cp4_checked(float* dst, const float* dbase,
                                            int dfloats, const float* src,
                                            int bytes, const float* sbase,
                                            long long sextent,
                                            unsigned int* st) {
  if (!span_ok(dst, 4, dbase, 4LL * dfloats, st)) return;
  if (bytes > 0 && !span_ok(src, bytes, sbase, sextent, st)) {
    src = sbase;
    bytes = 0;
  }
  cp_async4(smem_u32(dst), src, bytes);
}

// AKM = true keeps A K-major in shared memory (FfmaTile: 16-byte copies of
// A, read along K); false stores it transposed (FfmaTileT).
// TA / TB: A / B stored transposed in global memory (A as K×M, B as N×K).
// A transposed in memory is exactly FfmaTileT's [BK][BM] layout (16-byte
// copies when VEC); B transposed lands one float at a time in a swizzled
// [BK][BN] layout (FfmaTileT with BSWZ).
template <int BM, int BN, int BK, int STAGES, bool VEC, bool AKM = false,
          bool TA = false, bool TB = false>
struct SimtKernel {
  static_assert(!(AKM && (TA || TB)), "K-major A only for A untransposed");
  using Tile = typename std::conditional<AKM, FfmaTile<BM, BN, BK>,
                                         FfmaTileT<BM, BN, BK, TB>>::type;
  static constexpr int kThreads = Tile::kThreads;
  static constexpr int kSmemBytes = STAGES * Tile::kStageBytes + 1024;

  // Issues this thread's share of the copies for k-stage `kt` into the ring
  // slot whose A and B parts start at As and Bs.
  static __device__ __forceinline__ void load_stage(const Problem& p, float* As,
                                                    float* Bs, int bm, int bn,
                                                    int kt, int tid) {
    const int k0 = kt * BK;
    // the operands' extents (for the checked build)
    const long long ext_a =
        TA ? matrix_extent_bytes(p.K, p.M, p.lda)
           : matrix_extent_bytes(p.M, p.K, p.lda);
    const long long ext_b =
        TB ? matrix_extent_bytes(p.N, p.K, p.ldb)
           : matrix_extent_bytes(p.K, p.N, p.ldb);
    constexpr int kFA = Tile::kStageFloatsA, kFB = Tile::kStageFloatsB;
    (void)ext_a, (void)ext_b;
    if constexpr (AKM) {
      // A, K-major: 16-byte chunks (zero-filled past M or K), swizzled
      constexpr int kChunksA = BM * BK / 4;
#pragma unroll
      for (int id = tid; id < kChunksA; id += kThreads) {
        const int m = id / (BK / 4), c = id % (BK / 4);
        const int gm = bm + m, gk = k0 + 4 * c;
        int bytes = 0;
        const float* src = p.A;
        if (gm < p.M && gk < p.K) {
          bytes = 4 * min(4, p.K - gk);
          src = p.A + (long long)gm * p.lda + gk;
        }
        cp16_checked(As + m * BK + ((c ^ a_swizzle<BK>(m)) * 4), As, kFA, src,
                     bytes, p.A, ext_a, p.status);
      }
    }
    if constexpr (TA && VEC) {
      // A stored K×M: row k of the stage is 4-float chunks of row k0 + k
      constexpr int kChunksA = BK * BM / 4;
#pragma unroll
      for (int id = tid; id < kChunksA; id += kThreads) {
        const int k = id / (BM / 4), c = id % (BM / 4);
        const int gk = k0 + k, gm = bm + 4 * c;
        int bytes = 0;
        const float* src = p.A;
        if (gk < p.K && gm < p.M) {
          bytes = 4 * min(4, p.M - gm);
          src = p.A + (long long)gk * p.lda + gm;
        }
        cp16_checked(As + Tile::a_index(k, 4 * c), As, kFA, src, bytes, p.A,
                     ext_a, p.status);
      }
    } else if constexpr (TA) {
      // A stored K×M, any alignment: a warp copies 32 consecutive m of one k
      constexpr int kElemsA = BK * BM;
#pragma unroll 4
      for (int id = tid; id < kElemsA; id += kThreads) {
        const int k = id / BM, m = id % BM;
        const int gk = k0 + k, gm = bm + m;
        const bool ok = gk < p.K && gm < p.M;
        const float* src = ok ? p.A + (long long)gk * p.lda + gm : p.A;
        cp4_checked(As + Tile::a_index(k, m), As, kFA, src, ok ? 4 : 0, p.A,
                    ext_a, p.status);
      }
    }
    // A, transposed on the way in: single-float copies, a warp covering 4
    // rows × 8 consecutive k (whole 32-byte sectors of each row).
    if constexpr (!AKM && !TA) {
    constexpr int kElemsA = BM * BK;
#pragma unroll
    for (int id = tid; id < kElemsA; id += kThreads) {
      const int kl = id & 7, ml = (id >> 3) & 3, rest = id >> 5;
      const int k = (rest % (BK / 8)) * 8 + kl;
      const int m = (rest / (BK / 8)) * 4 + ml;
      const int gm = bm + m, gk = k0 + k;
      const bool ok = gm < p.M && gk < p.K;
      const float* src = ok ? p.A + (long long)gm * p.lda + gk : p.A;
      cp4_checked(As + Tile::a_index(k, m), As, kFA, src, ok ? 4 : 0, p.A,
                  ext_a, p.status);
    }
    }
    if constexpr (TB) {
      // B stored N×K, transposed on the way in like A above: a warp copies
      // 4 rows n × 8 consecutive k into eight different swizzled chunks
      constexpr int kElemsB = BK * BN;
#pragma unroll
      for (int id = tid; id < kElemsB; id += kThreads) {
        const int kl = id & 7, nl = (id >> 3) & 3, rest = id >> 5;
        const int k = (rest % (BK / 8)) * 8 + kl;
        const int n = (rest / (BK / 8)) * 4 + nl;
        const int gn = bn + n, gk = k0 + k;
        const bool ok = gn < p.N && gk < p.K;
        const float* src = ok ? p.B + (long long)gn * p.ldb + gk : p.B;
        cp4_checked(Bs + Tile::b_index(k, n), Bs, kFB, src, ok ? 4 : 0, p.B,
                    ext_b, p.status);
      }
    } else if (VEC) {
      constexpr int kChunksB = BK * BN / 4;
#pragma unroll
      for (int id = tid; id < kChunksB; id += kThreads) {
        const int k = id / (BN / 4), c = id % (BN / 4);
        const int gk = k0 + k, gn = bn + 4 * c;
        int bytes = 0;
        const float* src = p.B;
        if (gk < p.K && gn < p.N) {
          bytes = 4 * min(4, p.N - gn);
          src = p.B + (long long)gk * p.ldb + gn;
        }
        cp16_checked(Bs + k * BN + 4 * c, Bs, kFB, src, bytes, p.B, ext_b,
                     p.status);
      }
    } else {
      constexpr int kElemsB = BK * BN;
#pragma unroll 4
      for (int id = tid; id < kElemsB; id += kThreads) {
        const int k = id / BN, n = id % BN;
        const int gk = k0 + k, gn = bn + n;
        const bool ok = gk < p.K && gn < p.N;
        const float* src = ok ? p.B + (long long)gk * p.ldb + gn : p.B;
        cp4_checked(Bs + k * BN + n, Bs, kFB, src, ok ? 4 : 0, p.B, ext_b,
                    p.status);
      }
    }
  }

  static __device__ __forceinline__ void run(Problem p, int tiles_m,
                                             int tiles_n, int c_vec) {
    // matrix blockIdx.z of a strided batch
    p.A += blockIdx.z * p.sA;
    p.B += blockIdx.z * p.sB;
    p.C += blockIdx.z * p.sC;
    extern __shared__ unsigned char smem_raw[];
    float* smem = reinterpret_cast<float*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* As = smem;
    float* Bs = smem + STAGES * Tile::kStageFloatsA;

    int tm, tn;
    tile_coords<8>(blockIdx.x, tiles_m, tiles_n, tm, tn);
    const int bm = tm * BM, bn = tn * BN;
    const int tid = threadIdx.x;

    Tile tile;
    tile.init(tid);
    typename Tile::Acc acc;
    Tile::zero(acc);

    const int kt_count = (p.K + BK - 1) / BK;
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
      if (s < kt_count)
        load_stage(p, As + s * Tile::kStageFloatsA, Bs + s * Tile::kStageFloatsB,
                   bm, bn, s, tid);
      cp_async_commit();
    }
    for (int kt = 0; kt < kt_count; ++kt) {
      cp_async_wait<STAGES - 2>();
      __syncthreads();
      const int next = kt + STAGES - 1;
      if (next < kt_count) {
        const int slot = next % STAGES;
        load_stage(p, As + slot * Tile::kStageFloatsA,
                   Bs + slot * Tile::kStageFloatsB, bm, bn, next, tid);
      }
      cp_async_commit();
      const int slot = kt % STAGES;
      tile.compute(As + slot * Tile::kStageFloatsA,
                   Bs + slot * Tile::kStageFloatsB, acc, p.status);
    }
    cp_async_wait<0>();
    tile.store(p, bm, bn, c_vec != 0, acc);
  }
};

template <int BM, int BN, int BK, int STAGES, bool VEC, int MINB, bool AKM,
          bool TA, bool TB>
__global__ void __launch_bounds__(FfmaTileT<BM, BN, BK>::kThreads, MINB)
    simt_gemm_kernel(Problem p, int tiles_m, int tiles_n, int c_vec) {
  griddep_wait();  // A, B and C may belong to the kernel before
  SimtKernel<BM, BN, BK, STAGES, VEC, AKM, TA, TB>::run(p, tiles_m, tiles_n,
                                                        c_vec);
}

// ------------------------------------------------- warp-specialised
// The same 8×8 K-major tile (FfmaTile, 128 × 128 × 32 stages), with the
// copies taken off the threads that multiply: warps 0-7 only wait, compute
// and release; warps 8-11 (one warpgroup) issue every cp.async of the ring.  The pages' two
// __syncthreads per tile ("3 · La mémoire partagée", §3.2-§3.3) become two
// mbarrier phases per ring slot, as in the TMA-fed kernel:
//   full[s]   expects one arrival from each of the 128 producer threads,
//             made by cp.async.mbarrier.arrive.noinc once that thread's
//             copies into slot s have landed;
//   empty[s]  one arrival per compute warp after it has read slot s; the
//             producer waits on it before refilling the slot.
// Compute warps no longer meet at a CTA barrier every stage, and none of
// them spends issue slots on copies or waits on its own copies.  Operands
// must be 16-byte aligned with leading dimensions multiples of 4 (16-byte
// copies, zero-filled past M, N and K).  Every wait is bounded (the status
// word and a CTA abort flag, as in the other pipelined kernels).
namespace simt_ws {

constexpr int kBM = 128, kBN = 128, kBK = 32, kStages = 4;
using Tile = FfmaTile<kBM, kBN, kBK>;
constexpr int kComputeThreads = Tile::kThreads;        // 256: warpgroups 0, 1
constexpr int kProducers = 128;                        // warpgroup 2
constexpr int kThreads = kComputeThreads + kProducers;
// Registers: the CTA is launched with 168 a thread (384 × 168 = 64,512 of
// the SM's 65,536); the producer warpgroup then gives up all but 88 and the
// two compute warpgroups take 208: 256 × 208 + 128 × 88 = 64,512, exactly
// the launch's allocation (an increase beyond what the decrease frees would
// wait forever).  With 56 or fewer for the producers their code spills.
constexpr int kLaunchRegs = 168, kComputeRegs = 208, kProducerRegs = 88;
static_assert(kComputeThreads * kComputeRegs + kProducers * kProducerRegs <=
                  kThreads * kLaunchRegs,
              "register split within the launch's allocation");
constexpr int kStageFloatsA = Tile::kStageFloatsA;     // 128 × 32
constexpr int kStageFloatsB = Tile::kStageFloatsB;     // 32 × 128
constexpr int kOffB = kStages * kStageFloatsA * 4;
constexpr int kOffBar = kOffB + kStages * kStageFloatsB * 4;
constexpr int kSmemBytes = kOffBar + 2 * kStages * 8 + 16 + 1024;
// Register reallocation between warpgroups (all four warps of a warpgroup
// execute the same one).
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N));
}

template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N));
}

__global__ void __launch_bounds__(kThreads, 1)
    simt_ws_kernel(Problem p, int tiles_m, int tiles_n, int c_vec,
                   WaitCfg wc) {
  griddep_wait();  // A, B and C may belong to the kernel before
  p.A += blockIdx.z * p.sA;
  p.B += blockIdx.z * p.sB;
  p.C += blockIdx.z * p.sC;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* As = reinterpret_cast<float*>(smem);
  float* Bs = reinterpret_cast<float*>(smem + kOffB);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  volatile int* abort = reinterpret_cast<volatile int*>(bars + 2 * kStages);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[kStages + s]); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int tm, tn;
  tile_coords<8>(blockIdx.x, tiles_m, tiles_n, tm, tn);
  const int bm = tm * kBM, bn = tn * kBN;
  const int nk = (p.K + kBK - 1) / kBK;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), kProducers);
      mbar_init(empty(s), kComputeThreads / 32);
    }
    *abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (tid >= kComputeThreads) {
    // ---------------------------------------------------------- producers
    setmaxnreg_dec<kProducerRegs>();
    // per stage each of the 128 producer threads copies 8 chunks of A
    // (rows pt/8 + 16i, chunk pt % 8 of the row's 8, swizzled as FfmaTile
    // reads) and 8 of B (row pt/32 + 4i, chunk pt % 32 of the row's 32)
    const int pt = tid - kComputeThreads;
    const long long ext_a = matrix_extent_bytes(p.M, p.K, p.lda);
    const long long ext_b = matrix_extent_bytes(p.K, p.N, p.ldb);
    (void)ext_a, (void)ext_b;
    const int ca = pt & 7, ra = pt >> 3;
    const int cb = pt & 31, rb = pt >> 5;
    if (!(wc.debug & kDebugStallProducer)) {
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % kStages;
        if (kt >= kStages &&
            !bounded_wait(empty(s), ((kt / kStages) - 1) & 1, wc.limit, abort,
                          0u)) {
          *abort = 1;
          if (pt == 0) record_status(wc.status, kStatusTimeoutEmpty);
          break;
        }
        const int k0 = kt * kBK;
        float* as = As + s * kStageFloatsA;
        float* bs = Bs + s * kStageFloatsB;
        const int gk = k0 + 4 * ca;
        const int abytes = gk < p.K ? 4 * min(4, p.K - gk) : 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int m = ra + 16 * i, gm = bm + m;
          const int bytes = gm < p.M ? abytes : 0;
          const float* src = bytes ? p.A + (long long)gm * p.lda + gk : p.A;
          cp16_checked(as + m * kBK + ((ca ^ a_swizzle<kBK>(m)) * 4), as,
                       kStageFloatsA, src, bytes, p.A, ext_a, p.status);
        }
        const int gn = bn + 4 * cb;
        const int bcols = gn < p.N ? 4 * min(4, p.N - gn) : 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int k = rb + 4 * i;
          const int bytes = k0 + k < p.K ? bcols : 0;
          const float* src =
              bytes ? p.B + (long long)(k0 + k) * p.ldb + gn : p.B;
          cp16_checked(bs + k * kBN + 4 * cb, bs, kStageFloatsB, src, bytes,
                       p.B, ext_b, p.status);
        }
        cp_async_mbar_arrive_noinc(full(s));
      }
    }
    cp_async_wait<0>();  // this thread's copies land before it leaves
  } else {
    // ---------------------------------------------------------- compute
    setmaxnreg_inc<kComputeRegs>();
    Tile tile;
    tile.init(tid);
    Tile::Acc acc;
    Tile::zero(acc);
    bool ok = true;
    for (int kt = 0; kt < nk; ++kt) {
      const int s = kt % kStages;
      if (!bounded_wait(full(s), (kt / kStages) & 1, wc.limit, abort, 0u)) {
        *abort = 1;
        record_status(wc.status, kStatusTimeoutFull);
        ok = false;
        break;
      }
      tile.compute(As + s * kStageFloatsA, Bs + s * kStageFloatsB, acc,
                   p.status);
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(s));
    }
    if (ok && !*abort) tile.store(p, bm, bn, c_vec != 0, acc);
  }
}

}  // namespace simt_ws

namespace {

cudaError_t launch_ws(const Problem& p, bool c_vec, const WaitCfg& wc,
                      cudaStream_t stream) {
  using namespace simt_ws;
  auto fn = simt_ws_kernel;
  cudaError_t e =
      ensure_smem_attr(reinterpret_cast<const void*>(fn), kSmemBytes);
  if (e != cudaSuccess) return e;
  const int tiles_m = (p.M + kBM - 1) / kBM, tiles_n = (p.N + kBN - 1) / kBN;
  const long long grid = (long long)tiles_m * tiles_n;
  if (grid > 0x7fffffffLL || p.batch < 1 || p.batch > 65535)
    return cudaErrorInvalidConfiguration;
  return launch_pdl(fn, dim3((unsigned)grid, 1, (unsigned)p.batch),
                    dim3(kThreads), kSmemBytes, stream, p, tiles_m, tiles_n,
                    (int)c_vec, wc);
}

template <int BM, int BN, int BK, int STAGES, bool VEC, int MINB,
          bool AKM = false, bool TA = false, bool TB = false>
cudaError_t launch_cfg(const Problem& p, bool c_vec, cudaStream_t stream) {
  using K = SimtKernel<BM, BN, BK, STAGES, VEC, AKM, TA, TB>;
  auto fn = simt_gemm_kernel<BM, BN, BK, STAGES, VEC, MINB, AKM, TA, TB>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(fn),
                                   K::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int tiles_m = (p.M + BM - 1) / BM, tiles_n = (p.N + BN - 1) / BN;
  const long long grid = (long long)tiles_m * tiles_n;
  if (grid > 0x7fffffffLL || p.batch < 1 || p.batch > 65535)
    return cudaErrorInvalidConfiguration;
  return launch_pdl(fn, dim3((unsigned)grid, 1, (unsigned)p.batch),
                    dim3(K::kThreads), K::kSmemBytes, stream, p, tiles_m,
                    tiles_n, (int)c_vec);
}

// Transposed operands: one tile configuration (128 x 128 x 32, 4 stages).
template <bool VEC>
cudaError_t launch_trans(const Problem& p, bool c_vec, cudaStream_t stream) {
  if (p.transA && p.transB)
    return launch_cfg<128, 128, 32, 4, VEC, 1, false, true, true>(p, c_vec,
                                                                  stream);
  if (p.transA)
    return launch_cfg<128, 128, 32, 4, VEC, 1, false, true, false>(p, c_vec,
                                                                   stream);
  return launch_cfg<128, 128, 32, 4, VEC, 1, false, false, true>(p, c_vec,
                                                                 stream);
}

template <bool VEC>
cudaError_t launch_vec(const Problem& p, int cfg, bool c_vec,
                       const WaitCfg& wc, cudaStream_t stream) {
  switch (cfg) {
    case kSimt128x64x16:
      return launch_cfg<128, 64, 16, 4, VEC, 3>(p, c_vec, stream);
    case kSimt64x64x16:
      return launch_cfg<64, 64, 16, 4, VEC, 4>(p, c_vec, stream);
    case kSimt128x128x16Occ1:
      return launch_cfg<128, 128, 16, 4, VEC, 1>(p, c_vec, stream);
    case kSimt128x128x32Occ1:
      return launch_cfg<128, 128, 32, 4, VEC, 1>(p, c_vec, stream);
    case kSimt128x128x16Occ1S6:
      return launch_cfg<128, 128, 16, 6, VEC, 1>(p, c_vec, stream);
    case kSimtKm128x128x32Occ1:
      // 16-byte copies of A need VEC (aligned A, lda % 4 == 0)
      return VEC ? launch_cfg<128, 128, 32, 4, true, 1, true>(p, c_vec, stream)
                 : launch_cfg<128, 128, 32, 4, false, 1>(p, c_vec, stream);
    case kSimtWs128x128x32:
      return VEC ? launch_ws(p, c_vec, wc, stream)
                 : launch_cfg<128, 128, 32, 4, false, 1>(p, c_vec, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace


cudaError_t launch_simt(const Problem& p, int cfg, bool vec, bool c_vec,
                        const WaitCfg& wc, cudaStream_t stream) {
  if (p.transA || p.transB)
    return vec ? launch_trans<true>(p, c_vec, stream)
               : launch_trans<false>(p, c_vec, stream);
  return vec ? launch_vec<true>(p, cfg, c_vec, wc, stream)
             : launch_vec<false>(p, cfg, c_vec, wc, stream);
}

}  // namespace gemm_f32_impl
