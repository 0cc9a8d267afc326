// The FP32 FFMA compute cores of the SIMT kernels: a BM×BN block tile,
// BK-deep shared-memory stages, 8×8 register micro-tiles.
//
// Both are the third tiling level of "3 · La mémoire partagée", §3.4 ("Le
// registre comme troisième niveau de tuile"): each thread keeps an 8×8 block
// of C in registers and, per k, does 64 multiply-adds for 16 loaded values.
// FfmaTile issues them as 32 packed two-lane FMAs (PTX fma.rn.f32x2, the
// Blackwell FP32 pair instruction: each lane an fmaf, round to nearest,
// no flush to zero), so the FMA pipe is fed with half the instructions.
//
// FfmaTile keeps A in its global row-major (K-contiguous) order, so TMA can
// copy it without a transpose, and each thread reads A along K with 16-byte
// loads that cover four k steps at once.  FfmaTileT (further down) stores A
// transposed as the page does.
//
// Shared-memory layout of one stage (fp32):
//   A: BM rows × BK floats.  Row m's 16-byte chunk c sits at chunk position
//      c ^ swz(m), swz(m) = ((m·BK·4) >> 7) & (BK/4 − 1).  That is the
//      XOR swizzle of §3.6 ("Le swizzling, l'alternative moderne": address ⊕
//      ((address ≫ s) & m)) with s = 7 and the mask of the row width; for
//      BK = 8, 16, 32 it equals the TMA 32-, 64- and 128-byte swizzle modes,
//      so the TMA kernel fills the very same layout.
//   B: BK rows × BN floats, unswizzled (a warp reads contiguous chunks).
//
// Thread placement: warps form (BM/64) × (BN/32); a warp covers 64 rows ×
// 32 columns with lanes as 8 (M) × 4 (N).  Lane (lm, ln) of warp (wm, wn)
// owns rows wm·64 + lm + 8i (i < 8) and columns wn·32 + ln·4 + 16g + j
// (g < 2, j < 4).  The eight rows one load instruction touches (lm = 0..7,
// same i) land in eight different bank groups under the swizzle, and the
// four B chunks of one instruction are adjacent: no bank conflicts.
#pragma once

#include "common.cuh"

namespace gemm_f32_impl {

template <int BK>
__host__ __device__ constexpr int a_swizzle(int m) {
  return ((m * BK * 4) >> 7) & (BK / 4 - 1);
}

// Two fp32 values in one 64-bit register pair (lo = first).
__device__ __forceinline__ unsigned long long pack_f32x2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void unpack_f32x2(unsigned long long v, float& lo,
                                             float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// d = a·b + d in each of the two lanes.
__device__ __forceinline__ void fma_f32x2(unsigned long long& d,
                                          unsigned long long a,
                                          unsigned long long b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

// The 16 bytes at p, a float4 inside the `floats`-element buffer at base
// (checked build: zeros and kStatusBounds when outside it).
__device__ __forceinline__ float4 lds4_checked(const float* p,
                                               const float* base, int floats,
                                               unsigned int* st) {
  return span_ok(p, 16, base, 4LL * floats, st)
             ? *reinterpret_cast<const float4*>(p)
             : make_float4(0.f, 0.f, 0.f, 0.f);
}

// Stores of the 8×8 block: v to C at p (float4 or one float), inside the
// matrix (checked build: skipped and kStatusBounds when outside it).
__device__ __forceinline__ void stg4_checked(float* p, float4 v,
                                             const Problem& pr) {
  if (span_ok(p, 16, pr.C, matrix_extent_bytes(pr.M, pr.N, pr.ldc),
              pr.status))
    *reinterpret_cast<float4*>(p) = v;
}

__device__ __forceinline__ void stg1_checked(float* p, float v,
                                             const Problem& pr) {
  if (span_ok(p, 4, pr.C, matrix_extent_bytes(pr.M, pr.N, pr.ldc),
              pr.status))
    *p = v;
}

template <int BM, int BN, int BK>
struct FfmaTile {
  static_assert(BM % 64 == 0 && BN % 32 == 0, "warp tile is 64 x 32");
  static_assert(BK == 8 || BK == 16 || BK == 32, "BK in {8, 16, 32}");
  static constexpr int kWarpsM = BM / 64;
  static constexpr int kWarpsN = BN / 32;
  static constexpr int kThreads = kWarpsM * kWarpsN * 32;
  static constexpr int kStageFloatsA = BM * BK;
  static constexpr int kStageFloatsB = BK * BN;
  static constexpr int kStageBytes = 4 * (kStageFloatsA + kStageFloatsB);
  // The 8×8 accumulators as pairs: acc[i][p] holds columns 2p and 2p + 1
  // of row i (in the column order of `store`).
  using Acc = unsigned long long[8][4];

  static __device__ __forceinline__ void zero(Acc& acc) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0ull;  // two +0.0f
  }

  // Per-thread fixed offsets (floats) into a stage.
  int a_row_off;      // (wm*64 + lm) * BK
  int a_chunk[BK / 4];  // ((q ^ swz) * 4)
  int b_col_off;      // wn*32 + ln*4
  int row0;           // wm*64 + lm (tile-relative)
  int col0;           // wn*32 + ln*4 (tile-relative)

  __device__ __forceinline__ void init(int tid) {
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = warp / kWarpsN, wn = warp % kWarpsN;
    const int lm = lane >> 2, ln = lane & 3;
    row0 = wm * 64 + lm;
    col0 = wn * 32 + ln * 4;
    a_row_off = row0 * BK;
    const int sw = a_swizzle<BK>(row0);
#pragma unroll
    for (int q = 0; q < BK / 4; ++q) a_chunk[q] = (q ^ sw) * 4;
    b_col_off = col0;
  }

  // acc += A_stage · B_stage for this thread's 8×8 block.  `st`: the
  // status word the checked build reports an out-of-stage index to.
  __device__ __forceinline__ void compute(const float* __restrict__ As,
                                          const float* __restrict__ Bs,
                                          Acc& acc,
                                          unsigned int* st = nullptr) const {
    const float* a_base = As + a_row_off;
    const float* b_base = Bs + b_col_off;
#pragma unroll
    for (int q = 0; q < BK / 4; ++q) {
      float4 a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        a[i] = lds4_checked(a_base + i * 8 * BK + a_chunk[q], As,
                            kStageFloatsA, st);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int k = 4 * q + kk;
        const float4 b0 = lds4_checked(b_base + k * BN, Bs, kStageFloatsB, st);
        const float4 b1 =
            lds4_checked(b_base + k * BN + 16, Bs, kStageFloatsB, st);
        const unsigned long long bp[4] = {
            pack_f32x2(b0.x, b0.y), pack_f32x2(b0.z, b0.w),
            pack_f32x2(b1.x, b1.y), pack_f32x2(b1.z, b1.w)};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float av = kk == 0 ? a[i].x
                           : kk == 1 ? a[i].y
                           : kk == 2 ? a[i].z
                                     : a[i].w;
          const unsigned long long aa = pack_f32x2(av, av);
#pragma unroll
          for (int j = 0; j < 4; ++j) fma_f32x2(acc[i][j], aa, bp[j]);
        }
      }
    }
  }

  // Writes the thread's 8×8 block to C (tile origin bm, bn), overwriting.
  // Interior tiles with a 16-byte-aligned C and ldc % 4 == 0 use float4
  // stores; every other case checks each element against M and N.
  __device__ __forceinline__ void store(const Problem& p, int bm, int bn,
                                        bool c_vec, const Acc& acc2) const {
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        unpack_f32x2(acc2[i][j], acc[i][2 * j], acc[i][2 * j + 1]);
    const bool interior = (bm + BM <= p.M) && (bn + BN <= p.N);
    const bool epi = p.bias != nullptr || p.act != kActNone;
    // the bias of the thread's 8 columns, loaded once (C stores may alias it)
    float bcol[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = bn + col0 + 16 * (j >> 2) + (j & 3);
      bcol[j] = (p.bias != nullptr && c < p.N) ? p.bias[c] : 0.f;
    }
    auto val = [&](int i, int j, int) {
      if (!epi) return acc[i][j];
      return epilogue_act(p.bias != nullptr ? acc[i][j] + bcol[j] : acc[i][j],
                          p.act);
    };
    if (interior && c_vec) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float* crow = p.C + (long long)(bm + row0 + 8 * i) * p.ldc + bn + col0;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const int c = bn + col0 + 16 * g;
          stg4_checked(crow + 16 * g,
                       make_float4(val(i, 4 * g, c), val(i, 4 * g + 1, c + 1),
                                   val(i, 4 * g + 2, c + 2),
                                   val(i, 4 * g + 3, c + 3)),
                       p);
        }
      }
      return;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = bm + row0 + 8 * i;
      if (r >= p.M) continue;
      float* crow = p.C + (long long)r * p.ldc;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int c = bn + col0 + 16 * g;
        if (c_vec && c + 3 < p.N) {
          stg4_checked(crow + c,
                       make_float4(val(i, 4 * g, c), val(i, 4 * g + 1, c + 1),
                                   val(i, 4 * g + 2, c + 2),
                                   val(i, 4 * g + 3, c + 3)),
                       p);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (c + j < p.N) stg1_checked(crow + c + j, val(i, 4 * g + j, c + j), p);
        }
      }
    }
  }
};

// Same 8×8 register tile with A stored transposed, as in "3 · La mémoire
// partagée", §3.4 (As[BK][BM]): per k a thread reads its eight A values as
// two 16-byte loads and its eight B values as two more, so 4 shared loads
// feed 64 multiply-adds (32 packed two-lane FMAs, as in FfmaTile) and only
// 16 operand registers are live per k step.
//
// Shared-memory layout of one stage (fp32):
//   A: BK rows (k) × BM floats (m).  The 16-byte chunk c = m/4 of row k sits
//      at chunk position c ^ (k & 7) (the XOR swizzle of §3.6 with the k
//      index as the "address ≫ s" part).  A copy instruction of a warp
//      writes 4 rows m × 8 values k, eight different k in eight different
//      chunk positions, and a read instruction takes eight adjacent chunks
//      of one k row: both are free of bank conflicts.
//   B: BK rows × BN floats, unswizzled.
// Thread placement: warps (BM/64) × (BN/32), lanes 8 (M) × 4 (N).  Lane
// (lm, ln) of warp (wm, wn) owns rows wm·64 + lm·4 + 32h + r (h < 2, r < 4)
// and columns wn·32 + ln·4 + 16g + j (g < 2, j < 4).
//
// BSWZ = true (B stored transposed in global memory, so its tile arrives
// one float at a time): B's 16-byte chunk c of row k sits at c ^ (k & 7),
// the same swizzle as A, and the thread's two B chunks are read from there.
template <int BM, int BN, int BK, bool BSWZ = false>
struct FfmaTileT {
  static_assert(BM % 64 == 0 && BN % 32 == 0, "warp tile is 64 x 32");
  static_assert(BK % 8 == 0 && BK <= 32, "BK in {8, 16, 24, 32}");
  static constexpr int kWarpsM = BM / 64;
  static constexpr int kWarpsN = BN / 32;
  static constexpr int kThreads = kWarpsM * kWarpsN * 32;
  static constexpr int kStageFloatsA = BM * BK;
  static constexpr int kStageFloatsB = BK * BN;
  static constexpr int kStageBytes = 4 * (kStageFloatsA + kStageFloatsB);
  // The 8×8 accumulators as pairs: acc[i][p] holds columns 2p and 2p + 1
  // of row_of(i) (in the column order of `store`).
  using Acc = unsigned long long[8][4];

  static __device__ __forceinline__ void zero(Acc& acc) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0ull;  // two +0.0f
  }

  int a_off[8];  // (c ^ g) * 4 for g = 0..7, c = row0 / 4
  int b_off[BSWZ ? 8 : 1];  // (c ^ g) * 4 for g = 0..7, c = col0 / 4
  int b_col_off;
  int row0, col0;

  // Offset (floats) of element (k, n) in a B stage.
  static __device__ __forceinline__ int b_index(int k, int n) {
    if (BSWZ) return k * BN + ((((n >> 2) ^ (k & 7)) << 2) | (n & 3));
    return k * BN + n;
  }

  // Offset (floats) of element (k, m) in an A stage.
  static __device__ __forceinline__ int a_index(int k, int m) {
    return k * BM + ((((m >> 2) ^ (k & 7)) << 2) | (m & 3));
  }

  __device__ __forceinline__ void init(int tid) {
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = warp / kWarpsN, wn = warp % kWarpsN;
    const int lm = lane >> 2, ln = lane & 3;
    row0 = wm * 64 + lm * 4;
    col0 = wn * 32 + ln * 4;
    const int c = row0 >> 2;
#pragma unroll
    for (int g = 0; g < 8; ++g) a_off[g] = (c ^ g) << 2;
    b_col_off = col0;
    if (BSWZ) {
      const int cb = col0 >> 2;
#pragma unroll
      for (int g = 0; g < 8; ++g) b_off[g] = (cb ^ g) << 2;
    }
  }

  __device__ __forceinline__ void compute(const float* __restrict__ As,
                                          const float* __restrict__ Bs,
                                          Acc& acc,
                                          unsigned int* st = nullptr) const {
    const float* b_base = Bs + b_col_off;
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      const float* a_row = As + k * BM + a_off[k & 7];
      const float4 a0 = lds4_checked(a_row, As, kStageFloatsA, st);
      const float4 a1 = lds4_checked(a_row + 32, As, kStageFloatsA, st);
      float4 b0, b1;
      if (BSWZ) {
        // col0 / 4 has bit 2 clear, so the second chunk (col0 + 16) sits at
        // the first one's position with bit 2 flipped: offset ^ 16 floats
        const float* b_row = Bs + k * BN;
        b0 = lds4_checked(b_row + b_off[k & 7], Bs, kStageFloatsB, st);
        b1 = lds4_checked(b_row + (b_off[k & 7] ^ 16), Bs, kStageFloatsB, st);
      } else {
        b0 = lds4_checked(b_base + k * BN, Bs, kStageFloatsB, st);
        b1 = lds4_checked(b_base + k * BN + 16, Bs, kStageFloatsB, st);
      }
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const unsigned long long bp[4] = {
          pack_f32x2(b0.x, b0.y), pack_f32x2(b0.z, b0.w),
          pack_f32x2(b1.x, b1.y), pack_f32x2(b1.z, b1.w)};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const unsigned long long aa = pack_f32x2(av[i], av[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) fma_f32x2(acc[i][j], aa, bp[j]);
      }
    }
  }

  __device__ __forceinline__ int row_of(int i) const {
    return row0 + (i & 3) + ((i >> 2) << 5);
  }

  __device__ __forceinline__ void store(const Problem& p, int bm, int bn,
                                        bool c_vec, const Acc& acc2) const {
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        unpack_f32x2(acc2[i][j], acc[i][2 * j], acc[i][2 * j + 1]);
    const bool interior = (bm + BM <= p.M) && (bn + BN <= p.N);
    const bool epi = p.bias != nullptr || p.act != kActNone;
    // the bias of the thread's 8 columns, loaded once (C stores may alias it)
    float bcol[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = bn + col0 + 16 * (j >> 2) + (j & 3);
      bcol[j] = (p.bias != nullptr && c < p.N) ? p.bias[c] : 0.f;
    }
    auto val = [&](int i, int j, int) {
      if (!epi) return acc[i][j];
      return epilogue_act(p.bias != nullptr ? acc[i][j] + bcol[j] : acc[i][j],
                          p.act);
    };
    if (interior && c_vec) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float* crow = p.C + (long long)(bm + row_of(i)) * p.ldc + bn + col0;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const int c = bn + col0 + 16 * g;
          stg4_checked(crow + 16 * g,
                       make_float4(val(i, 4 * g, c), val(i, 4 * g + 1, c + 1),
                                   val(i, 4 * g + 2, c + 2),
                                   val(i, 4 * g + 3, c + 3)),
                       p);
        }
      }
      return;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = bm + row_of(i);
      if (r >= p.M) continue;
      float* crow = p.C + (long long)r * p.ldc;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int c = bn + col0 + 16 * g;
        if (c_vec && c + 3 < p.N) {
          stg4_checked(crow + c,
                       make_float4(val(i, 4 * g, c), val(i, 4 * g + 1, c + 1),
                                   val(i, 4 * g + 2, c + 2),
                                   val(i, 4 * g + 3, c + 3)),
                       p);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (c + j < p.N) stg1_checked(crow + c + j, val(i, 4 * g + j, c + j), p);
        }
      }
    }
  }
};

}  // namespace gemm_f32_impl
