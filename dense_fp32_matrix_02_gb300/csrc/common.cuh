// Shared device helpers for the gemm_f32 kernels: inline-PTX wrappers for
// cp.async, mbarrier and TMA, the kernel status word and the launch-side
// description of one GEMM problem.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gemm_f32_impl {

// Status word bits written by kernels (read and cleared by the host).
enum : unsigned int {
  kStatusTimeoutFull = 1u,   // a consumer gave up waiting for a full stage
  kStatusTimeoutEmpty = 2u,  // the producer gave up waiting for an empty stage
  kStatusTimeoutDrain = 4u,  // copies still in flight when giving up
  kStatusTimeoutMma = 8u,    // tensor-core completion wait gave up
  kStatusBounds = 16u,       // checked build: an index out of its extent
};

// Debug flags passed to the pipelined kernels (tests only).
enum : unsigned int {
  kDebugStallProducer = 1u,  // producer issues no copies: consumers time out
};

// One problem as the kernels see it.  Leading dimensions in elements.
// Batched calls add per-matrix element strides; a kernel launched with
// gridDim.z = batch handles matrix blockIdx.z.  transA / transB: the operand
// is stored transposed (A as K×M with row stride lda, B as N×K with ldb);
// storeT: the product is written to C transposed.
struct Problem {
  int M, N, K;
  const float* A;
  long long lda;
  const float* B;
  long long ldb;
  float* C;
  long long ldc;
  long long sA = 0, sB = 0, sC = 0;  // batch strides (elements)
  int batch = 1;
  int transA = 0, transB = 0;
  // store Cᵀ (row n of the stored matrix = column n of the computed tile)
  int storeT = 0;
  // fused epilogue: C = act(A·B + bias), bias indexed by column (or NULL)
  const float* bias = nullptr;
  int act = 0;  // 0 identity, 1 GELU
  // kernel status word (the checked build reports out-of-extent indices)
  unsigned int* status = nullptr;
};

enum : int { kActNone = 0, kActGelu = 1 };

// act(v + bias[col]): GELU(x) = x·Φ(x) = x/2·(1 + erf(x/√2)).
__device__ __forceinline__ float epilogue_act(float v, int act) {
  if (act == kActGelu) v = 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
  return v;
}

__device__ __forceinline__ float apply_epilogue(float v, const float* bias,
                                                int act, int col) {
  if (bias) v += bias[col];
  return epilogue_act(v, act);
}

// The operands as plain row-major arrays, for the tensor kernels' repair of
// non-finite outputs: element (m, k) of the product's left operand is
// A[m·lda + k] (A[k·lda + m] when transA), element (k, n) of the right one
// B[k·ldb + n] (B[n·ldb + k] when transB); matrix z of a batch starts sA,
// sB elements further.
struct RawOperands {
  const float* A;
  long long lda, sA;
  const float* B;
  long long ldb, sB;
  int transA, transB;
};

// Σ_k a(m, k)·b(k, n) over k in [k0, k1), ascending, with fmaf: the IEEE
// single-precision value of one element of the product (o.A, o.B already
// at the matrix of the batch in question).
//
// The three-TF32 split cannot follow IEEE arithmetic when an operand is
// infinite: x = ±Inf gives small = Inf − Inf = NaN, so every output that
// operand reaches comes out NaN, where IEEE gives ±Inf (or NaN only for
// Inf·0 or Inf − Inf).  Finite operands never produce a NaN there, so an
// output that is NaN has a non-finite operand in its row of A or column of
// B, and its IEEE value is non-finite too; the tensor kernels recompute
// exactly those elements with this loop before storing them (no cost on
// the main loop: one compare per output and one warp vote in the
// epilogue, and the loop runs only where a NaN appeared).
__device__ __forceinline__ float ieee_dot(const RawOperands& o, int m, int n,
                                          int k0, int k1) {
  const float* a = o.A;
  const float* b = o.B;
  float s = 0.f;
  for (int k = k0; k < k1; ++k) {
    const float x = o.transA ? a[(long long)k * o.lda + m]
                             : a[(long long)m * o.lda + k];
    const float y = o.transB ? b[(long long)n * o.ldb + k]
                             : b[(long long)k * o.ldb + n];
    s = fmaf(x, y, s);
  }
  return s;
}

// true if any of the CNT values (fp32 bit patterns) is a NaN.
template <int CNT>
__device__ __forceinline__ bool any_nan(const uint32_t (&v)[CNT]) {
  bool any = false;
#pragma unroll
  for (int r = 0; r < CNT; ++r) any |= (v[r] & 0x7fffffffu) > 0x7f800000u;
  return any;
}

// Bounded-wait configuration shared by all pipelined kernels.
struct WaitCfg {
  long long limit;        // ns of %globaltimer before a wait gives up
  unsigned int debug;     // kDebug* bits
  unsigned int* status;   // device status word
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- cp.async
// 16-byte copy global -> shared; bytes beyond src_bytes (0..16) are zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src,
                                           int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst),
               "l"(src), "r"(src_bytes)
               : "memory");
}

// 4-byte copy global -> shared; src_bytes 0 writes a zero.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src,
                                          int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst),
               "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Arrive on the mbarrier once every cp.async this thread issued so far has
// landed (the barrier's expected count includes this arrival: .noinc).
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(
                   bar)
               : "memory");
}

// ---------------------------------------------------------------- shared loads
__device__ __forceinline__ float4 lds128(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(
          bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar,
                                                      uint32_t bytes) {
  asm volatile(
      "{\n .reg .b64 st;\n"
      " mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

// One non-blocking probe of phase `parity`; true once that phase completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may sleep up to `hint_ns` waiting for the
// phase instead of returning at once; it wakes when the phase completes.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar,
                                                    uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}

// Bounded wait on one phase of an mbarrier: false once the CTA abort flag
// (if given) is raised or `limit_ns` of %globaltimer time have passed.
// sleep_ns > 0 lets each probe suspend the thread until the phase completes
// (for at most sleep_ns) instead of polling, leaving issue slots to the
// warps that compute; 0 polls, for single-thread roles (TMA producer, MMA
// issuer) that must react at once.
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity,
                                             long long limit_ns,
                                             volatile int* abort,
                                             uint32_t sleep_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (sleep_ns ? mbar_try_wait_sleep(bar, parity, sleep_ns)
                 : mbar_try_wait(bar, parity))
      return true;
    if (sleep_ns || (i & 15u) == 0) {
      if (abort && *abort) return false;
      if ((long long)(globaltimer_ns() - t0) > limit_ns) return false;
    }
  }
}

// ------------------------------------------------ thread-block clusters
// This CTA's rank within its cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}

// Barrier over every thread of every CTA in the cluster: shared-memory
// writes made before it (release) are visible to the cluster's threads
// after it (acquire).  Each warp must reach it converged.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n"
      "barrier.cluster.wait.acquire.aligned;\n" ::
          : "memory");
}

// The shared::cluster address of this CTA's shared address `addr` as seen
// in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n"
               : "=r"(r)
               : "r"(addr), "r"(rank));
  return r;
}

// (volatile, so it stays after the cluster barrier before it; no memory
// clobber, so the arithmetic between such loads does not order them)
__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];\n"
               : "=r"(v)
               : "r"(addr)
               : "memory");
  return v;
}

// ------------------------------------------------ programmatic launch
// A kernel launched with programmatic stream serialization may start while
// the kernel before it in the stream is still running; griddep_wait blocks
// until that kernel has completed and its memory operations are visible, so
// every thread calls it before touching global memory the earlier kernel
// may write or read.  Without that launch attribute it returns at once.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// Lets the next kernel in the stream (launched programmatically) be
// scheduled before this one ends; it still waits in griddep_wait.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// ---------------------------------------------------------------- TMA
// 2-D tiled bulk tensor load into shared memory, completion counted on the
// mbarrier in transaction bytes.  c0 is the innermost coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap,
                                            uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%3, %4}], [%2];\n" ::"r"(dst),
      "l"(tmap), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// 3-D tiled bulk tensor load (c0 innermost, c2 the batch index).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap,
                                            uint32_t bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%3, %4, %5}], [%2];\n" ::"r"(dst),
      "l"(tmap), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// 2-D tiled bulk tensor store from shared memory (c0 innermost); elements
// outside the tensor are not written.  Tracked by the issuing thread's
// bulk async-groups.
__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src,
                                             int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], "
      "[%1];\n" ::"l"(tmap),
      "r"(src), "r"(c0), "r"(c1)
      : "memory");
}

// The same for a 3-D tensor (c2: the batch coordinate).
__device__ __forceinline__ void tma_store_3d(const void* tmap, uint32_t src,
                                             int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, "
      "%4}], [%1];\n" ::"l"(tmap),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}

// Waits until at most N of this thread's bulk groups are still reading
// their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;\n" ::"n"(N) : "memory");
}

// Waits until at most N of this thread's bulk groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ void record_status(unsigned int* status,
                                              unsigned int bit) {
  if (status) atomicOr(status, bit);
}

// ------------------------------------------------ checked build
// Built with GEMM_F32_BOUNDS_CHECK=1 (libgemm_f32_debug.so), the FFMA and
// tensor kernels check every shared-memory, tensor-memory and global index
// they compute against the extent it must lie in (the stage buffer, the
// TMEM allocation, the matrix); a failed check sets kStatusBounds in the
// status word and the access is skipped, so the kernel neither faults nor
// touches memory it does not own.  It stands in for a memory checker.  In
// the normal build every check is the constant true and compiles away.
#ifndef GEMM_F32_BOUNDS_CHECK
#define GEMM_F32_BOUNDS_CHECK 0
#endif

// [p, p + bytes) inside [base, base + extent)?  (generic addresses: global
// memory, or shared memory through a generic pointer)
__device__ __forceinline__ bool span_ok(const void* p, long long bytes,
                                        const void* base, long long extent,
                                        unsigned int* status) {
#if GEMM_F32_BOUNDS_CHECK
  const long long off = reinterpret_cast<const char*>(p) -
                        reinterpret_cast<const char*>(base);
  if (off < 0 || off + bytes > extent) {
    record_status(status, kStatusBounds);
    return false;
  }
#else
  (void)p, (void)bytes, (void)base, (void)extent, (void)status;
#endif
  return true;
}

// The same for a shared-memory address (state space offset).
__device__ __forceinline__ bool smem_span_ok(uint32_t addr, int bytes,
                                             uint32_t base, int extent,
                                             unsigned int* status) {
#if GEMM_F32_BOUNDS_CHECK
  if (addr < base || addr + (uint32_t)bytes > base + (uint32_t)extent) {
    record_status(status, kStatusBounds);
    return false;
  }
#else
  (void)addr, (void)bytes, (void)base, (void)extent, (void)status;
#endif
  return true;
}

// A tensor-memory access of `cols` columns at taddr (lane in bits 31..16,
// column in 15..0) inside an allocation of `alloc_cols` columns at `tmem`,
// by a warp allowed lanes [32·q, 32·q + 32).
__device__ __forceinline__ bool tmem_span_ok(uint32_t taddr, int cols,
                                             uint32_t tmem, int alloc_cols,
                                             int q, unsigned int* status) {
#if GEMM_F32_BOUNDS_CHECK
  const uint32_t col = (taddr & 0xffffu) - (tmem & 0xffffu);
  const uint32_t lane = taddr >> 16;
  if ((taddr & 0xffffu) < (tmem & 0xffffu) ||
      col + (uint32_t)cols > (uint32_t)alloc_cols ||
      lane != (uint32_t)(32 * q)) {
    record_status(status, kStatusBounds);
    return false;
  }
#else
  (void)taddr, (void)cols, (void)tmem, (void)alloc_cols, (void)q,
      (void)status;
#endif
  return true;
}

// Bytes from the first element of a rows × cols matrix with row stride ld
// (elements) to one past its last: the extent its elements lie in.
__host__ __device__ __forceinline__ long long matrix_extent_bytes(
    long long rows, long long cols, long long ld) {
  return rows > 0 && cols > 0 ? 4 * ((rows - 1) * ld + cols) : 0;
}

// Tile order: walks GROUP tile-rows at a time so concurrently running CTAs
// share A row-panels and B column-panels in L2.
template <int GROUP>
__device__ __forceinline__ void tile_coords(int linear, int tiles_m,
                                            int tiles_n, int& tm, int& tn) {
  const int per_group = GROUP * tiles_n;
  const int g = linear / per_group;
  const int first_m = g * GROUP;
  const int rows = min(tiles_m - first_m, GROUP);
  const int in_group = linear - g * per_group;
  tm = first_m + in_group % rows;
  tn = in_group / rows;
}

}  // namespace gemm_f32_impl
