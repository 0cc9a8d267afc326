// Inline-PTX wrappers for the 5th-generation tensor cores (tcgen05) of
// sm_100/sm_103: Tensor Memory (TMEM) allocation, loads and stores, MMA
// issue and completion tracking, and the shared-memory matrix descriptor.
// Written from the public PTX ISA description of the tcgen05 instructions.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace gemm_f32_impl {

// ------------------------------------------------------------ TMEM alloc
// Whole-warp instructions.  The allocated base address (lane 0, first
// column) is written to shared memory at `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile(
      "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
          slot),
      "r"(ncols)
      : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile(
      "tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::
          : "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(
                   taddr),
               "r"(ncols)
               : "memory");
}

// ------------------------------------------------------------ ordering
__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// Makes this thread's generic-proxy shared-memory writes visible to the
// async proxy (TMA, tensor core) once a barrier orders them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// The mbarrier at `bar` receives one arrival once every tcgen05.mma this
// thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];\n" ::"r"(bar)
      : "memory");
}

// The split the tensor core sees when it reads x itself: big = x with its
// 13 low mantissa bits dropped (TF32 truncation), small = x - big (exact).
__device__ __forceinline__ uint32_t tf32_small_of_truncated(float x) {
  const float big = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
  return __float_as_uint(__fsub_rn(x, big));
}

// ------------------------------------------------------------ MMA
// D[tmem] (+)= A[tmem] · B[smem]ᵀ, kind::tf32, one CTA.  `accumulate` = 0
// overwrites D.
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem,
                                            uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor for kind::tf32 with an fp32 accumulator, both
// operands K-major, M×N per instruction (K = 8).
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4)                          // D format: f32
         | (2u << 7)                        // A format: tf32
         | (2u << 10)                       // B format: tf32
         | (0u << 15) | (0u << 16)          // A, B K-major
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// Shared-memory matrix descriptor, K-major, 64-byte swizzle: rows of 64
// bytes, 8-row groups 512 bytes apart.  `addr` is the shared address of the
// first element the instruction reads.
__device__ __forceinline__ uint64_t smem_desc_kmajor_sw64(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                   // leading byte offset (unused)
  d |= (uint64_t)(512 >> 4) << 32;          // stride byte offset: 8 rows
  d |= (uint64_t)1 << 46;                   // descriptor version
  d |= (uint64_t)4 << 61;                   // swizzle: 64 B
  return d;
}

// D[tmem] (+)= A[smem] · B[smem], kind::f16 (bfloat16 or binary16 operands,
// both of the same type), one CTA.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc,
                                           uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor for kind::f16 with an fp32 accumulator.  ab_type:
// 0 binary16, 1 bfloat16 (A and B alike).  A is K-major; B is K-major
// (b_mn_major = false) or N-major, i.e. stored K×N with N contiguous.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int ab_type,
                                                 bool b_mn_major) {
  return (1u << 4)                          // D format: f32
         | ((uint32_t)ab_type << 7)         // A format
         | ((uint32_t)ab_type << 10)        // B format
         | (0u << 15)                       // A K-major
         | ((b_mn_major ? 1u : 0u) << 16)   // B major-ness
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle: 8-row × 128-byte
// atoms (rows 128 bytes apart, 16-byte chunks XOR-ed by the row index mod 8,
// the pattern TMA writes with CU_TENSOR_MAP_SWIZZLE_128B into 1024-byte
// aligned shared memory).  K-major: atoms of 8 M/N rows stacked sbo bytes
// apart along M/N (lbo unused).  MN-major: atom rows run along K; atoms are
// lbo bytes apart along M/N (64 16-bit elements each) and sbo bytes apart
// along K (8 rows each).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr,
                                                    uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);              // start address
  d |= (uint64_t)((lbo_bytes & 0x3FFFFu) >> 4) << 16;   // leading offset
  d |= (uint64_t)((sbo_bytes & 0x3FFFFu) >> 4) << 32;   // stride offset
  d |= (uint64_t)1 << 46;                               // descriptor version
  d |= (uint64_t)2 << 61;                               // swizzle: 128 B
  return d;
}

// ------------------------------------------------------------ TMEM ld/st
// 32 lanes × 32 bits, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, "
      "%7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
      "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]),
      "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// 32 lanes × 32 bits, 8 consecutive columns per thread.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, "
      "%7, %8};\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
      "r"(v[6]), "r"(v[7])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, "
      "%7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]),
        "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]),
        "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
        "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

// 32 lanes × 32 bits, 32 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, "
      "%7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, "
      "%21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]),
        "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]),
        "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
        "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
        "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

}  // namespace gemm_f32_impl
