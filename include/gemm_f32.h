/*
 * gemm_f32 — single-precision matrix multiply C = A·B for NVIDIA GB300
 * (sm_103a), row-major, behind a plain C ABI.
 *
 * The operation (the pages this library implements):
 *   "3 · La mémoire partagée", §3.1 "Le problème que ça résout" defines the
 *   product: every output C[i][j] is the sum over k of A[i][k]·B[k][j],
 *   one multiply and one add per term (2·M·N·K operations), accumulated in
 *   single precision, and written over C (no scaling, no accumulation into
 *   the old C).  "共享内存与同步", section "SharedArray —— 静态共享内存"
 *   (tiled_sgemm) gives the general m, n, k form with row-major float
 *   operands.  §3.3-§3.4 of the first page describe the shared-memory tile
 *   and register micro-tile that the kernels here are built on.
 *
 * Layout: all three matrices are row-major float32 in device memory.
 *   A is M×K with row stride lda (elements), B is K×N with row stride ldb,
 *   C is M×N with row stride ldc.  Element (i, j) of C lives at
 *   C[i*ldc + j].  Only C[i*ldc + j] for i < M, j < N is written; the
 *   padding between N and ldc is left untouched.
 *
 * Ownership: the caller owns A, B and C.  The library never allocates or
 * frees device memory on these calls, never synchronizes the stream and
 * keeps no pointer after the call returns.  Work is queued on `stream`
 * (NULL = the legacy default stream) and is complete when the stream is.
 * C must not overlap A or B (not checked).
 *
 * Errors: every entry point returns a gemm_f32_status and never throws.
 * Nothing is launched unless the call returns GEMM_F32_OK.
 *
 * Thread safety: calls from several host threads are safe; per-device
 * one-time set-up is guarded internally.
 */
#ifndef GEMM_F32_H
#define GEMM_F32_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GEMM_F32_API __attribute__((visibility("default")))
#else
#define GEMM_F32_API
#endif

/* A CUDA stream; binary compatible with cudaStream_t / CUstream. */
typedef struct CUstream_st *gemm_f32_stream_t;

typedef enum {
    GEMM_F32_OK = 0,
    /* M, N or K < 0; lda < K, ldb < N or ldc < N; a NULL pointer for a
     * matrix with at least one element; an unknown algo value. */
    GEMM_F32_ERR_INVALID_ARG = 1,
    /* A forced algorithm whose preconditions do not hold (alignment, sizes,
     * device architecture).  GEMM_F32_ALGO_AUTO never returns this. */
    GEMM_F32_ERR_UNSUPPORTED = 2,
    /* A CUDA runtime error while setting up or launching; the code is
     * available from gemm_f32_last_cuda_error(). */
    GEMM_F32_ERR_CUDA = 3,
    /* A kernel's bounded wait gave up (reported by gemm_f32_device_status). */
    GEMM_F32_ERR_TIMEOUT = 4,
    /* gemm_f32_noalloc: the product needs more split-K scratch than the
     * library's static buffer holds. */
    GEMM_F32_ERR_SCRATCH_LIMIT = 5,
    /* Checked build only (gemm_f32_bounds_checked() == 1): a kernel computed
     * a shared-memory, tensor-memory or global index outside the extent it
     * must lie in and skipped that access (reported by
     * gemm_f32_device_status). */
    GEMM_F32_ERR_BOUNDS = 6
} gemm_f32_status;

typedef enum {
    /* Pick the fastest kernel whose preconditions hold. */
    GEMM_F32_ALGO_AUTO = 0,
    /* FP32 FFMA register-tiled kernel, operands staged by cp.async into a
     * multi-stage swizzled shared-memory ring.  Any pointer alignment and
     * any leading dimension. */
    GEMM_F32_ALGO_SIMT = 1,
    /* FP32 FFMA register-tiled kernel whose operand tiles TMA copies into
     * a 4-stage ring under mbarrier full/empty phases (no per-thread copy
     * instructions, no __syncthreads in the main loop).  Needs A and B
     * 16-byte aligned, lda and ldb multiples of 4, and K >= 1. */
    GEMM_F32_ALGO_TMA = 2,
    /* Tensor-core kernel (tcgen05, TMEM accumulator) computing each product
     * as three TF32 products of a big/small operand split, accumulated in
     * fp32; within the single-precision tolerance for finite inputs.  NaN
     * and ±Inf inputs give the IEEE result: outputs the split turns into
     * NaN (an infinite operand) are recomputed in IEEE single precision
     * before they are stored, so ±Inf stays ±Inf.  Needs A and B
     * 16-byte aligned, lda and ldb multiples of 4, K >= 1 and an sm_10x GPU.
     * GEMM_F32_ALGO_AUTO picks it whenever these hold. */
    GEMM_F32_ALGO_TF32X3 = 3
} gemm_f32_algo;

/*
 * C = A·B.  M, N, K >= 0.  M == 0 or N == 0: returns OK and launches
 * nothing.  K == 0: C[0:M, 0:N] is set to 0 (the empty sum).  On the
 * tensor path, tiles that would leave SMs idle — every tile of a product
 * too small to fill the GPU, or the tiles of a larger product's last,
 * partly filled round — split K over up to 8 CTAs each, which run as one
 * thread-block cluster and add their partial tiles in distributed shared
 * memory in a fixed order: no scratch is needed and results are
 * deterministic.
 */
GEMM_F32_API int gemm_f32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
             const float *B, int64_t ldb, float *C, int64_t ldc,
             gemm_f32_stream_t stream);

/* As gemm_f32, with the kernel family forced by `algo` (gemm_f32_algo). */
GEMM_F32_API int gemm_f32_ex(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                const float *B, int64_t ldb, float *C, int64_t ldc,
                gemm_f32_stream_t stream, int algo);

/* Activations for gemm_f32_bias_act. */
typedef enum {
    GEMM_F32_ACT_NONE = 0,
    /* GELU(x) = x·Φ(x) = x/2·(1 + erf(x/√2)), Φ the standard normal
     * distribution function */
    GEMM_F32_ACT_GELU = 1
} gemm_f32_act;

/*
 * Fused epilogue: C = act(A·B + bias), where bias (length N, device memory,
 * may be NULL) is added to every row.  "Rendre le GPU rapide" names the
 * bias add fused into the matrix multiply and a separate GELU kernel among
 * the things a tuned library does that an unfused pipeline pays for in
 * memory passes; here both run in the multiply's epilogue (or, when K is
 * split, in the reduction), so C is written once.  Scratch and kernel
 * choice as for gemm_f32_ws (workspace may be NULL with 0 bytes).
 */
GEMM_F32_API int gemm_f32_bias_act(int64_t M, int64_t N, int64_t K,
                                   const float *A, int64_t lda,
                                   const float *B, int64_t ldb,
                                   const float *bias, int act, float *C,
                                   int64_t ldc, void *workspace,
                                   int64_t workspace_bytes,
                                   gemm_f32_stream_t stream);

/* Operand forms for gemm_f32_batched. */
typedef enum {
    GEMM_F32_OP_N = 0, /* the operand as stored */
    GEMM_F32_OP_T = 1  /* the operand's transpose (no copy is made) */
} gemm_f32_op;

/*
 * Strided batch of products with optional transposes, without copies
 * ("Rendre le GPU rapide" multiplies activations by transposed weight
 * matrices in its layers; each product is the pages' C = A·B):
 *   for b in [0, batch):  C_b = op(A_b) · op(B_b)
 * where X_b = X + b·strideX (elements).  op(A) is M×K: with opA = N, A_b is
 * stored M×K row-major (lda >= K); with opA = T it is stored K×M (lda >= M)
 * and used transposed.  op(B) is K×N: stored K×N (ldb >= N) or, with
 * opB = T, N×K (ldb >= K).  C_b is M×N (ldc >= N).  Strides may be 0 (the
 * same operand for every product); output matrices must not overlap.
 * batch = 0, M = 0 or N = 0 launches nothing; batch <= 65535.  Kernel
 * choice as for gemm_f32: the 3xTF32 tensor kernel where its layouts allow
 * (16-byte aligned operands, leading dimensions and strides multiples of 4,
 * every form), the FFMA kernel otherwise.  Within the tolerance of gemm_f32
 * for every form.
 */
GEMM_F32_API int gemm_f32_batched(int opA, int opB, int64_t M, int64_t N,
                                  int64_t K, const float *A, int64_t lda,
                                  int64_t strideA, const float *B, int64_t ldb,
                                  int64_t strideB, float *C, int64_t ldc,
                                  int64_t strideC, int64_t batch,
                                  gemm_f32_stream_t stream);

/*
 * As gemm_f32_batched, with caller-lent scratch (`workspace`: 16-byte
 * aligned device memory, or NULL with 0 bytes).  For the form
 * opA = T, opB = N on the tensor kernel, when the workspace holds the
 * transposed copies (M rows of K rounded up to a multiple of 4, one copy
 * per product, or one for all when strideA = 0 or batch = 1, each on a
 * 256-byte boundary), A is first transposed into it by an HBM-bound copy
 * kernel and the product runs as opA = N: this costs one pass over A and
 * saves the tensor kernel the transposition of every A tile in shared
 * memory.  For batch = 1 the rest of the workspace is split-K scratch as
 * in gemm_f32_ws (also for opA = opB = N).  With less scratch, and for the
 * other forms, the call runs as gemm_f32_batched.  The workspace is in use
 * until the stream passes this call.  GEMM_F32_ERR_INVALID_ARG for
 * workspace_bytes < 0 or a NULL workspace with workspace_bytes > 0, and
 * for everything gemm_f32_batched rejects.
 */
GEMM_F32_API int gemm_f32_batched_ws(int opA, int opB, int64_t M, int64_t N,
                                     int64_t K, const float *A, int64_t lda,
                                     int64_t strideA, const float *B,
                                     int64_t ldb, int64_t strideB, float *C,
                                     int64_t ldc, int64_t strideC,
                                     int64_t batch, void *workspace,
                                     int64_t workspace_bytes,
                                     gemm_f32_stream_t stream);

/* Scratch bytes gemm_f32_batched_ws uses at most for these sizes and forms
 * on the current device (0: none; negative: minus a status). */
GEMM_F32_API int64_t gemm_f32_batched_workspace_size(int opA, int opB,
                                                     int64_t M, int64_t N,
                                                     int64_t K,
                                                     int64_t batch);

/* 16-bit operand formats of the mixed-precision products. */
typedef enum {
    GEMM_F32_MIXED_BF16 = 0, /* bfloat16: the upper half of a float32 */
    GEMM_F32_MIXED_F16 = 1   /* IEEE binary16: 5 exponent, 10 stored bits */
} gemm_f32_mixed_type;

/*
 * Mixed-precision product, "Rendre le GPU rapide", "Les Tensor Cores": only
 * the multiply's operands are 16-bit floats; products and sums are fp32
 * and C is fp32.  NOT within gemm_f32's tolerance for fp32 operands (the
 * operands carry 8 or 11 significant bits); exact when the operands and
 * every partial sum are representable, e.g. integers in [-8, 8] with
 * K <= 2^18.  It is a separate entry, never chosen by gemm_f32.
 *
 * gemm_f32_mixed16: A (M×K, lda) and B (K×N, ldb) already hold 16-bit
 * values of `type` (gemm_f32_mixed_type), row-major in device memory, 16-byte
 * aligned, with lda and ldb multiples of 8 (else GEMM_F32_ERR_UNSUPPORTED);
 * C is fp32 M×N (ldc >= N, any alignment).  Tensor cores (tcgen05,
 * kind::f16) with fp32 accumulation in tensor memory; needs an sm_10x GPU.
 * M == 0 or N == 0 launches nothing; K == 0 sets C to 0.
 */
GEMM_F32_API int gemm_f32_mixed16(int type, int64_t M, int64_t N, int64_t K,
                                  const void *A, int64_t lda, const void *B,
                                  int64_t ldb, float *C, int64_t ldc,
                                  gemm_f32_stream_t stream);

/*
 * dst = src rounded to the 16-bit `type` for a rows×cols block of fp32
 * (row stride lds) into 16-bit storage (row stride ldd), both in device
 * memory: round to nearest, ties to even, overflow to ±Inf, binary16
 * subnormals kept; NaN stays NaN.  The pages round bfloat16 the same way
 * (add half a step plus the lowest kept bit, then cut).
 */
GEMM_F32_API int gemm_f32_round16(int type, int64_t rows, int64_t cols,
                                  const float *src, int64_t lds, void *dst,
                                  int64_t ldd, gemm_f32_stream_t stream);

/*
 * The mixed-precision product of fp32 operands: A and B are rounded to
 * `type` (as gemm_f32_round16) into `workspace`, then multiplied as by
 * gemm_f32_mixed16.  Any alignment and any leading dimensions >= the row
 * widths.  `workspace` is 16-byte aligned device memory of at least
 * gemm_f32_mixed_workspace_size(M, N, K) bytes (else
 * GEMM_F32_ERR_INVALID_ARG); it holds the rounded A (M rows of K rounded
 * up to a multiple of 8) and then, from the next 256-byte boundary, the
 * rounded B (K rows of N rounded up likewise), and is in use until the
 * stream passes this call.
 */
GEMM_F32_API int gemm_f32_mixed(int type, int64_t M, int64_t N, int64_t K,
                                const float *A, int64_t lda, const float *B,
                                int64_t ldb, float *C, int64_t ldc,
                                void *workspace, int64_t workspace_bytes,
                                gemm_f32_stream_t stream);

/* Workspace bytes gemm_f32_mixed needs for an M×N×K product (negative
 * status for negative sizes). */
GEMM_F32_API int64_t gemm_f32_mixed_workspace_size(int64_t M, int64_t N,
                                                   int64_t K);

/*
 * How gemm_f32_mixed16 (and gemm_f32_mixed) cut an M×N×K product on the
 * current device, for tests and tuning.  out[0]: tile width in columns
 * (256, or 128 / 64 when N is at most that); out[1]: tiles run whole;
 * out[2]: column strips each remaining tile is cut into (1, 2 or 4: the
 * tiles of the last, partly filled round of the persistent grid, or all of
 * them when there are fewer tiles than SMs); out[3]: persistent CTAs;
 * out[4]: tile rows (256 when K >= 2048, N > 128 and there is a 256 × 256
 * tile for every SM, else 128).  Every unit runs the whole K.  The
 * environment variable GEMM_F32_MIXED_NARROW=0 keeps every tile whole and
 * 256 wide; GEMM_F32_MIXED_BM=128 or 256 forces the tile rows.  Returns
 * GEMM_F32_OK, GEMM_F32_ERR_INVALID_ARG (M or N < 1, K < 0, out NULL) or
 * GEMM_F32_ERR_CUDA.
 */
GEMM_F32_API int gemm_f32_mixed_plan(int64_t M, int64_t N, int64_t K,
                                     int64_t out[5]);

/*
 * FP32 FMA throughput probe (measurement, not part of any product): launches
 * a kernel of independent FMA chains, `iters` loop iterations per thread, on
 * every SM at full residency; `sink` is device memory of at least 256 floats
 * (never written in practice).  Time it on `stream` and divide
 * gemm_f32_ffma_peak_flops(iters) by the time for the FP32 pipe's measured
 * rate, the ceiling of the FFMA kernels.  Launches only; no sync.
 */
GEMM_F32_API int gemm_f32_ffma_peak_launch(int64_t iters, float *sink,
                                           gemm_f32_stream_t stream);

/* Floating-point operations (2 per FMA) one gemm_f32_ffma_peak_launch with
 * `iters` performs on the current device; negative status on error. */
GEMM_F32_API int64_t gemm_f32_ffma_peak_flops(int64_t iters);

/*
 * As gemm_f32 (automatic kernel choice), with caller-owned device scratch
 * that the library may use where a cluster cannot hold a tile's splits:
 * more than 8 splits per tile (a few tiles with a long K).  A second
 * kernel then sums the partial tiles in a fixed order, so results stay
 * deterministic.  gemm_f32_workspace_size is 0 for every other product.
 * `workspace` must be 16-byte aligned device memory of `workspace_bytes`
 * bytes (NULL with 0 is allowed); if it is smaller than
 * gemm_f32_workspace_size(M, N, K) the call runs without splitting.  The
 * workspace is in use until the stream passes this call: calls that may
 * overlap on the GPU need separate workspaces.
 */
GEMM_F32_API int gemm_f32_ws(int64_t M, int64_t N, int64_t K, const float *A,
                             int64_t lda, const float *B, int64_t ldb,
                             float *C, int64_t ldc, void *workspace,
                             int64_t workspace_bytes,
                             gemm_f32_stream_t stream);

/*
 * As gemm_f32_ws, but the split-K scratch is a buffer inside the library
 * itself, so this call allocates no memory at all.  It is for callers that
 * must not allocate device memory: code running inside a framework or
 * server that hands out all device memory from its own pool (a direct
 * cudaMalloc would go around that pool's budget), and latency-critical
 * paths where an allocation's implicit synchronisation and unbounded
 * latency are not acceptable.  The pages have no counterpart to it.
 *
 * The buffer is a static device array of gemm_f32_noalloc_scratch_bytes()
 * (16 MiB) that every GPU holds from the library's first use on it until
 * the process exits.  The first call on each device looks up the buffer's
 * device address (cudaGetSymbolAddress) with that device current; make
 * that first call before any stream capture.  A product whose split needs
 * more scratch than the buffer holds is rejected with
 * GEMM_F32_ERR_SCRATCH_LIMIT (nothing is launched); products that need no
 * split run as gemm_f32 would.  All calls on a device share the buffer and
 * it keeps whatever the last call left there; nothing in it needs to start
 * at zero (every split writes the whole partial tile it later adds), but
 * calls that may overlap on the GPU (different streams, or not yet
 * finished) race on it and must be serialised by the caller.  The device
 * address is looked up once per device and kept for the life of the
 * process: do not call this entry after a cudaDeviceReset of a device it
 * has already run on (the reset unloads the library's device code, and the
 * kept address would no longer name the buffer).
 */
GEMM_F32_API int gemm_f32_noalloc(int64_t M, int64_t N, int64_t K,
                                  const float *A, int64_t lda, const float *B,
                                  int64_t ldb, float *C, int64_t ldc,
                                  gemm_f32_stream_t stream);

/* Capacity in bytes of the static scratch buffer gemm_f32_noalloc uses. */
GEMM_F32_API int64_t gemm_f32_noalloc_scratch_bytes(void);

/* Scratch bytes gemm_f32_ws would use for an M×N×K product on the current
 * device when A, B and C are 16-byte aligned with leading dimensions that
 * are multiples of 4 (the layouts that can use scratch; others need none).
 * 0 = none.  Negative status on error. */
GEMM_F32_API int64_t gemm_f32_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * C = A·B for A, B and C in host memory (row-major, leading dimensions lda,
 * ldb, ldc); page-locked host memory lets the copies run asynchronously and
 * at full speed.  The caller lends device buffers dA (M×K), dB (K×N) and dC
 * (M×N), row-major with leading dimensions K, N and N, and optional split-K
 * scratch as for gemm_f32_ws; the library allocates no memory.  B is copied
 * to the GPU first, then A in row chunks: each chunk is multiplied on
 * `stream` while the next one is being copied, and each finished chunk of C
 * is copied back while the next one is multiplied.  The work starts after
 * what is already queued on `stream`, and `stream` completes once C is in
 * host memory; the host buffers must stay valid until then.  Two copy
 * streams and a set of events per device are created on first use and kept.
 * The pages have no counterpart (they keep data on the GPU).
 */
GEMM_F32_API int gemm_f32_host(int64_t M, int64_t N, int64_t K,
                               const float *hA, int64_t lda, const float *hB,
                               int64_t ldb, float *hC, int64_t ldc, float *dA,
                               float *dB, float *dC, void *workspace,
                               int64_t workspace_bytes,
                               gemm_f32_stream_t stream);

/* The algorithm gemm_f32 with GEMM_F32_ALGO_AUTO would run for these
 * arguments on the current device (no launch).  Negative on bad args. */
GEMM_F32_API int gemm_f32_select_algo(int64_t M, int64_t N, int64_t K, const float *A,
                         int64_t lda, const float *B, int64_t ldb, float *C,
                         int64_t ldc);

/*
 * The automatic plan gemm_f32_ws would run for these arguments and a
 * workspace of gemm_f32_workspace_size bytes on the current device (no
 * launch), for tests and tuning.  out[0]: kernel family (gemm_f32_algo);
 * out[1]: tensor-kernel variant, 0 tiled, 1 streaming (B held in tensor
 * memory: N <= 128, K <= 128 and at least one 128-row tile per SM; the
 * environment variable GEMM_F32_STREAM=0 turns it off); out[2]: split-K
 * ways of the split tiles (1: none; 2..8 reduce within thread-block
 * clusters, more through scratch; GEMM_F32_CLUSTER_REDUCE=0 takes the
 * scratch for every split); out[3]: tiles computed whole before the split
 * ones; out[4]: rows of C per tensor tile (256 when K >= 2048,
 * else 128; 0 for the FFMA kernels).  Returns a status
 * (GEMM_F32_ERR_INVALID_ARG also for out == NULL).
 */
GEMM_F32_API int gemm_f32_plan(int64_t M, int64_t N, int64_t K,
                               const float *A, int64_t lda, const float *B,
                               int64_t ldb, const float *C, int64_t ldc,
                               int64_t out[5]);

/*
 * Host logic only, no CUDA call (tests of the planner, and planning on a
 * machine without the GPU): the plan gemm_f32_plan would make on a device
 * with `sm_count` SMs and compute capability major `cc_major` (10 for the
 * tcgen05 family).  A, B and C are only checked for 16-byte alignment and
 * NULL, never read.  out[] as for gemm_f32_plan.  GEMM_F32_ERR_INVALID_ARG
 * for bad sizes, out == NULL or sm_count < 1.
 */
GEMM_F32_API int gemm_f32_plan_sms(int64_t M, int64_t N, int64_t K,
                                   const float *A, int64_t lda,
                                   const float *B, int64_t ldb,
                                   const float *C, int64_t ldc, int sm_count,
                                   int cc_major, int64_t out[5]);

/* Host logic only, no CUDA call: the plan gemm_f32_mixed_plan would make on
 * a device with `sm_count` SMs.  out[] and errors as for
 * gemm_f32_mixed_plan (GEMM_F32_ERR_INVALID_ARG also for sm_count < 1). */
GEMM_F32_API int gemm_f32_mixed_plan_sms(int64_t M, int64_t N, int64_t K,
                                         int sm_count, int64_t out[5]);

/*
 * Host logic only, no CUDA call: the row chunks gemm_f32_host cuts an M × N
 * product into on a device with `sm_count` SMs.  Writes the first row of
 * each chunk to bounds[0..n-1] and M to bounds[n] (bounds holds at least 17
 * entries) and returns n (1 to 16), or GEMM_F32_ERR_INVALID_ARG negated
 * (M or N < 1, sm_count < 1, bounds NULL).
 */
GEMM_F32_API int gemm_f32_host_chunks(int64_t M, int64_t N, int sm_count,
                                      int64_t bounds[17]);

/* Static description of a status code. */
GEMM_F32_API const char *gemm_f32_status_string(int status);

/* cudaError_t of the most recent GEMM_F32_ERR_CUDA on this host thread. */
GEMM_F32_API int gemm_f32_last_cuda_error(void);

/*
 * Waits for `stream`, then reads and clears the current device's kernel
 * status word.  Returns GEMM_F32_OK; GEMM_F32_ERR_BOUNDS if, in the checked
 * build, a kernel's index check failed since the last call;
 * GEMM_F32_ERR_TIMEOUT if a kernel's bounded mbarrier wait gave up; or
 * GEMM_F32_ERR_CUDA.  This is the only entry point that synchronizes.
 */
GEMM_F32_API int gemm_f32_device_status(gemm_f32_stream_t stream);

/*
 * The checked build.  libgemm_f32_debug.so (built with
 * GEMM_F32_BOUNDS_CHECK=1; python -m dense_fp32_matrix_02_gb300.build
 * --checked) exports the same entry points as libgemm_f32.so, but its FFMA
 * and tensor kernels test every shared-memory, tensor-memory and global
 * index they compute against the extent it must lie in (the stage buffer,
 * the TMEM allocation, the matrix) before the access; a failed test sets a
 * status bit, reported as GEMM_F32_ERR_BOUNDS by gemm_f32_device_status,
 * and the access is skipped, so nothing faults.  It is a test build that
 * stands in for a memory checker (the pages' race and out-of-range
 * symptoms, "3 · La mémoire partagée" §3.2, §3.3), slower than the normal
 * one.  The pages have no counterpart to the entries below.
 *
 * gemm_f32_bounds_checked: 1 in the checked build, 0 in the normal one.
 * gemm_f32_bounds_probe: in the checked build, launches one thread that
 * runs the kernels' check on an index one element past a 4-element extent
 * (nothing is read or written), so the next gemm_f32_device_status must
 * return GEMM_F32_ERR_BOUNDS; in the normal build launches nothing.
 * Returns GEMM_F32_OK or GEMM_F32_ERR_CUDA.
 */
GEMM_F32_API int gemm_f32_bounds_checked(void);
GEMM_F32_API int gemm_f32_bounds_probe(gemm_f32_stream_t stream);

/* The deadline, in nanoseconds of the GPU's global timer, after which an
 * mbarrier wait in the pipelined kernels gives up (<= 0 restores the
 * default of 2 s).  Applies to later launches; returns the previous value.
 * A kernel that gives up sets the status word read by
 * gemm_f32_device_status, releases what it holds and ends without writing
 * its tile of C.  Process-wide setting. */
GEMM_F32_API int64_t gemm_f32_set_wait_timeout_ns(int64_t ns);

/* Test hook, process-wide, for later launches: bit 0 makes the copy
 * producer of the pipelined kernels issue no copies, so that their waits run
 * out and the timeout path can be checked.  0 (the default) disables every
 * hook.  Returns the previous flags. */
GEMM_F32_API unsigned int gemm_f32_set_debug_flags(unsigned int flags);

/* Library version, major*10000 + minor*100 + patch. */
GEMM_F32_API int gemm_f32_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_F32_H */
