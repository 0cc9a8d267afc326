// C ABI of libgemm_f32: argument checks, kernel selection and launch.
//
// The ABI is declared in include/gemm_f32.h.  Every entry point returns a
// status and never throws; only gemm_f32_device_status synchronizes.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <set>
#include <utility>

#include "gemm_f32.h"
#include "kernels.h"

using namespace gemm_f32_impl;

// Kernel status word (kStatus* bits), one per device; read and cleared by
// gemm_f32_device_status.
__device__ unsigned int g_kernel_status;

// The checked build's self-test: the kernels' index check applied to one
// element past a 4-element extent (the status word itself); nothing is
// read or written through the index, the check only reports it.
__global__ void bounds_probe_kernel(unsigned int* status) {
  (void)span_ok(status + 4, 4, status, 16, status);
}

namespace {

constexpr long long kDefaultWaitNs = 2000000000LL;  // 2 s
constexpr int kMaxDevices = 64;

thread_local int t_last_cuda_error = 0;
std::atomic<long long> g_wait_ns{kDefaultWaitNs};
std::atomic<unsigned int> g_debug_flags{0};

struct DeviceInfo {
  bool ready = false;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  unsigned int* status = nullptr;
};

std::mutex g_mu;
DeviceInfo g_devices[kMaxDevices];
std::set<std::pair<int, const void*>> g_smem_attr_done;

int fail_cuda(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return GEMM_F32_ERR_CUDA;
}

// Per-device facts, fetched once with that device current.
cudaError_t device_info(const DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_devices[dev];
  if (!d.ready) {
    cudaDeviceProp prop;
    if ((e = cudaGetDeviceProperties(&prop, dev)) != cudaSuccess) return e;
    void* status = nullptr;
    if ((e = cudaGetSymbolAddress(&status, g_kernel_status)) != cudaSuccess)
      return e;
    d.sm_count = prop.multiProcessorCount;
    d.cc_major = prop.major;
    d.cc_minor = prop.minor;
    d.status = static_cast<unsigned int*>(status);
    d.ready = true;
  }
  *out = &d;
  return cudaSuccess;
}

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

int env_int(const char* name, int fallback) {
  const char* v = std::getenv(name);
  if (!v || !*v) return fallback;
  return std::atoi(v);
}

struct Plan {
  int algo;      // gemm_f32_algo actually run
  int simt_cfg;  // for ALGO_SIMT
  int tc_cfg;    // for ALGO_TF32X3
  int splits;    // split-K factor for ALGO_TF32X3 (1 = none)
  int full_tiles;  // tiles computed whole before the split ones
  bool cluster;    // every tile split, reduced within thread-block clusters
  bool tc_stream;  // ALGO_TF32X3 on the streaming kernel (narrow B)
  long long ws_bytes;  // scratch the plan needs (0 = none)
  bool vec;      // 16-byte operand copies
  bool c_vec;    // 16-byte C stores
};

int check_args(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
               const float* B, int64_t ldb, const float* C, int64_t ldc) {
  if (M < 0 || N < 0 || K < 0) return GEMM_F32_ERR_INVALID_ARG;
  if (lda < K || ldb < N || ldc < N) return GEMM_F32_ERR_INVALID_ARG;
  if (M > 0x7fffffff || N > 0x7fffffff || K > 0x7fffffff)
    return GEMM_F32_ERR_UNSUPPORTED;
  if (M > 0 && N > 0) {
    if (!C) return GEMM_F32_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B)) return GEMM_F32_ERR_INVALID_ARG;
  }
  return GEMM_F32_OK;
}

int choose_simt_cfg(int64_t M, int64_t N, const DeviceInfo& d) {
  const int forced = env_int("GEMM_F32_SIMT_CFG", -1);
  if (forced >= 0 && forced < kSimtCfgCount) return forced;
  if (N <= 64) return kSimt128x64x16;
  const int64_t tiles = ((M + 127) / 128) * ((N + 127) / 128);
  if (tiles < d.sm_count) return kSimt128x64x16;
  // 16-byte operands: the warp-specialised kernel (a producer warpgroup
  // issues the copies; 4096^3: 54.4 TFLOP/s against 45.3 for the best
  // single-role kernel).  Otherwise A transposed on its way into shared
  // memory by 4-byte copies (4096^3: 41.8).
  return kSimtWs128x128x32;
}

int choose_tc_cfg(int64_t M, int64_t N, int64_t K, const DeviceInfo& d) {
  const int forced = env_int("GEMM_F32_TC_CFG", -1);
  if (forced >= 0 && forced < kTcCfgCount) return forced;
  // Both let the tensor core truncate the raw operands to TF32 (half the
  // converters' work).  256 x 128 tiles at one CTA per SM convert each B
  // tile for twice the MMAs and won on every measured shape with K >= 2048
  // (by 2-18 %, from 32 such tiles up to 8192^3; 4096^3: 341 against 310
  // TFLOP/s); for shorter K, 128 x 128 tiles at two CTAs per SM (finer
  // grain, one CTA's epilogue overlapping the other's main loop).
  (void)M;
  (void)N;
  (void)d;
  return K >= 2048 ? kTc256Raw : kTc128Raw;
}

// Split-K for the tensor path, so that the CTAs fill the GPU:
//  * tiles fill fewer than half of the CTA slots: every tile is split,
//    slots / tiles ways;
//  * otherwise the tiles of the last, partly filled round (tiles mod slots
//    of them) are split floor(slots / tail) ways, so they spread over the
//    whole GPU instead of running one per SM while the rest idle (a lone
//    tile costs about as long as a full round);
// at least 8 k stages per split, at most 16 splits.  GEMM_F32_SPLITS forces
// every tile to split that many ways; GEMM_F32_TAIL_SPLIT=0 keeps the last
// round whole.  Up to kMaxClusterSplits ways, the splits of a tile run as
// one thread-block cluster and add their partial tiles in distributed
// shared memory: no scratch and no reduction kernel (a split tail runs as
// a second launch after the whole tiles'; GEMM_F32_CLUSTER_REDUCE=0 takes
// the scratch and the reduction kernel instead).
void choose_splits(int64_t M, int64_t N, int64_t K, int tile_m,
                   const DeviceInfo& d, Plan* plan) {
  const int forced = env_int("GEMM_F32_SPLITS", 0);
  const int64_t nk = (K + 15) / 16;
  const int64_t tiles = ((M + tile_m - 1) / tile_m) * ((N + 127) / 128);
  const int64_t slots = (tile_m == 128 ? 2 : 1) * (int64_t)d.sm_count;
  int64_t s = 1, full = tiles;
  if (forced > 0) {
    s = std::min<int64_t>(std::min<int64_t>(forced, nk), 16);
    full = 0;
  } else if (2 * tiles < slots) {
    s = std::min<int64_t>(std::min<int64_t>(slots / tiles, nk / 8), 16);
    full = 0;
  } else if (tiles % slots != 0 && env_int("GEMM_F32_TAIL_SPLIT", 1) != 0) {
    const int64_t tail = tiles % slots;
    s = std::min<int64_t>(std::min<int64_t>(slots / tail, nk / 8), 16);
    full = tiles - tail;
  }
  if (s < 2) {
    s = 1;
    full = tiles;
  }
  plan->splits = (int)s;
  plan->full_tiles = (int)full;
  plan->cluster = s >= 2 && s <= kMaxClusterSplits &&
                  env_int("GEMM_F32_CLUSTER_REDUCE", 1) != 0;
  plan->ws_bytes = plan->cluster
                       ? 0
                       : tf32x3_partials_bytes(tile_m, tiles - full, (int)s);
}

// Decides which kernel runs.  Returns a status; fills *plan on success.
int make_plan(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
              const float* B, int64_t ldb, const float* C, int64_t ldc,
              int algo, const DeviceInfo& d, Plan* plan) {
  const bool vec = aligned16(A) && aligned16(B) && lda % 4 == 0 &&
                   ldb % 4 == 0;
  plan->vec = vec;
  plan->c_vec = aligned16(C) && ldc % 4 == 0;
  plan->simt_cfg = choose_simt_cfg(M, N, d);
  plan->tc_cfg = choose_tc_cfg(M, N, K, d);
  plan->splits = 1;
  plan->full_tiles = 0;
  plan->cluster = false;
  plan->tc_stream = false;
  plan->ws_bytes = 0;
  const bool tcgen05_ok = d.cc_major == 10 && vec && K >= 1;
  switch (algo) {
    case GEMM_F32_ALGO_AUTO:
      plan->algo = (tcgen05_ok && env_int("GEMM_F32_AUTO_SIMT", 0) == 0)
                       ? GEMM_F32_ALGO_TF32X3
                       : GEMM_F32_ALGO_SIMT;
      break;
    case GEMM_F32_ALGO_SIMT:
      plan->algo = GEMM_F32_ALGO_SIMT;
      return GEMM_F32_OK;
    case GEMM_F32_ALGO_TF32X3:
      if (!tcgen05_ok) return GEMM_F32_ERR_UNSUPPORTED;
      plan->algo = GEMM_F32_ALGO_TF32X3;
      break;
    case GEMM_F32_ALGO_TMA:
      if (!(vec && K >= 1)) return GEMM_F32_ERR_UNSUPPORTED;
      plan->algo = GEMM_F32_ALGO_TMA;
      return GEMM_F32_OK;
    default:
      return GEMM_F32_ERR_INVALID_ARG;
  }
  if (plan->algo == GEMM_F32_ALGO_TF32X3) {
    // B narrow and shallow enough to live in TMEM, and at least one
    // 128-row tile per SM: the persistent streaming kernel
    if (tf32x3_stream_fits(N, K) && (M + 127) / 128 >= d.sm_count &&
        env_int("GEMM_F32_STREAM", 1) != 0)
      plan->tc_stream = true;
    else
      choose_splits(M, N, K, tf32x3_tile_m(plan->tc_cfg), d, plan);
  }
  return GEMM_F32_OK;
}

}  // namespace

namespace gemm_f32_impl {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

cudaError_t ensure_smem_attr(const void* fn, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  auto key = std::make_pair(dev, fn);
  if (g_smem_attr_done.count(key)) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           bytes);
  if (e == cudaSuccess) g_smem_attr_done.insert(key);
  return e;
}

}  // namespace gemm_f32_impl

extern "C" {

}  // extern "C"

namespace {

// One call: checks, plan, launch.  `ws`/`ws_bytes` is optional scratch; a
// plan that wants more than given runs without split-K.
int run_gemm(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
             const float* B, int64_t ldb, float* C, int64_t ldc,
             gemm_f32_stream_t stream, int algo, void* ws, int64_t ws_bytes,
             const float* bias = nullptr, int act = 0) {
  if (act != kActNone && act != kActGelu) return GEMM_F32_ERR_INVALID_ARG;
  if (algo < GEMM_F32_ALGO_AUTO || algo > GEMM_F32_ALGO_TF32X3)
    return GEMM_F32_ERR_INVALID_ARG;
  if (ws_bytes < 0 || (ws_bytes > 0 && !ws)) return GEMM_F32_ERR_INVALID_ARG;
  int st = check_args(M, N, K, A, lda, B, ldb, C, ldc);
  if (st != GEMM_F32_OK) return st;
  if (M == 0 || N == 0) return GEMM_F32_OK;
  const DeviceInfo* d = nullptr;
  cudaError_t e = device_info(&d);
  if (e != cudaSuccess) return fail_cuda(e);
  Plan plan;
  st = make_plan(M, N, K, A, lda, B, ldb, C, ldc, algo, *d, &plan);
  if (st != GEMM_F32_OK) return st;
  if (plan.ws_bytes > 0 &&
      (plan.ws_bytes > ws_bytes || !aligned16(ws))) {
    plan.splits = 1;
    plan.ws_bytes = 0;
  }

  Problem p;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.A = A;
  p.lda = lda;
  p.B = B;
  p.ldb = ldb;
  p.C = C;
  p.ldc = ldc;
  p.bias = bias;
  p.act = act;
  p.status = d->status;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (plan.algo) {
    case GEMM_F32_ALGO_SIMT: {
      WaitCfg wc;
      wc.limit = g_wait_ns.load();
      wc.debug = g_debug_flags.load();
      wc.status = d->status;
      e = launch_simt(p, plan.simt_cfg, plan.vec, plan.c_vec, wc, s);
      break;
    }
    case GEMM_F32_ALGO_TMA: {
      WaitCfg wc;
      wc.limit = g_wait_ns.load();
      wc.debug = g_debug_flags.load();
      wc.status = d->status;
      e = launch_tma_ffma(p, plan.c_vec, wc, s);
      break;
    }
    case GEMM_F32_ALGO_TF32X3: {
      WaitCfg wc;
      wc.limit = g_wait_ns.load();
      wc.debug = g_debug_flags.load();
      wc.status = d->status;
      e = plan.tc_stream
              ? launch_tf32x3_stream(p, d->sm_count, wc, s)
              : launch_tf32x3(p, plan.tc_cfg, plan.full_tiles, plan.splits,
                              plan.splits > 1 && !plan.cluster
                                  ? static_cast<float*>(ws)
                                  : nullptr,
                              plan.cluster, wc, s);
      break;
    }
    default:
      return GEMM_F32_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) return fail_cuda(e);
  return GEMM_F32_OK;
}

}  // namespace

namespace gemm_f32_impl {

int record_cuda_error(cudaError_t e) { return fail_cuda(e); }

long long auto_plan_scratch_bytes(int64_t M, int64_t N, int64_t K,
                                  const float* A, int64_t lda, const float* B,
                                  int64_t ldb, const float* C, int64_t ldc) {
  const int st = check_args(M, N, K, A, lda, B, ldb, C, ldc);
  if (st != GEMM_F32_OK) return -st;
  if (M == 0 || N == 0) return 0;
  const DeviceInfo* d = nullptr;
  cudaError_t e = device_info(&d);
  if (e != cudaSuccess) return -fail_cuda(e);
  Plan plan;
  const int ps = make_plan(M, N, K, A, lda, B, ldb, C, ldc,
                           GEMM_F32_ALGO_AUTO, *d, &plan);
  if (ps != GEMM_F32_OK) return -ps;
  return plan.ws_bytes;
}

int run_auto_with_scratch(int64_t M, int64_t N, int64_t K, const float* A,
                          int64_t lda, const float* B, int64_t ldb, float* C,
                          int64_t ldc, void* scratch, int64_t scratch_bytes,
                          gemm_f32_stream_t stream) {
  return run_gemm(M, N, K, A, lda, B, ldb, C, ldc, stream, GEMM_F32_ALGO_AUTO,
                  scratch, scratch_bytes);
}

}  // namespace gemm_f32_impl

namespace {

bool mult4(int64_t x) { return x % 4 == 0; }

// Bytes of one transposed copy of a K×M stored A (op(A) = Aᵀ written M×K,
// rows of K rounded up to a multiple of 4), rounded up to 256 bytes.
int64_t transposed_copy_bytes(int64_t M, int64_t K) {
  return (M * ((K + 3) / 4 * 4) * 4 + 255) / 256 * 256;
}

// `ws`/`ws_bytes`: optional scratch.  With opA = T, opB = N on the tensor
// path and room for the transposed copies, A is transposed into it first
// and the product runs as opA = N (for batch = 1 through run_gemm, whose
// split-K scratch is the rest of ws).
int run_batched(int opA, int opB, int64_t M, int64_t N, int64_t K,
                const float* A, int64_t lda, int64_t sA, const float* B,
                int64_t ldb, int64_t sB, float* C, int64_t ldc, int64_t sC,
                int64_t batch, gemm_f32_stream_t stream, void* ws,
                int64_t ws_bytes) {
  if ((opA != GEMM_F32_OP_N && opA != GEMM_F32_OP_T) ||
      (opB != GEMM_F32_OP_N && opB != GEMM_F32_OP_T))
    return GEMM_F32_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || batch < 0) return GEMM_F32_ERR_INVALID_ARG;
  const bool ta = opA == GEMM_F32_OP_T, tb = opB == GEMM_F32_OP_T;
  if (lda < (ta ? M : K) || ldb < (tb ? K : N) || ldc < N)
    return GEMM_F32_ERR_INVALID_ARG;
  if (sA < 0 || sB < 0 || sC < 0) return GEMM_F32_ERR_INVALID_ARG;
  if (ws_bytes < 0 || (ws_bytes > 0 && !ws)) return GEMM_F32_ERR_INVALID_ARG;
  if (M > 0x7fffffff || N > 0x7fffffff || K > 0x7fffffff || batch > 65535)
    return GEMM_F32_ERR_UNSUPPORTED;
  if (M == 0 || N == 0 || batch == 0) return GEMM_F32_OK;
  if (!C || (K > 0 && (!A || !B))) return GEMM_F32_ERR_INVALID_ARG;
  if (!ta && !tb && batch == 1)  // the plain product
    return run_gemm(M, N, K, A, lda, B, ldb, C, ldc, stream,
                    GEMM_F32_ALGO_AUTO, ws, ws_bytes);
  const DeviceInfo* d = nullptr;
  cudaError_t e = device_info(&d);
  if (e != cudaSuccess) return fail_cuda(e);
  Problem p;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.A = A;
  p.lda = lda;
  p.B = B;
  p.ldb = ldb;
  p.C = C;
  p.ldc = ldc;
  p.sA = sA;
  p.sB = sB;
  p.sC = sC;
  p.batch = static_cast<int>(batch);
  p.transA = ta ? 1 : 0;
  p.transB = tb ? 1 : 0;
  p.status = d->status;
  const bool vec = aligned16(A) && aligned16(B) && mult4(lda) && mult4(ldb) &&
                   mult4(sA) && mult4(sB);
  const bool c_vec = aligned16(C) && mult4(ldc) && mult4(sC);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The tensor kernel takes every form (TN through its converters) when
  // TMA can describe every operand: aligned, and batch strides 0 or at
  // least one whole stored matrix.
  const int64_t rows_a = ta ? K : M, rows_b = tb ? N : K;
  const bool strides_ok = (batch == 1) ||
                          ((sA == 0 || sA >= rows_a * lda) &&
                           (sB == 0 || sB >= rows_b * ldb));
  if (d->cc_major == 10 && vec && K >= 1 && strides_ok &&
      env_int("GEMM_F32_AUTO_SIMT", 0) == 0) {
    Problem q = p;
    if (ta && tb) {  // C = (B·A)ᵀ: swap the operands, store the transpose
      q.M = p.N;
      q.N = p.M;
      q.A = B;
      q.lda = ldb;
      q.sA = sB;
      q.B = A;
      q.ldb = lda;
      q.sB = sA;
      q.transA = 0;
      q.transB = 0;
      q.storeT = 1;
    }
    // Aᵀ·B: a transposed copy of A, then the plain form, when ws has room
    const int64_t copies = (batch == 1 || sA == 0) ? 1 : batch;
    const int64_t one = transposed_copy_bytes(M, K);
    if (ta && !tb && aligned16(ws) && ws_bytes / copies >= one) {
      const int64_t ldt = (K + 3) / 4 * 4;
      float* at = static_cast<float*>(ws);
      e = launch_transpose(A, lda, sA, at, ldt, one / 4, K, M, copies,
                           d->sm_count, s);
      if (e != cudaSuccess) return fail_cuda(e);
      if (batch == 1)
        return run_gemm(M, N, K, at, ldt, B, ldb, C, ldc, stream,
                        GEMM_F32_ALGO_AUTO, static_cast<char*>(ws) + one,
                        ws_bytes - one);
      q.A = at;
      q.lda = ldt;
      q.sA = copies == 1 ? 0 : one / 4;
      q.transA = 0;
    }
    WaitCfg wc;
    wc.limit = g_wait_ns.load();
    wc.debug = g_debug_flags.load();
    wc.status = d->status;
    // the same tile choice as single products
    int cfg = kTc128Raw;
    const int forced = env_int("GEMM_F32_TC_CFG", -1);
    if (forced == kTc128Raw || forced == kTc256Raw)
      cfg = forced;
    else if (forced < 0 && K >= 2048 && !q.transA)
      cfg = kTc256Raw;
    e = launch_tf32x3(q, cfg, 0, 1, nullptr, false, wc, s);
  } else {
    WaitCfg wc;
    wc.limit = g_wait_ns.load();
    wc.debug = g_debug_flags.load();
    wc.status = d->status;
    e = launch_simt(p, choose_simt_cfg(M, N, *d), vec, c_vec, wc, s);
  }
  if (e != cudaSuccess) return fail_cuda(e);
  return GEMM_F32_OK;
}

// out[] of gemm_f32_plan for the AUTO plan on device d.
int report_plan(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                const float* B, int64_t ldb, const float* C, int64_t ldc,
                const DeviceInfo& d, int64_t out[5]) {
  Plan plan;
  const int st = make_plan(M, N, K, A, lda, B, ldb, C, ldc,
                           GEMM_F32_ALGO_AUTO, d, &plan);
  if (st != GEMM_F32_OK) return st;
  out[0] = plan.algo;
  out[1] = plan.tc_stream ? 1 : 0;
  out[2] = plan.splits;
  out[3] = plan.full_tiles;
  out[4] = plan.algo != GEMM_F32_ALGO_TF32X3 ? 0
           : plan.tc_stream                   ? 128
                                              : tf32x3_tile_m(plan.tc_cfg);
  return GEMM_F32_OK;
}

}  // namespace

extern "C" {

int gemm_f32_bias_act(int64_t M, int64_t N, int64_t K, const float* A,
                      int64_t lda, const float* B, int64_t ldb,
                      const float* bias, int act, float* C, int64_t ldc,
                      void* workspace, int64_t workspace_bytes,
                      gemm_f32_stream_t stream) {
  return run_gemm(M, N, K, A, lda, B, ldb, C, ldc, stream, GEMM_F32_ALGO_AUTO,
                  workspace, workspace_bytes, bias, act);
}

int gemm_f32_batched(int opA, int opB, int64_t M, int64_t N, int64_t K,
                     const float* A, int64_t lda, int64_t strideA,
                     const float* B, int64_t ldb, int64_t strideB, float* C,
                     int64_t ldc, int64_t strideC, int64_t batch,
                     gemm_f32_stream_t stream) {
  return run_batched(opA, opB, M, N, K, A, lda, strideA, B, ldb, strideB, C,
                     ldc, strideC, batch, stream, nullptr, 0);
}

int gemm_f32_batched_ws(int opA, int opB, int64_t M, int64_t N, int64_t K,
                        const float* A, int64_t lda, int64_t strideA,
                        const float* B, int64_t ldb, int64_t strideB,
                        float* C, int64_t ldc, int64_t strideC,
                        int64_t batch, void* workspace,
                        int64_t workspace_bytes, gemm_f32_stream_t stream) {
  return run_batched(opA, opB, M, N, K, A, lda, strideA, B, ldb, strideB, C,
                     ldc, strideC, batch, stream, workspace, workspace_bytes);
}

int64_t gemm_f32_batched_workspace_size(int opA, int opB, int64_t M,
                                        int64_t N, int64_t K,
                                        int64_t batch) {
  if ((opA != GEMM_F32_OP_N && opA != GEMM_F32_OP_T) ||
      (opB != GEMM_F32_OP_N && opB != GEMM_F32_OP_T) || M < 0 || N < 0 ||
      K < 0 || batch < 0)
    return -GEMM_F32_ERR_INVALID_ARG;
  if (M == 0 || N == 0 || K == 0 || batch == 0) return 0;
  int64_t bytes = 0;
  if (opA == GEMM_F32_OP_T && opB == GEMM_F32_OP_N)
    bytes = transposed_copy_bytes(M, K) * batch;
  if (batch == 1 && opB == GEMM_F32_OP_N) {
    const int64_t split = gemm_f32_workspace_size(M, N, K);
    if (split < 0) return split;
    bytes += split;
  }
  return bytes;
}

int gemm_f32_ex(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                const float* B, int64_t ldb, float* C, int64_t ldc,
                gemm_f32_stream_t stream, int algo) {
  return run_gemm(M, N, K, A, lda, B, ldb, C, ldc, stream, algo, nullptr, 0);
}

int gemm_f32_ws(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                const float* B, int64_t ldb, float* C, int64_t ldc,
                void* workspace, int64_t workspace_bytes,
                gemm_f32_stream_t stream) {
  return run_gemm(M, N, K, A, lda, B, ldb, C, ldc, stream,
                  GEMM_F32_ALGO_AUTO, workspace, workspace_bytes);
}

int64_t gemm_f32_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  const DeviceInfo* d = nullptr;
  cudaError_t e = device_info(&d);
  if (e != cudaSuccess) {
    t_last_cuda_error = static_cast<int>(e);
    return -GEMM_F32_ERR_CUDA;
  }
  Plan plan;
  // the plan for 16-byte aligned operands whose leading dimensions are the
  // row widths rounded up to multiples of 4: the layouts that can use it
  const float* aligned = reinterpret_cast<const float*>(16);
  const int64_t lda = (K + 3) / 4 * 4, ldn = (N + 3) / 4 * 4;
  const int st = make_plan(M, N, K, aligned, lda, aligned, ldn, aligned, ldn,
                           GEMM_F32_ALGO_AUTO, *d, &plan);
  if (st != GEMM_F32_OK) return -st;
  return plan.ws_bytes;
}

int gemm_f32(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
             const float* B, int64_t ldb, float* C, int64_t ldc,
             gemm_f32_stream_t stream) {
  return gemm_f32_ex(M, N, K, A, lda, B, ldb, C, ldc, stream,
                     GEMM_F32_ALGO_AUTO);
}

int gemm_f32_select_algo(int64_t M, int64_t N, int64_t K, const float* A,
                         int64_t lda, const float* B, int64_t ldb, float* C,
                         int64_t ldc) {
  int st = check_args(M, N, K, A, lda, B, ldb, C, ldc);
  if (st != GEMM_F32_OK) return -st;
  const DeviceInfo* d = nullptr;
  cudaError_t e = device_info(&d);
  if (e != cudaSuccess) {
    t_last_cuda_error = static_cast<int>(e);
    return -GEMM_F32_ERR_CUDA;
  }
  Plan plan;
  st = make_plan(M, N, K, A, lda, B, ldb, C, ldc, GEMM_F32_ALGO_AUTO, *d,
                 &plan);
  if (st != GEMM_F32_OK) return -st;
  return plan.algo;
}

int gemm_f32_plan(int64_t M, int64_t N, int64_t K, const float* A,
                  int64_t lda, const float* B, int64_t ldb, const float* C,
                  int64_t ldc, int64_t out[5]) {
  if (!out) return GEMM_F32_ERR_INVALID_ARG;
  const int st = check_args(M, N, K, A, lda, B, ldb, C, ldc);
  if (st != GEMM_F32_OK) return st;
  const DeviceInfo* d = nullptr;
  cudaError_t e = device_info(&d);
  if (e != cudaSuccess) return fail_cuda(e);
  return report_plan(M, N, K, A, lda, B, ldb, C, ldc, *d, out);
}

int gemm_f32_plan_sms(int64_t M, int64_t N, int64_t K, const float* A,
                      int64_t lda, const float* B, int64_t ldb,
                      const float* C, int64_t ldc, int sm_count, int cc_major,
                      int64_t out[5]) {
  if (!out || sm_count < 1) return GEMM_F32_ERR_INVALID_ARG;
  const int st = check_args(M, N, K, A, lda, B, ldb, C, ldc);
  if (st != GEMM_F32_OK) return st;
  DeviceInfo d;  // facts given, not queried; never used to launch
  d.sm_count = sm_count;
  d.cc_major = cc_major;
  return report_plan(M, N, K, A, lda, B, ldb, C, ldc, d, out);
}

const char* gemm_f32_status_string(int status) {
  switch (status) {
    case GEMM_F32_OK:
      return "ok";
    case GEMM_F32_ERR_INVALID_ARG:
      return "invalid argument";
    case GEMM_F32_ERR_UNSUPPORTED:
      return "unsupported: the forced algorithm's preconditions do not hold";
    case GEMM_F32_ERR_CUDA:
      return "CUDA runtime error";
    case GEMM_F32_ERR_TIMEOUT:
      return "a kernel's bounded wait gave up";
    case GEMM_F32_ERR_SCRATCH_LIMIT:
      return "the product needs more split-K scratch than the library's "
             "static buffer holds (see gemm_f32_noalloc_scratch_bytes)";
    case GEMM_F32_ERR_BOUNDS:
      return "checked build: a kernel's index fell outside its extent (the "
             "access was skipped)";
    default:
      return "unknown status";
  }
}

int gemm_f32_last_cuda_error(void) { return t_last_cuda_error; }

int gemm_f32_device_status(gemm_f32_stream_t stream) {
  const DeviceInfo* d = nullptr;
  cudaError_t e = device_info(&d);
  if (e != cudaSuccess) return fail_cuda(e);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return fail_cuda(e);
  unsigned int word = 0;
  if ((e = cudaMemcpyFromSymbol(&word, g_kernel_status, sizeof(word))) !=
      cudaSuccess)
    return fail_cuda(e);
  if (word) {
    const unsigned int zero = 0;
    if ((e = cudaMemcpyToSymbol(g_kernel_status, &zero, sizeof(zero))) !=
        cudaSuccess)
      return fail_cuda(e);
    return (word & kStatusBounds) ? GEMM_F32_ERR_BOUNDS
                                  : GEMM_F32_ERR_TIMEOUT;
  }
  return GEMM_F32_OK;
}

int gemm_f32_bounds_checked(void) { return GEMM_F32_BOUNDS_CHECK ? 1 : 0; }

int gemm_f32_bounds_probe(gemm_f32_stream_t stream) {
  if (!GEMM_F32_BOUNDS_CHECK) return GEMM_F32_OK;
  const DeviceInfo* d = nullptr;
  cudaError_t e = device_info(&d);
  if (e != cudaSuccess) return fail_cuda(e);
  bounds_probe_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      d->status);
  if ((e = cudaGetLastError()) != cudaSuccess) return fail_cuda(e);
  return GEMM_F32_OK;
}

int64_t gemm_f32_set_wait_timeout_ns(int64_t ns) {
  return g_wait_ns.exchange(ns > 0 ? ns : kDefaultWaitNs);
}

unsigned int gemm_f32_set_debug_flags(unsigned int flags) {
  return g_debug_flags.exchange(flags);
}

// ------------------------------------------------ mixed precision (16-bit)
}  // extern "C"

namespace {

// Rows per 16-bit tile: 256 (two M = 128 MMAs per k-step sharing each B
// stage, one accumulator filling TMEM) when K >= 2048 and there is a
// 256 × 256 tile for every SM (4096^3 bf16: 1548 against 1378 TFLOP/s);
// else 128 (two accumulators, so one tile's epilogue overlaps the next
// tile's MMAs: ahead on few tiles and short K).  GEMM_F32_MIXED_BM=128 or
// 256 forces it.
int mixed_tile_rows(int64_t M, int64_t N, int64_t K, const DeviceInfo& d) {
  const int forced = env_int("GEMM_F32_MIXED_BM", 0);
  if (forced == 128 || forced == 256) return forced;
  const int64_t tiles256 = ((M + 255) / 256) * ((N + 255) / 256);
  return (K >= 2048 && N > 128 && tiles256 >= d.sm_count) ? 256 : 128;
}

// out[] of gemm_f32_mixed_plan on device d.
void report_mixed_plan(int64_t M, int64_t N, int64_t K, const DeviceInfo& d,
                       int64_t out[5]) {
  const gemm_f32_impl::Plan16 plan = gemm_f32_impl::plan_mixed16(
      M, N, d.sm_count, env_int("GEMM_F32_MIXED_NARROW", 1) != 0,
      mixed_tile_rows(M, N, K, d));
  out[0] = plan.wn;
  out[1] = plan.full;
  out[2] = plan.parts;
  out[3] = plan.grid;
  out[4] = plan.bm;
}

}  // namespace

extern "C" {

int64_t gemm_f32_mixed_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return -GEMM_F32_ERR_INVALID_ARG;
  const int64_t a = M * ((K + 7) / 8 * 8) * 2;
  const int64_t b = K * ((N + 7) / 8 * 8) * 2;
  return (a + 255) / 256 * 256 + b;
}

int gemm_f32_round16(int type, int64_t rows, int64_t cols, const float* src,
                     int64_t lds, void* dst, int64_t ldd,
                     gemm_f32_stream_t stream) {
  if (type != GEMM_F32_MIXED_BF16 && type != GEMM_F32_MIXED_F16)
    return GEMM_F32_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || lds < cols || ldd < cols)
    return GEMM_F32_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return GEMM_F32_OK;
  if (!src || !dst || (reinterpret_cast<uintptr_t>(dst) & 1u))
    return GEMM_F32_ERR_INVALID_ARG;
  const DeviceInfo* d = nullptr;
  cudaError_t e = device_info(&d);
  if (e != cudaSuccess) return fail_cuda(e);
  e = gemm_f32_impl::launch_round16(type, rows, cols, src, lds,
                                    static_cast<uint16_t*>(dst), ldd,
                                    d->sm_count,
                                    reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GEMM_F32_OK : fail_cuda(e);
}

int gemm_f32_mixed16(int type, int64_t M, int64_t N, int64_t K,
                     const void* A, int64_t lda, const void* B, int64_t ldb,
                     float* C, int64_t ldc, gemm_f32_stream_t stream) {
  if (type != GEMM_F32_MIXED_BF16 && type != GEMM_F32_MIXED_F16)
    return GEMM_F32_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || lda < K || ldb < N || ldc < N)
    return GEMM_F32_ERR_INVALID_ARG;
  if (M > 0x7fffffff || N > 0x7fffffff || K > 0x7fffffff)
    return GEMM_F32_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return GEMM_F32_OK;
  if (!C || (K > 0 && (!A || !B))) return GEMM_F32_ERR_INVALID_ARG;
  const DeviceInfo* d = nullptr;
  cudaError_t e = device_info(&d);
  if (e != cudaSuccess) return fail_cuda(e);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) {
    e = gemm_f32_impl::launch_fill_zero(C, ldc, M, N, d->sm_count, s);
    return e == cudaSuccess ? GEMM_F32_OK : fail_cuda(e);
  }
  if (d->cc_major != 10 || !aligned16(A) || !aligned16(B) || lda % 8 != 0 ||
      ldb % 8 != 0)
    return GEMM_F32_ERR_UNSUPPORTED;
  gemm_f32_impl::Problem16 p;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.type = type;
  p.A = A;
  p.lda = lda;
  p.B = B;
  p.ldb = ldb;
  p.C = C;
  p.ldc = ldc;
  gemm_f32_impl::WaitCfg wc;
  wc.limit = g_wait_ns.load();
  wc.debug = g_debug_flags.load();
  wc.status = d->status;
  const gemm_f32_impl::Plan16 plan = gemm_f32_impl::plan_mixed16(
      M, N, d->sm_count, env_int("GEMM_F32_MIXED_NARROW", 1) != 0,
      mixed_tile_rows(M, N, K, *d));
  e = gemm_f32_impl::launch_mixed16(p, plan, aligned16(C) && ldc % 4 == 0,
                                    wc, s);
  return e == cudaSuccess ? GEMM_F32_OK : fail_cuda(e);
}

int gemm_f32_mixed_plan(int64_t M, int64_t N, int64_t K, int64_t out[5]) {
  if (M < 1 || N < 1 || K < 0 || !out) return GEMM_F32_ERR_INVALID_ARG;
  const DeviceInfo* d = nullptr;
  cudaError_t e = device_info(&d);
  if (e != cudaSuccess) return fail_cuda(e);
  report_mixed_plan(M, N, K, *d, out);
  return GEMM_F32_OK;
}

int gemm_f32_mixed_plan_sms(int64_t M, int64_t N, int64_t K, int sm_count,
                            int64_t out[5]) {
  if (M < 1 || N < 1 || K < 0 || !out || sm_count < 1)
    return GEMM_F32_ERR_INVALID_ARG;
  DeviceInfo d;  // facts given, not queried; never used to launch
  d.sm_count = sm_count;
  d.cc_major = 10;
  report_mixed_plan(M, N, K, d, out);
  return GEMM_F32_OK;
}

int gemm_f32_mixed(int type, int64_t M, int64_t N, int64_t K, const float* A,
                   int64_t lda, const float* B, int64_t ldb, float* C,
                   int64_t ldc, void* workspace, int64_t workspace_bytes,
                   gemm_f32_stream_t stream) {
  if (type != GEMM_F32_MIXED_BF16 && type != GEMM_F32_MIXED_F16)
    return GEMM_F32_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || lda < K || ldb < N || ldc < N)
    return GEMM_F32_ERR_INVALID_ARG;
  if (M > 0x7fffffff || N > 0x7fffffff || K > 0x7fffffff)
    return GEMM_F32_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return GEMM_F32_OK;
  if (!C || (K > 0 && (!A || !B))) return GEMM_F32_ERR_INVALID_ARG;
  if (K == 0)
    return gemm_f32_mixed16(type, M, N, 0, nullptr, 0, nullptr, N, C, ldc,
                            stream);
  const int64_t need = gemm_f32_mixed_workspace_size(M, N, K);
  if (!workspace || workspace_bytes < need || !aligned16(workspace))
    return GEMM_F32_ERR_INVALID_ARG;
  const int64_t lda16 = (K + 7) / 8 * 8, ldb16 = (N + 7) / 8 * 8;
  char* ws = static_cast<char*>(workspace);
  void* a16 = ws;
  void* b16 = ws + (M * lda16 * 2 + 255) / 256 * 256;
  int st = gemm_f32_round16(type, M, K, A, lda, a16, lda16, stream);
  if (st != GEMM_F32_OK) return st;
  st = gemm_f32_round16(type, K, N, B, ldb, b16, ldb16, stream);
  if (st != GEMM_F32_OK) return st;
  return gemm_f32_mixed16(type, M, N, K, a16, lda16, b16, ldb16, C, ldc,
                          stream);
}

int gemm_f32_version(void) { return 100; }

}  // extern "C"
