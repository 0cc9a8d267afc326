"""GPU parity: every kernel of libgemm_f32 against the float64 oracle.

All calls go through the C ABI (ctypes binding).  Acceptance per element:
|C - C_ref| <= 1e-5·sqrt(K)·(|A|·|B|)_ij + 1e-30; on small-integer inputs
the result must equal the oracle bit for bit.  Every case, the full-size
workloads included, compares every element of C with the oracle.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_02_gb300 import synth
from helpers import assert_bitexact, assert_within_tolerance

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from dense_fp32_matrix_02_gb300 import gemm as G  # noqa: E402

DEV = torch.device("cuda:0")
SIMT_CFGS = list(range(7))  # kSimtCfgCount


def _env(name, value):
    """Context: sets one environment variable the library reads per call."""
    import contextlib
    import os

    @contextlib.contextmanager
    def ctx():
        old = os.environ.get(name)
        if value is not None:
            os.environ[name] = str(value)
        try:
            yield
        finally:
            if old is None:
                os.environ.pop(name, None)
            else:
                os.environ[name] = old
    return ctx()


def _forced(algo, cfg=None):
    """Context: forces the SIMT tile config."""
    return _env("GEMM_F32_SIMT_CFG", cfg)


TC_CFGS = [0, 1, 2, 3]


def _padded(x):
    """Device copy of x whose row stride is a multiple of 4 elements."""
    rows, cols = x.shape
    ld = max(4, (cols + 3) // 4 * 4)
    store = torch.zeros(max(rows, 1), ld, device=DEV)
    store[:rows, :cols] = torch.from_numpy(x).to(DEV)
    return store[:rows, :cols]


def run_gpu(a, b, algo=G.ALGO_AUTO, c_fill=float("nan"), pad=False):
    """C = A·B on the GPU; pad=True gives every matrix a row stride that is
    a multiple of 4 (what the TMA-fed kernels need) whatever its width."""
    if pad:
        ta, tb = _padded(a), _padded(b)
        tc = _padded(np.full((a.shape[0], b.shape[1]), c_fill, np.float32))
    else:
        ta = torch.from_numpy(a).to(DEV)
        tb = torch.from_numpy(b).to(DEV)
        tc = torch.full((a.shape[0], b.shape[1]), c_fill, dtype=torch.float32,
                        device=DEV)
    G.gemm_f32_ex(ta, tb, tc, algo=algo)
    torch.cuda.synchronize()
    return tc.cpu().numpy()


def check_full(a, b, c, exact=False, what=""):
    ref, bound, _ = oracle.gemm(a, b)
    if exact:
        assert_bitexact(c, ref, what)
    else:
        assert_within_tolerance(c, ref, bound, a.shape[1], what)


_WORKLOAD_REF = {}


def workload_reference(w):
    """(A, B, C_ref, bound) of a named workload; the oracle's product is
    computed once and kept for the next test (the two latest workloads)."""
    if w.name not in _WORKLOAD_REF:
        while len(_WORKLOAD_REF) >= 2:
            _WORKLOAD_REF.pop(next(iter(_WORKLOAD_REF)))
        a, b = w.operands()
        ref, bound, _ = oracle.gemm(a, b)
        _WORKLOAD_REF[w.name] = (a, b, ref, bound)
    return _WORKLOAD_REF[w.name]


def run_like_bench(a, b):
    """C = A·B the way bench.py times it: unpadded operands (ld = row
    width), gemm_f32_ws with exactly the scratch gemm_f32_workspace_size
    asks for, on the current stream.  Returns (C, scratch bytes)."""
    M, K = a.shape
    N = b.shape[1]
    need = G.workspace_size(M, N, K)
    ws = torch.empty(max(need // 4, 1), device=DEV) if need else None
    ta = torch.from_numpy(a).to(DEV)
    tb = torch.from_numpy(b).to(DEV)
    tc = torch.full((M, N), float("nan"), device=DEV)
    G.gemm_f32_ws_ptr(M, N, K, ta.data_ptr(), K, tb.data_ptr(), N,
                      tc.data_ptr(), N, ws.data_ptr() if ws is not None else 0,
                      need, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return tc.cpu().numpy(), need


def expected_tail_plan(M, N, K):
    """The split the planner must choose for a product whose tiles fill
    at least half of the CTA slots: (tile rows, splits, whole tiles)."""
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    rows = 256 if K >= 2048 else 128
    slots = sms * (1 if rows == 256 else 2)
    tiles = -(-M // rows) * -(-N // 128)
    tail = tiles % slots
    if 2 * tiles < slots or tail == 0:
        return None
    s = min(slots // tail, -(-K // 16) // 8, 16)
    return (rows, s, tiles - tail) if s >= 2 else (rows, 1, tiles)


# ------------------------------------------------------------- workloads
SMALL = ["sq64", "sq1024", "rag1000", "skinny"]
LARGE = ["sq4096", "mlp"]


@pytest.mark.parametrize("name", SMALL)
def test_workload_full_auto(name):
    """gemm_f32 and the path bench.py times (gemm_f32_ws with its
    scratch), every element against the oracle."""
    w = synth.WORKLOADS[name]
    a, b = w.operands()
    check_full(a, b, run_gpu(a, b), what=name)
    check_full(a, b, run_like_bench(a, b)[0], what=name + " bench path")


@pytest.mark.parametrize("name", SMALL)
def test_workload_integer_bitexact(name):
    w = synth.WORKLOADS[name].integer_variant()
    a, b = w.operands()
    check_full(a, b, run_gpu(a, b), exact=True, what=w.name)
    check_full(a, b, run_like_bench(a, b)[0], exact=True,
               what=w.name + " bench path")


@pytest.mark.parametrize("integer", [False, True], ids=["float", "int"])
@pytest.mark.parametrize("name", LARGE)
def test_workload_large_full(name, integer):
    """The full-size workloads, every element against the oracle (the
    small-integer variants bit for bit), through two entry points:

    * the path bench.py times: gemm_f32_ws with the scratch it asks for
      (whole tiles, then the last, partly filled round split over K and
      reduced), with the split the planner must choose;
    * gemm_f32 itself (no scratch, nothing split)."""
    w = synth.WORKLOADS[name]
    if integer:
        w = w.integer_variant()
    a, b, ref, bound = workload_reference(w)
    want = expected_tail_plan(w.M, w.N, w.K)
    p = G.plan(w.M, w.N, w.K)
    if want is not None:
        assert (p["tile_rows"], p["splits"], p["whole_tiles"]) == want, p
    c, need = run_like_bench(a, b)
    # up to 8 splits a tile reduce within thread-block clusters: no scratch
    assert (need > 0) == (p["splits"] > 8)
    plain = run_gpu(a, b)
    for got, path in ((c, "bench path"), (plain, "gemm_f32")):
        if integer:
            assert_bitexact(got, ref, f"{w.name} {path}")
        else:
            assert_within_tolerance(got, ref, bound, w.K, f"{w.name} {path}")
    if p["splits"] > 1:
        # the partial tiles through scratch and the reduction kernel: the
        # same sums in the same order, the same bits
        with _env("GEMM_F32_CLUSTER_REDUCE", 0):
            c2, need2 = run_like_bench(a, b)
        assert need2 > 0
        assert np.array_equal(c.view(np.uint32), c2.view(np.uint32))
    assert G.device_status() == 0


# ------------------------------------------------------------- every kernel
@pytest.mark.parametrize("cfg", SIMT_CFGS)
@pytest.mark.parametrize("shape", [(64, 64, 64), (1000, 1000, 1000),
                                   (300, 260, 77), (129, 65, 33)])
def test_simt_configs(cfg, shape):
    M, N, K = shape
    a, b = synth.make_operands(M, N, K, seed=M + N + K)
    with _forced(G.ALGO_SIMT, cfg):
        check_full(a, b, run_gpu(a, b, G.ALGO_SIMT), what=f"simt{cfg}{shape}")
    ai, bi = synth.make_operands(M, N, K, seed=M + N + K, dist_a="int",
                                 dist_b="int")
    with _forced(G.ALGO_SIMT, cfg):
        check_full(ai, bi, run_gpu(ai, bi, G.ALGO_SIMT), exact=True,
                   what=f"simt{cfg}{shape} int")


# ------------------------------------------------------------- edges
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 5), (17, 13, 11),
                                   (7, 1, 200), (1, 300, 9), (131, 127, 129),
                                   (16, 16, 1), (3, 517, 2)])
def test_small_and_prime_shapes(M, N, K):
    a, b = synth.make_operands(M, N, K, seed=5)
    check_full(a, b, run_gpu(a, b), what=f"{M}x{N}x{K}")


def test_sweep_1_to_17():
    for M in (1, 5, 16, 17):
        for N in range(1, 18):
            for K in (1, 4, 7, 16, 17):
                a, b = synth.make_operands(M, N, K, seed=M * 1000 + N * 10 + K,
                                           dist_a="int", dist_b="int")
                check_full(a, b, run_gpu(a, b), exact=True,
                           what=f"{M}x{N}x{K}")


def test_k_zero_writes_zeros():
    a = np.zeros((37, 0), np.float32)
    b = np.zeros((0, 45), np.float32)
    c = run_gpu(a, b)
    assert c.shape == (37, 45) and (c == 0).all()


def test_empty_c_is_noop():
    ta = torch.ones(0, 5, device=DEV)
    tb = torch.ones(5, 3, device=DEV)
    tc = torch.empty(0, 3, device=DEV)
    G.gemm_f32(ta, tb, tc)
    ta = torch.ones(4, 5, device=DEV)
    tb = torch.ones(5, 0, device=DEV)
    G.gemm_f32(ta, tb, torch.empty(4, 0, device=DEV))
    torch.cuda.synchronize()


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_unaligned_pointers_and_odd_leading_dims(offset):
    """Operands that start off a 16-byte boundary, with odd strides."""
    M, N, K = 150, 133, 97
    a, b = synth.make_operands(M, N, K, seed=offset)
    lda, ldb, ldc = K + offset, N + 2 * offset + 1, N + 3
    ta = torch.zeros(M * lda + offset, device=DEV)
    tb = torch.zeros(K * ldb + offset, device=DEV)
    tc = torch.full((M * ldc + offset + 64,), 7.0, device=DEV)
    ta[offset:offset + M * lda].view(M, lda)[:, :K] = torch.from_numpy(a).to(DEV)
    tb[offset:offset + K * ldb].view(K, ldb)[:, :N] = torch.from_numpy(b).to(DEV)
    G.gemm_f32_ptr(M, N, K, ta.data_ptr() + 4 * offset, lda,
                   tb.data_ptr() + 4 * offset, ldb,
                   tc.data_ptr() + 4 * offset, ldc,
                   torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    host = tc.cpu().numpy()
    c = host[offset:offset + M * ldc].reshape(M, ldc)
    check_full(a, b, c[:, :N], what=f"offset {offset}")
    # padding columns and the guard region after C are untouched
    assert (c[:, N:] == 7.0).all()
    assert (host[:offset] == 7.0).all() and (host[offset + M * ldc:] == 7.0).all()


def test_aligned_padded_leading_dims_and_guard():
    M, N, K = 200, 136, 72
    a, b = synth.make_operands(M, N, K, seed=9)
    ldc = 160
    ta = torch.from_numpy(np.pad(a, ((0, 0), (0, 8)))).to(DEV)[:, :K]
    tb = torch.from_numpy(np.pad(b, ((0, 0), (0, 24)))).to(DEV)[:, :N]
    store = torch.full((M + 2, ldc), -3.0, device=DEV)
    tc = store[:M, :N]
    G.gemm_f32(ta, tb, tc)
    torch.cuda.synchronize()
    host = store.cpu().numpy()
    check_full(a, b, host[:M, :N], what="padded")
    assert (host[:M, N:] == -3.0).all() and (host[M:] == -3.0).all()


def test_deterministic_repeat():
    w = synth.WORKLOADS["rag1000"]
    a, b = w.operands()
    c1 = run_gpu(a, b)
    c2 = run_gpu(a, b)
    assert np.array_equal(c1.view(np.uint32), c2.view(np.uint32))


def test_nan_and_inf_propagate_simt():
    """The FFMA kernel follows IEEE arithmetic for NaN and Inf inputs."""
    a, b = synth.make_operands(64, 64, 64, seed=3)
    a[5, 7] = np.nan
    b[9, 11] = np.inf
    c = run_gpu(a, b, G.ALGO_SIMT)
    ref, bound, _ = oracle.gemm(a, b)
    assert np.array_equal(np.isnan(c), np.isnan(ref))
    fin = np.isfinite(ref)
    assert np.array_equal(np.isinf(c), np.isinf(ref))
    assert_within_tolerance(c[fin], ref[fin], bound[fin], 64, "finite part")


def _plant_nonfinite(a, b):
    """NaN and ±Inf in A and B, at places that give every IEEE case: a NaN
    row, +Inf and -Inf rows and columns, Inf·0 (B holds exact zeros),
    Inf·Inf, and +Inf meeting -Inf in one sum."""
    M, K = a.shape
    N = b.shape[1]
    a, b = a.copy(), b.copy()
    a[5 % M, 7 % K] = np.nan
    b[9 % K, 11 % N] = np.inf
    a[(M - 3) % M, (K - 2) % K] = -np.inf
    a[20 % M, 3 % K] = np.inf
    b[3 % K, 40 % N] = np.inf            # Inf·Inf in C[20, 40]
    b[(K - 1) % K, 2 % N] = -np.inf       # with a[20, 3]: +Inf and -Inf
    a[20 % M, (K - 1) % K] = 1.0          #   meet in C[20, 2]
    return a, b


def _check_ieee(c, a, b, what, tol_scale=1.0):
    """Non-finite outputs exactly where IEEE (the oracle) has them, with the
    same NaN / ±Inf class; the finite ones within tolerance."""
    ref, bound, _ = oracle.gemm(a, b)
    K = a.shape[1]
    assert np.array_equal(np.isnan(c), np.isnan(ref)), what + " NaN set"
    assert np.array_equal(np.isposinf(c), np.isposinf(ref)), what + " +Inf"
    assert np.array_equal(np.isneginf(c), np.isneginf(ref)), what + " -Inf"
    fin = np.isfinite(ref)
    assert fin.sum() > c.size // 2
    assert_within_tolerance(c[fin], ref[fin], tol_scale * bound[fin], K,
                            what + " finite part")


@pytest.mark.parametrize("algo", [G.ALGO_AUTO, G.ALGO_TF32X3],
                         ids=["auto", "tf32x3"])
@pytest.mark.parametrize("shape,ws", [
    ((64, 64, 64), False),            # one 128-row tile
    ((300, 260, 1000), True),         # 128-row tiles split over K
    ((512, 384, 2048), True),         # 256-row tiles split over K
    ((700, 300, 2100), False),        # 256-row tiles, whole
    ((2100, 2420, 1000), True)],      # whole tiles and a split tail
    ids=lambda x: "x".join(map(str, x)) if isinstance(x, tuple) else str(x))
def test_nan_and_inf_ieee_tensor(algo, shape, ws):
    """The 3xTF32 kernels give IEEE results for NaN and Inf inputs: the
    outputs the split turns into NaN are recomputed in IEEE arithmetic, so
    ±Inf comes out as ±Inf and NaN only where IEEE has NaN (Inf·0,
    Inf − Inf, a NaN operand)."""
    M, N, K = shape
    a, b = synth.make_operands(M, N, K, seed=K, dist_a="uniform",
                               dist_b="int")
    a, b = _plant_nonfinite(a, b)
    if ws:
        if algo != G.ALGO_AUTO:
            pytest.skip("scratch goes with the automatic plan")
        c, _ = run_gpu_ws(a, b)
        # splits added in the cluster or by the reduction kernel
        with _env("GEMM_F32_CLUSTER_REDUCE", 0):
            c2, need = run_gpu_ws(a, b)
        assert need > 0
        _check_ieee(c2, a, b, f"{shape} reduction kernel")
    else:
        c = run_gpu(a, b, algo, pad=True)
    _check_ieee(c, a, b, f"{shape}")
    assert G.device_status() == 0


def test_nan_and_inf_ieee_streaming_kernel():
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    M = 128 * sms + 77
    assert G.plan(M, 64, 64)["variant"] == "streaming"
    a, b = synth.make_operands(M, 64, 64, seed=8, dist_b="int")
    a, b = _plant_nonfinite(a, b)
    a[M - 1, 0] = np.inf  # the ragged last tile
    _check_ieee(run_gpu(a, b), a, b, "streaming")


@pytest.mark.parametrize("epilogue", [False, True], ids=["plain", "gelu"])
def test_nan_and_inf_ieee_streaming_lane_stores(epilogue):
    """The streaming kernel with C that no tensor map describes (odd row
    stride: per-lane stores), with more than 8 tiles a CTA (the 10-stage
    ring) and, optionally, bias + GELU: non-finite outputs exactly where
    IEEE has them, recomputed after the stores."""
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    M, N, K = 9 * 128 * sms + 77, 60, 40
    assert G.plan(M, N, K)["variant"] == "streaming"
    a, b = synth.make_operands(M, N, K, seed=18, dist_b="int")
    a, b = _plant_nonfinite(a, b)
    a[M - 1, 0] = -np.inf
    store = torch.full((M, N + 1), -5.0, device=DEV)
    bias = synth.make_operands(1, N, 1, seed=19)[1][0]
    if epilogue:
        G.gemm_f32_bias_act(_padded(a), _padded(b),
                            torch.from_numpy(bias).to(DEV), G.ACT_GELU,
                            c=store[:, :N])
    else:
        G.gemm_f32_ex(_padded(a), _padded(b), store[:, :N])
    torch.cuda.synchronize()
    host = store.cpu().numpy()
    assert (host[:, N] == -5.0).all()
    c = host[:, :N]
    if not epilogue:
        _check_ieee(c, a, b, "streaming, lane stores")
        return
    ref, bound, _ = oracle.gemm(a, b)
    want = oracle.epilogue(ref, bias, G.ACT_GELU)
    assert np.array_equal(np.isnan(c), np.isnan(want))
    assert np.array_equal(np.isposinf(c), np.isposinf(want))
    assert np.array_equal(np.isneginf(c), np.isneginf(want))
    fin = np.isfinite(want)
    tol = 1.2 * oracle.tolerance(bound, K) + 4 * 2.0**-24 * (
        np.abs(oracle.epilogue(ref, bias, 0)) + np.abs(want))
    assert (np.abs(c[fin] - want[fin]) <= tol[fin]).all()


@pytest.mark.parametrize("form", ["NT", "TT", "TN"])
def test_nan_and_inf_ieee_transposed_forms(form):
    """Operands read transposed in place (NT, TN: the converters transpose
    A; TT: the swapped product stored transposed)."""
    M, N, K = 300, 260, 520
    a, b = synth.make_operands(M, N, K, seed=3, dist_b="int")
    a, b = _plant_nonfinite(a, b)
    ta, tb = form[0] == "T", form[1] == "T"
    sa = torch.from_numpy(a.T.copy() if ta else a).to(DEV)
    sb = torch.from_numpy(b.T.copy() if tb else b).to(DEV)
    c = torch.full((M, N), -7.0, device=DEV)
    # no scratch: Aᵀ·B is read in place too
    G.gemm_f32_batched_ptr(int(ta), int(tb), M, N, K, sa.data_ptr(),
                           sa.shape[1], 0, sb.data_ptr(), sb.shape[1], 0,
                           c.data_ptr(), N, 0, 1,
                           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    _check_ieee(c.cpu().numpy(), a, b, form)
    if form == "TN":  # and through the transposed copy in scratch
        c2 = G.gemm_f32_batched(sa, sb, trans_a=True)
        torch.cuda.synchronize()
        _check_ieee(c2[0].cpu().numpy(), a, b, "TN copy")


def test_nan_and_inf_ieee_fused_epilogue():
    """bias + GELU after the repair: GELU(+Inf) = +Inf, GELU(-Inf) and
    GELU(NaN) = NaN, as the oracle's float64 epilogue gives."""
    M, N, K = 300, 260, 1000
    a, b = synth.make_operands(M, N, K, seed=5, dist_b="int")
    a, b = _plant_nonfinite(a, b)
    bias = synth.make_operands(1, N, 1, seed=6)[1][0]
    c = G.gemm_f32_bias_act(torch.from_numpy(a).to(DEV),
                            torch.from_numpy(b).to(DEV),
                            torch.from_numpy(bias).to(DEV), G.ACT_GELU)
    torch.cuda.synchronize()
    c = c.cpu().numpy()
    ref, bound, _ = oracle.gemm(a, b)
    want = oracle.epilogue(ref, bias, G.ACT_GELU)
    assert np.array_equal(np.isnan(c), np.isnan(want))
    assert np.array_equal(np.isposinf(c), np.isposinf(want))
    assert np.array_equal(np.isneginf(c), np.isneginf(want))
    fin = np.isfinite(want)
    tol = 1.2 * oracle.tolerance(bound, K) + 4 * 2.0**-24 * (
        np.abs(oracle.epilogue(ref, bias, 0)) + np.abs(want))
    assert (np.abs(c[fin] - want[fin]) <= tol[fin]).all()


def test_stream_ordering_on_side_stream():
    """Work is queued on the given stream, not the default one."""
    a, b = synth.make_operands(512, 512, 512, seed=1)
    ta, tb = torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        tc = G.gemm_f32(ta, tb)
    s.synchronize()
    check_full(a, b, tc.cpu().numpy(), what="side stream")


def test_device_status_clean():
    run_gpu(*synth.make_operands(64, 64, 64, seed=0))
    assert G.device_status() == 0


def test_select_algo_reports_a_kernel():
    ta = torch.zeros(256, 256, device=DEV)
    p = ta.data_ptr()
    assert G.select_algo(256, 256, 256, p, 256, p, 256, p, 256) == G.ALGO_TF32X3
    # misaligned operand or odd leading dimension: the FFMA kernel
    assert G.select_algo(256, 256, 256, p + 4, 256, p, 256, p, 256) == \
        G.ALGO_SIMT
    assert G.select_algo(256, 255, 256, p, 256, p, 255, p, 255) == G.ALGO_SIMT
    # K = 0 is a zero fill, done by the FFMA kernel
    assert G.select_algo(256, 256, 0, p, 0, p, 256, p, 256) == G.ALGO_SIMT


# ------------------------------------------------------------- 3xTF32
@pytest.mark.parametrize("tc_cfg", TC_CFGS)
@pytest.mark.parametrize("shape", [(128, 128, 16), (256, 128, 32),
                                   (64, 64, 64), (1000, 1000, 1000),
                                   (300, 260, 77), (129, 65, 33),
                                   (517, 3, 260), (8, 1000, 8), (1, 1, 1),
                                   (700, 520, 2000)])
def test_tf32x3_shapes(shape, tc_cfg):
    M, N, K = shape
    a, b = synth.make_operands(M, N, K, seed=M * 3 + N * 5 + K)
    with _env("GEMM_F32_TC_CFG", tc_cfg):
        check_full(a, b, run_gpu(a, b, G.ALGO_TF32X3, pad=True),
                   what=f"tf32x3 cfg{tc_cfg} {shape}")
        ai, bi = synth.make_operands(M, N, K, seed=M + N + K, dist_a="int",
                                     dist_b="int")
        check_full(ai, bi, run_gpu(ai, bi, G.ALGO_TF32X3, pad=True),
                   exact=True, what=f"tf32x3 cfg{tc_cfg} {shape} int")
    assert G.device_status() == 0


@pytest.mark.parametrize("tc_cfg", TC_CFGS)
def test_tf32x3_identity_is_exact(tc_cfg):
    """A·I = A and I·B = B bit for bit when every value's TF32 big/small
    split is exact (the two lowest mantissa bits clear).  For the raw-operand
    configurations this pins the tensor core's reading of an fp32 operand to
    TF32 truncation: rounding it would move about half of the values."""
    rng = np.random.default_rng(23)
    x = rng.standard_normal((192, 64)).astype(np.float32)
    x = (x.view(np.uint32) & np.uint32(0xFFFFFFFC)).view(np.float32)
    eye = np.eye(64, dtype=np.float32)
    with _env("GEMM_F32_TC_CFG", tc_cfg):
        c = run_gpu(x, eye, G.ALGO_TF32X3)
        assert np.array_equal(c.view(np.uint32), x.view(np.uint32)), \
            f"A·I != A in {int((c != x).sum())} places"
        xt = np.ascontiguousarray(x[:64, :])
        c = run_gpu(eye, xt, G.ALGO_TF32X3)
        assert np.array_equal(c.view(np.uint32), xt.view(np.uint32)), \
            f"I·B != B in {int((c != xt).sum())} places"


def test_tf32x3_wide_dynamic_range():
    """Operands spanning many binades keep the per-element tolerance."""
    rng = np.random.default_rng(17)
    M, N, K = 200, 190, 300
    a = (rng.standard_normal((M, K)) * 2.0 ** rng.integers(-20, 20, (M, K))
         ).astype(np.float32)
    b = (rng.standard_normal((K, N)) * 2.0 ** rng.integers(-20, 20, (K, N))
         ).astype(np.float32)
    check_full(a, b, run_gpu(a, b, G.ALGO_TF32X3, pad=True),
               what="wide range")


def test_tf32x3_unsupported_when_misaligned():
    ta = torch.zeros(64 * 64 + 1, device=DEV)
    p = ta.data_ptr()
    with pytest.raises(G.GemmError) as e:
        G.gemm_f32_ptr(8, 8, 8, p + 4, 8, p, 8, p, 8, 0, G.ALGO_TF32X3)
    assert e.value.status == 2
    with pytest.raises(G.GemmError):
        G.gemm_f32_ptr(8, 7, 8, p, 8, p, 7, p, 7, 0, G.ALGO_TF32X3)


@pytest.mark.parametrize("tc_cfg", TC_CFGS)
def test_tf32x3_timeout_path_reports_and_recovers(tc_cfg):
    """A producer that issues no copies makes every wait run out: the
    kernel frees TMEM, leaves, and the status word says TIMEOUT; the next
    call works."""
    a, b = synth.make_operands(300, 200, 100, seed=2)
    with _env("GEMM_F32_TC_CFG", tc_cfg):
        old_t = G.set_wait_timeout_ns(2_000_000)
        old_f = G.set_debug_flags(G.DEBUG_STALL_PRODUCER)
        try:
            run_gpu(a, b, G.ALGO_TF32X3, pad=True)
            assert G.device_status() == 4
        finally:
            G.set_debug_flags(old_f)
            G.set_wait_timeout_ns(old_t)
        assert G.device_status() == 0
        check_full(a, b, run_gpu(a, b, G.ALGO_TF32X3, pad=True),
                   what="after timeout")
    assert G.device_status() == 0


# ------------------------------------------------------------- streaming
def _tile_rows():
    """Rows that give every SM one 128-row tile: the smallest M for which
    the automatic plan streams A past a B held in tensor memory."""
    return torch.cuda.get_device_properties(DEV).multi_processor_count * 128


def _stream_shapes():
    r = _tile_rows()
    return [(65536, 64, 64),         # the tall-skinny workload
            (r + 77, 128, 128),      # B at the kernel's limits
            (r, 1, 1),
            (2 * r + 5, 100, 77),    # ragged N and K, a partial last tile
            (r + 1, 33, 16),
            (3 * r - 3, 65, 120),
            (9 * r + 77, 64, 64),    # > 8 tiles a CTA: the 10-stage ring
            (9 * r + 5, 128, 128)]   # the same with B at the limits


@pytest.mark.parametrize("case", range(8))
def test_stream_kernel_shapes(case):
    """N <= 128, K <= 128 and a tile per SM: the persistent kernel that
    keeps Bᵀ in TMEM; every element against the oracle, and integers
    exact."""
    M, N, K = _stream_shapes()[case]
    a, b = synth.make_operands(M, N, K, seed=case, dist_a="normal",
                               dist_b="normal")
    check_full(a, b, run_gpu(a, b, pad=True), what=f"stream {M}x{N}x{K}")
    ai, bi = synth.make_operands(M, N, K, seed=case + 50, dist_a="int",
                                 dist_b="int")
    check_full(ai, bi, run_gpu(ai, bi, pad=True), exact=True,
               what=f"stream int {M}x{N}x{K}")
    assert G.device_status() == 0


def test_device_free_plans_equal_the_device_plans():
    """The planner given this GPU's SM count (no CUDA call) decides as the
    one that queries the device."""
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    major = torch.cuda.get_device_properties(DEV).major
    for M, N, K in [(4096, 4096, 4096), (8192, 3072, 768), (1024,) * 3,
                    (1000,) * 3, (65536, 64, 64), (64, 64, 64),
                    (300, 700, 4096), (19456, 1, 1), (517, 300, 77)]:
        assert G.plan(M, N, K) == G.plan(M, N, K, sm_count=sms,
                                         cc_major=major), (M, N, K)
        assert G.mixed_plan(M, N, K) == G.mixed_plan(M, N, K,
                                                     sm_count=sms), (M, N, K)


def test_plan_reports_the_streaming_kernel():
    """gemm_f32_plan: the streaming variant exactly for N, K <= 128 with a
    128-row tile per SM (and not with GEMM_F32_STREAM=0); tiled otherwise."""
    r = _tile_rows()
    for M, N, K in _stream_shapes():
        assert G.plan(M, N, K) == {"algo": G.ALGO_TF32X3,
                                   "variant": "streaming", "splits": 1,
                                   "whole_tiles": 0, "tile_rows": 128}, \
            (M, N, K)
    for M, N, K in [(r - 128, 64, 64), (r, 129, 64), (r, 64, 129),
                    (4096, 4096, 4096)]:
        assert G.plan(M, N, K)["variant"] == "tiled", (M, N, K)
    with _env("GEMM_F32_STREAM", 0):
        assert G.plan(65536, 64, 64)["variant"] == "tiled"
    # unaligned operands: the FFMA kernel
    assert G.plan(65536, 64, 64, a_ptr=20)["algo"] == G.ALGO_SIMT
    with pytest.raises(G.GemmError):
        G.plan(-1, 4, 4)


def test_stream_kernel_off_matches_oracle_too():
    """GEMM_F32_STREAM=0 sends the same shapes to the tiled tensor kernel."""
    for M, N, K in _stream_shapes()[:2]:
        a, b = synth.make_operands(M, N, K, seed=9)
        with _env("GEMM_F32_STREAM", 0):
            c = run_gpu(a, b, pad=True)
        check_full(a, b, c, what=f"tiled {M}x{N}x{K}")


@pytest.mark.parametrize("act", [0, 1])
def test_stream_kernel_bias_act(act):
    M, N, K = _stream_shapes()[3]
    a, b = synth.make_operands(M, N, K, seed=4, dist_a="normal",
                               dist_b="normal")
    bias = synth.make_operands(1, N, 1, seed=8)[1][0]
    c = G.gemm_f32_bias_act(_padded(a), _padded(b),
                            torch.from_numpy(bias).to(DEV), act)
    torch.cuda.synchronize()
    _check_epilogue(a, b, bias, act, c.cpu().numpy(), what=f"stream act {act}")


def test_stream_kernel_odd_ldc():
    """C with an odd leading dimension (lane stores, no alignment needed);
    the padding column is left alone."""
    M, N, K = _tile_rows() + 3, 60, 40
    a, b = synth.make_operands(M, N, K, seed=12)
    store = torch.full((M, N + 1), -5.0, device=DEV)
    G.gemm_f32_ex(_padded(a), _padded(b), store[:, :N])
    torch.cuda.synchronize()
    host = store.cpu().numpy()
    check_full(a, b, host[:, :N], what="stream odd ldc")
    assert (host[:, N] == -5.0).all()


def test_stream_kernel_timeout_path_reports_and_recovers():
    M, N, K = _tile_rows() + 5, 64, 64
    a, b = synth.make_operands(M, N, K, seed=2)
    old_t = G.set_wait_timeout_ns(2_000_000)
    old_f = G.set_debug_flags(G.DEBUG_STALL_PRODUCER)
    try:
        run_gpu(a, b, pad=True)
        assert G.device_status() == 4
    finally:
        G.set_debug_flags(old_f)
        G.set_wait_timeout_ns(old_t)
    assert G.device_status() == 0
    check_full(a, b, run_gpu(a, b, pad=True), what="stream after timeout")
    assert G.device_status() == 0


# ------------------------------------------------------------- split-K
def run_gpu_ws(a, b, ws_bytes=None):
    """C = A·B through gemm_f32_ws with a workspace of the size it asks."""
    M, K = a.shape
    N = b.shape[1]
    need = G.workspace_size(M, N, K) if ws_bytes is None else ws_bytes
    ws = torch.empty(max(need // 4, 1), device=DEV) if need else None
    ta, tb = _padded(a), _padded(b)
    tc = _padded(np.full((M, N), np.nan, np.float32))
    G.gemm_f32(ta, tb, tc, workspace=ws if ws is not None else
               torch.empty(0, device=DEV))
    torch.cuda.synchronize()
    return tc.cpu().numpy(), need


def _slots():
    return 2 * torch.cuda.get_device_properties(DEV).multi_processor_count


def test_workspace_size_policy():
    """Scratch = split tiles × splits × one TILE_M × 128 fp32 partial
    tile; TILE_M = 256 (one CTA per SM) for K >= 2048, else 128 (two CTAs
    per SM)."""
    slots = _slots()
    sms = slots // 2
    tile = 128 * 128 * 4
    # few tiles: all split, slots // tiles ways (at least 8 k stages each);
    # up to 8 ways the splits reduce within a cluster (no scratch), else
    # (or with GEMM_F32_CLUSTER_REDUCE=0) in scratch
    assert G.plan(1024, 1024, 1024)["tile_rows"] == 128
    s1024 = min(slots // 64, 8)
    assert G.workspace_size(1024, 1024, 1024) == (0 if s1024 <= 8 else
                                                  64 * s1024 * tile)
    with _env("GEMM_F32_CLUSTER_REDUCE", 0):
        assert G.workspace_size(1024, 1024, 1024) == 64 * s1024 * tile
    # a partly filled last round of 256 x 128 tiles: its tiles split
    # sms // tail ways
    p = G.plan(4096, 4096, 4096)
    assert p["tile_rows"] == 256
    tail = 512 % sms
    s = min(sms // tail, 4096 // 16 // 8, 16)
    assert G.workspace_size(4096, 4096, 4096) == (tail * s * 2 * tile
                                                  if s > 8 else 0)
    with _env("GEMM_F32_CLUSTER_REDUCE", 0):
        assert G.workspace_size(4096, 4096, 4096) == (tail * s * 2 * tile
                                                      if s > 1 else 0)
    assert p["splits"] == (s if s > 1 else 1)
    assert p["whole_tiles"] == (512 - tail if s > 1 else 0)
    # K below 2048: 128-row tiles; few 256-row tiles are split over K
    assert G.plan(4096, 4096, 1024)["tile_rows"] == 128
    assert G.plan(4096, 4096, 2047)["tile_rows"] == 128
    p = G.plan(1024, 1024, 4096)
    assert p["tile_rows"] == 256
    assert p["splits"] == min(sms // 32, 4096 // 16 // 8, 16)
    assert G.workspace_size(1024, 1024, 4096) == (
        0 if p["splits"] <= 8 else 32 * p["splits"] * 2 * tile)
    with _env("GEMM_F32_CLUSTER_REDUCE", 0):
        assert G.workspace_size(1024, 1024, 4096) == \
            32 * p["splits"] * 2 * tile
    # whole rounds: nothing to split
    assert G.workspace_size(128 * (slots // 19), 128 * 19, 4096) == 0
    assert G.workspace_size(64, 64, 64) == 0               # K too short
    assert G.workspace_size(0, 5, 5) == 0


@pytest.mark.parametrize("shape", [(512, 384, 2048), (1000, 1000, 2100),
                                   (300, 700, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
def test_splitk_256_row_tiles(shape):
    """K >= 2048 with few tiles: 256 × 128 tiles split over K (the split
    count the plan reports), every element against the oracle, integers
    exact."""
    M, N, K = shape
    p = G.plan(M, N, K)
    assert p["tile_rows"] == 256 and p["splits"] > 1, p
    a, b = synth.make_operands(M, N, K, seed=K, dist_a="normal")
    c, need = run_gpu_ws(a, b)
    assert (need > 0) == (p["splits"] > 8)   # clusters up to 8 splits
    check_full(a, b, c, what=f"256 split {shape}")
    ai, bi = synth.make_operands(M, N, K, seed=K + 1, dist_a="int",
                                 dist_b="int")
    ci, _ = run_gpu_ws(ai, bi)
    check_full(ai, bi, ci, exact=True, what=f"256 split {shape} int")
    # the reduction kernel adds the same partials in the same order
    with _env("GEMM_F32_CLUSTER_REDUCE", 0):
        c2, need2 = run_gpu_ws(a, b)
    assert need2 > 0
    assert np.array_equal(c.view(np.uint32), c2.view(np.uint32))


@pytest.mark.parametrize("name", ["sq1024", "rag1000"])
def test_splitk_workloads(name):
    """Every tile split 4 ways: the splits of a tile run as one cluster and
    add their partial tiles in distributed shared memory (no scratch, also
    through gemm_f32 itself); with GEMM_F32_CLUSTER_REDUCE=0 they go
    through scratch and the reduction kernel instead, with the same bits."""
    w = synth.WORKLOADS[name]
    a, b = w.operands()
    assert G.plan(w.M, w.N, w.K)["splits"] > 1
    c, need = run_gpu_ws(a, b)
    assert need == 0
    check_full(a, b, c, what=f"{name} split-K")
    assert np.array_equal(c.view(np.uint32), run_gpu(a, b).view(np.uint32))
    with _env("GEMM_F32_CLUSTER_REDUCE", 0):
        c2, need2 = run_gpu_ws(a, b)
    assert need2 > 0
    assert np.array_equal(c.view(np.uint32), c2.view(np.uint32))
    wi = w.integer_variant()
    ai, bi = wi.operands()
    ci, _ = run_gpu_ws(ai, bi)
    check_full(ai, bi, ci, exact=True, what=f"{wi.name} split-K")
    with _env("GEMM_F32_CLUSTER_REDUCE", 0):
        ci2, _ = run_gpu_ws(ai, bi)
    check_full(ai, bi, ci2, exact=True, what=f"{wi.name} split-K kernel")
    assert G.device_status() == 0


@pytest.mark.parametrize("splits", [2, 3, 5, 16])
@pytest.mark.parametrize("shape", [(300, 260, 1000), (129, 65, 333),
                                   (64, 64, 64), (17, 1000, 520)])
def test_splitk_forced(splits, shape):
    M, N, K = shape
    a, b = synth.make_operands(M, N, K, seed=splits + M)
    with _env("GEMM_F32_SPLITS", splits):
        need = G.workspace_size(M, N, K)
        s = min(splits, (K + 15) // 16, 16)
        tiles = ((M + 127) // 128) * ((N + 127) // 128)
        cluster = 2 <= s <= 8
        assert need == (tiles * s * 128 * 128 * 4 if s > 1 and not cluster
                        else 0)
        c, _ = run_gpu_ws(a, b)
        check_full(a, b, c, what=f"split {splits} {shape}")
        ai, bi = synth.make_operands(M, N, K, seed=splits, dist_a="int",
                                     dist_b="int")
        ci, _ = run_gpu_ws(ai, bi)
        check_full(ai, bi, ci, exact=True, what=f"split {splits} {shape} int")
        if cluster:  # the reduction kernel gives the same bits
            with _env("GEMM_F32_CLUSTER_REDUCE", 0):
                c2, need2 = run_gpu_ws(a, b)
            assert need2 == tiles * s * 128 * 128 * 4
            assert np.array_equal(c.view(np.uint32), c2.view(np.uint32))


def test_splitk_small_workspace_falls_back():
    a, b = synth.WORKLOADS["sq1024"].operands()
    with _env("GEMM_F32_CLUSTER_REDUCE", 0):
        need = G.workspace_size(1024, 1024, 1024)
        assert need > 0
        c, _ = run_gpu_ws(a, b, ws_bytes=need - 4)
    check_full(a, b, c, what="too-small workspace")


# a last round of tiles split over the GPU: 17 x 19 = 323 tiles on 304
# CTA slots leave a 19-tile tail (the bottom tile-row, ragged in M and N
# for the second shape; K ragged too)
TAIL_SHAPES = [(17 * 128, 19 * 128, 512), (2100, 2420, 1000)]


@pytest.mark.parametrize("shape", TAIL_SHAPES,
                         ids=lambda s: "x".join(map(str, s)))
def test_tail_split_shapes(shape):
    M, N, K = shape
    if ((M + 127) // 128) * ((N + 127) // 128) <= _slots():
        pytest.skip("this GPU fills the tiles in one round")
    a, b = synth.make_operands(M, N, K, seed=M + K)
    p = G.plan(M, N, K)
    assert p["splits"] > 1 and p["whole_tiles"] > 0, p
    # the split tail tiles as thread-block clusters (no scratch) ...
    c, need = run_gpu_ws(a, b)
    assert need == 0
    check_full(a, b, c, what=f"tail split {shape}")
    ai, bi = synth.make_operands(M, N, K, seed=N, dist_a="int", dist_b="int")
    ci, _ = run_gpu_ws(ai, bi)
    check_full(ai, bi, ci, exact=True, what=f"tail split {shape} int")
    c2, _ = run_gpu_ws(a, b)
    assert np.array_equal(c.view(np.uint32), c2.view(np.uint32))
    assert np.array_equal(c.view(np.uint32), run_gpu(a, b, pad=True).view(
        np.uint32))
    # ... and through scratch and the reduction kernel: the same bits
    with _env("GEMM_F32_CLUSTER_REDUCE", 0):
        c3, need3 = run_gpu_ws(a, b)
        ci3, _ = run_gpu_ws(ai, bi)
    assert need3 > 0
    assert np.array_equal(c.view(np.uint32), c3.view(np.uint32))
    check_full(ai, bi, ci3, exact=True, what=f"tail split {shape} int kernel")
    assert G.device_status() == 0


def test_tail_split_256_row_tiles():
    """256 × 128 tiles (K >= 2048) with whole tiles in front of a split
    tail: 8 tile columns and enough tile rows to leave a 16-tile or larger
    last round (152 SMs: 21 × 8 = 168 tiles, 152 whole and 16 split 9
    ways).  M, N and K are ragged.  Every element against the oracle,
    integers bit for bit, a repeat bit-identical."""
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    rows = -(-(sms + 16) // 8)
    M, N, K = rows * 256 - 77, 8 * 128 - 50, 2048 + 13
    p = G.plan(M, N, K)
    assert p["tile_rows"] == 256 and p["splits"] > 8, p  # scratch, kernel
    assert p["whole_tiles"] == sms, p
    assert (p["tile_rows"], p["splits"], p["whole_tiles"]) == \
        expected_tail_plan(M, N, K)
    a, b = synth.make_operands(M, N, K, seed=21, dist_a="normal")
    c, need = run_gpu_ws(a, b)
    assert need > 0
    check_full(a, b, c, what="256-row tail split")
    c2, _ = run_gpu_ws(a, b)
    assert np.array_equal(c.view(np.uint32), c2.view(np.uint32))
    ai, bi = synth.make_operands(M, N, K, seed=22, dist_a="int", dist_b="int")
    ci, _ = run_gpu_ws(ai, bi)
    check_full(ai, bi, ci, exact=True, what="256-row tail split int")
    assert G.device_status() == 0


def test_tail_split_fused_epilogue():
    M, N, K = 2100, 2420, 1000
    a, b = synth.make_operands(M, N, K, seed=77, dist_a="normal",
                               dist_b="normal")
    bias = synth.make_operands(1, N, 1, seed=78)[1][0]
    need = G.workspace_size(M, N, K)
    ws = torch.empty(max(need // 4, 1), device=DEV)
    c = G.gemm_f32_bias_act(torch.from_numpy(a).to(DEV),
                            torch.from_numpy(b).to(DEV),
                            torch.from_numpy(bias).to(DEV), G.ACT_GELU,
                            workspace=ws)
    torch.cuda.synchronize()
    _check_epilogue(a, b, bias, G.ACT_GELU, c.cpu().numpy(), "tail gelu")


def test_splitk_deterministic():
    a, b = synth.WORKLOADS["rag1000"].operands()
    c1, _ = run_gpu_ws(a, b)
    c2, _ = run_gpu_ws(a, b)
    assert np.array_equal(c1.view(np.uint32), c2.view(np.uint32))


# ------------------------------------------------------------- host buffers
@pytest.mark.parametrize("shape,pinned,pad", [
    ((1000, 1000, 1000), True, 0), ((2048, 1536, 512), True, 0),
    ((517, 300, 77), True, 3), ((517, 300, 77), False, 5),
    ((9, 7, 0), True, 0), ((1, 1, 1), False, 0),
    # several chunks: equal tile rows with an odd K ([0, 256, 512, 600]),
    # and half-wave ends around wave-sized chunks ([0, 512, 1280, 2048,
    # 2500] on 152 SMs)
    ((600, 30000, 33), True, 0), ((2500, 4096, 24), True, 1)])
def test_host_pipeline(shape, pinned, pad):
    """gemm_f32_host: host operands (strided or not, pinned or not) through
    lent device buffers, chunked and overlapped, equal the oracle."""
    M, N, K = shape
    a, b = synth.make_operands(M, N, K, seed=M + N + K)
    ha = torch.zeros(M, K + pad)
    hb = torch.zeros(K, N + pad)
    hc = torch.full((M, N + pad), float("nan"))
    if pinned:
        ha, hb, hc = ha.pin_memory(), hb.pin_memory(), hc.pin_memory()
    ha[:, :K] = torch.from_numpy(a)
    hb[:, :N] = torch.from_numpy(b)
    da = torch.empty(max(M * K, 1), device=DEV)
    db = torch.empty(max(K * N, 1), device=DEV)
    dc = torch.empty(M * N, device=DEV)
    need = G.workspace_size(M, N, K)
    ws = torch.empty(max(need // 4, 1), device=DEV) if need else None
    s = torch.cuda.Stream()
    G.gemm_f32_host(ha[:, :K], hb[:, :N], hc[:, :N], da, db, dc,
                    workspace=ws, stream=s)
    s.synchronize()
    c = hc[:, :N].numpy()
    if K == 0:
        assert (c == 0).all()
    else:
        check_full(a, b, c, what=f"host {shape}")
    if pad:
        assert torch.isnan(hc[:, N:]).all()   # padding untouched
    assert G.device_status() == 0


# ------------------------------------------------------------- TMA + FFMA
@pytest.mark.parametrize("shape", [(128, 128, 32), (64, 64, 64),
                                   (1000, 1000, 1000), (300, 260, 77),
                                   (129, 65, 33), (1, 1, 1), (8, 1000, 300),
                                   (700, 520, 2000)])
def test_tma_ffma_shapes(shape):
    M, N, K = shape
    a, b = synth.make_operands(M, N, K, seed=M + 7 * N + K)
    check_full(a, b, run_gpu(a, b, G.ALGO_TMA, pad=True),
               what=f"tma {shape}")
    ai, bi = synth.make_operands(M, N, K, seed=K + 1, dist_a="int",
                                 dist_b="int")
    check_full(ai, bi, run_gpu(ai, bi, G.ALGO_TMA, pad=True), exact=True,
               what=f"tma {shape} int")
    assert G.device_status() == 0


def test_tma_ffma_sq4096_full():
    w = synth.WORKLOADS["sq4096"]
    a, b, ref, bound = workload_reference(w)
    assert_within_tolerance(run_gpu(a, b, G.ALGO_TMA), ref, bound, w.K,
                            "tma sq4096")


def test_tma_ffma_unsupported_when_misaligned():
    ta = torch.zeros(64 * 64 + 1, device=DEV)
    p = ta.data_ptr()
    with pytest.raises(G.GemmError) as e:
        G.gemm_f32_ptr(8, 8, 8, p + 4, 8, p, 8, p, 8, 0, G.ALGO_TMA)
    assert e.value.status == 2


def test_tma_ffma_timeout_path_reports_and_recovers():
    a, b = synth.make_operands(300, 200, 100, seed=2)
    old_t = G.set_wait_timeout_ns(2_000_000)
    old_f = G.set_debug_flags(G.DEBUG_STALL_PRODUCER)
    try:
        run_gpu(a, b, G.ALGO_TMA, pad=True)
        assert G.device_status() == 4
    finally:
        G.set_debug_flags(old_f)
        G.set_wait_timeout_ns(old_t)
    check_full(a, b, run_gpu(a, b, G.ALGO_TMA, pad=True), what="tma after")
    assert G.device_status() == 0


def test_simt_ws_timeout_path_reports_and_recovers():
    """The warp-specialised cp.async kernel: a producer that issues no
    copies makes the compute warps' bounded waits run out."""
    a, b = synth.make_operands(300, 200, 100, seed=2)
    old_t = G.set_wait_timeout_ns(2_000_000)
    old_f = G.set_debug_flags(G.DEBUG_STALL_PRODUCER)
    try:
        with _forced(G.ALGO_SIMT, 6):
            run_gpu(a, b, G.ALGO_SIMT, pad=True)
        assert G.device_status() == 4
    finally:
        G.set_debug_flags(old_f)
        G.set_wait_timeout_ns(old_t)
    with _forced(G.ALGO_SIMT, 6):
        check_full(a, b, run_gpu(a, b, G.ALGO_SIMT, pad=True),
                   what="simt ws after")
    assert G.device_status() == 0


@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (1000, 1000, 1000),
                                   (300, 260, 77), (129, 65, 33)],
                         ids=lambda s: "x".join(map(str, s)))
def test_simt_ws_kernel(shape):
    """The warp-specialised cp.async kernel (aligned operands, padded
    leading dimensions): every element against the oracle, integers exact,
    the full-size case included."""
    M, N, K = shape
    a, b = synth.make_operands(M, N, K, seed=M + 7)
    with _forced(G.ALGO_SIMT, 6):
        check_full(a, b, run_gpu(a, b, G.ALGO_SIMT, pad=True),
                   what=f"simt ws {shape}")
    ai, bi = synth.make_operands(M, N, K, seed=M + 8, dist_a="int",
                                 dist_b="int")
    with _forced(G.ALGO_SIMT, 6):
        check_full(ai, bi, run_gpu(ai, bi, G.ALGO_SIMT, pad=True), exact=True,
                   what=f"simt ws {shape} int")
    assert G.device_status() == 0


# ------------------------------------------------------------- batched, op
def _batched_case(form, M, N, K, batch, seed, gap=0, dist="uniform",
                  broadcast_b=False, broadcast_a=False, ws=None):
    """Operands stored as the form says, with `gap` extra floats between
    rows and matrices; returns (host A list, host B list, device views).
    ws: None calls gemm_f32_batched; "full" gemm_f32_batched_ws with the
    scratch gemm_f32_batched_workspace_size asks for (NaN-filled), "short"
    with 256 bytes less."""
    rng_seed = seed
    As, Bs = [], []
    for i in range(batch):
        a, b = synth.make_operands(M, N, K, seed=rng_seed + i, dist_a=dist,
                                   dist_b=dist)
        As.append(As[0] if (broadcast_a and i) else a)
        Bs.append(Bs[0] if (broadcast_b and i) else b)
    ta, tb = form[0] == "T", form[1] == "T"
    a_store = [x.T.copy() if ta else x for x in As]      # stored shapes
    b_store = [x.T.copy() if tb else x for x in Bs]
    ra, ca = a_store[0].shape
    rb, cb = b_store[0].shape
    lda, ldb = ca + gap, cb + gap
    sA, sB = ra * lda + gap, rb * ldb + gap
    na = 1 if broadcast_a else batch
    bufA = torch.full((na * sA + 1,), float("nan"), device=DEV)
    nb = 1 if broadcast_b else batch
    bufB = torch.full((nb * sB + 1,), float("nan"), device=DEV)
    for i in range(na):
        bufA[i * sA:i * sA + ra * lda].view(ra, lda)[:, :ca] = \
            torch.from_numpy(a_store[i]).to(DEV)
    for i in range(nb):
        bufB[i * sB:i * sB + rb * ldb].view(rb, ldb)[:, :cb] = \
            torch.from_numpy(b_store[i]).to(DEV)
    ldc, sC = N + gap, M * (N + gap) + gap
    bufC = torch.full((batch * sC + 1,), -7.0, device=DEV)
    args = (int(ta), int(tb), M, N, K, bufA.data_ptr(), lda,
            0 if broadcast_a else sA, bufB.data_ptr(), ldb,
            0 if broadcast_b else sB, bufC.data_ptr(), ldc, sC, batch)
    if ws is None:
        G.gemm_f32_batched_ptr(*args, torch.cuda.current_stream().cuda_stream)
    else:
        need = G.batched_workspace_size(int(ta), int(tb), M, N, K, batch)
        nbytes = need if ws == "full" else max(need - 256, 0)
        scratch = torch.full((max(nbytes // 4, 1),), float("nan"), device=DEV)
        G.gemm_f32_batched_ws_ptr(*args, scratch.data_ptr() if nbytes else 0,
                                  nbytes,
                                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    host = bufC.cpu().numpy()
    Cs = [host[i * sC:i * sC + M * ldc].reshape(M, ldc) for i in range(batch)]
    return As, Bs, Cs, host, sC, ldc


@pytest.mark.parametrize("form", ["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("shape,batch,gap", [((300, 260, 77), 3, 0),
                                             ((129, 65, 33), 2, 3),
                                             ((64, 64, 64), 4, 4),
                                             ((256, 384, 512), 2, 0),
                                             ((1, 1, 1), 1, 0)])
def test_batched_forms(form, shape, batch, gap):
    M, N, K = shape
    As, Bs, Cs, host, sC, ldc = _batched_case(form, M, N, K, batch, seed=M,
                                              gap=gap)
    for i in range(batch):
        check_full(As[i], Bs[i], Cs[i][:, :N], what=f"{form} b{i} {shape}")
        assert (Cs[i][:, N:] == -7.0).all()          # row padding untouched
    if gap:
        for i in range(batch):                       # gaps between matrices
            assert (host[i * sC + M * ldc:(i + 1) * sC] == -7.0).all()
    Ai, Bi, Ci, _, _, _ = _batched_case(form, M, N, K, batch, seed=K,
                                        gap=gap, dist="int")
    for i in range(batch):
        check_full(Ai[i], Bi[i], Ci[i][:, :N], exact=True,
                   what=f"{form} b{i} {shape} int")
    assert G.device_status() == 0


@pytest.mark.parametrize("form", ["TN", "NN", "NT", "TT"])
@pytest.mark.parametrize("ws", ["full", "short"])
@pytest.mark.parametrize("shape,batch,gap", [((300, 260, 77), 3, 0),
                                             ((129, 65, 33), 2, 3),
                                             ((64, 64, 64), 4, 4),
                                             ((1000, 700, 300), 1, 0),
                                             ((257, 384, 513), 2, 4),
                                             ((1, 1, 1), 1, 0)])
def test_batched_forms_with_workspace(form, ws, shape, batch, gap):
    """gemm_f32_batched_ws: Aᵀ·B through a transposed copy of A when the
    scratch holds it (else in place), every other form as without scratch;
    padding and gaps untouched, integers exact."""
    M, N, K = shape
    As, Bs, Cs, host, sC, ldc = _batched_case(form, M, N, K, batch,
                                              seed=M + 1, gap=gap, ws=ws)
    for i in range(batch):
        check_full(As[i], Bs[i], Cs[i][:, :N], what=f"{form} ws b{i}")
        assert (Cs[i][:, N:] == -7.0).all()
    if gap:
        for i in range(batch):
            assert (host[i * sC + M * ldc:(i + 1) * sC] == -7.0).all()
    Ai, Bi, Ci, _, _, _ = _batched_case(form, M, N, K, batch, seed=K + 1,
                                        gap=gap, dist="int", ws=ws)
    for i in range(batch):
        check_full(Ai[i], Bi[i], Ci[i][:, :N], exact=True,
                   what=f"{form} ws b{i} int")
    assert G.device_status() == 0


@pytest.mark.parametrize("form", ["NN", "NT", "TT", "TN"])
@pytest.mark.parametrize("shape,batch,gap", [((300, 260, 77), 3, 0),
                                             ((257, 384, 513), 2, 4)])
def test_batched_forms_256_row_tiles(form, shape, batch, gap):
    """The 256 × 128 tile configurations of every form (forced; the
    automatic choice takes them for K >= 2048 with a tile per SM): ragged
    edges, padding and gaps untouched, integers exact."""
    M, N, K = shape
    with _env("GEMM_F32_TC_CFG", 3):
        As, Bs, Cs, host, sC, ldc = _batched_case(form, M, N, K, batch,
                                                  seed=M + 3, gap=gap)
        Ai, Bi, Ci, _, _, _ = _batched_case(form, M, N, K, batch, seed=K + 3,
                                            gap=gap, dist="int")
    for i in range(batch):
        check_full(As[i], Bs[i], Cs[i][:, :N], what=f"{form} 256 b{i}")
        assert (Cs[i][:, N:] == -7.0).all()
        check_full(Ai[i], Bi[i], Ci[i][:, :N], exact=True,
                   what=f"{form} 256 b{i} int")
    if gap:
        for i in range(batch):
            assert (host[i * sC + M * ldc:(i + 1) * sC] == -7.0).all()
    assert G.device_status() == 0


def test_tn_workspace_shared_a():
    """Aᵀ·B with strideA = 0: one transposed copy serves every product."""
    As, Bs, Cs, _, _, _ = _batched_case("TN", 300, 200, 136, 4, seed=3,
                                        broadcast_a=True, ws="full")
    for i in range(4):
        check_full(As[i], Bs[i], Cs[i][:, :200], what=f"shared A {i}")


def test_batched_workspace_size():
    M, N, K = 1000, 700, 300
    t_bytes = (M * ((K + 3) // 4 * 4) * 4 + 255) // 256 * 256
    split = G.workspace_size(M, N, K)
    assert G.batched_workspace_size(G.OP_T, G.OP_N, M, N, K, 1) == \
        t_bytes + split
    assert G.batched_workspace_size(G.OP_T, G.OP_N, M, N, K, 3) == 3 * t_bytes
    assert G.batched_workspace_size(G.OP_N, G.OP_N, M, N, K, 1) == split
    assert G.batched_workspace_size(G.OP_N, G.OP_T, M, N, K, 1) == 0
    assert G.batched_workspace_size(G.OP_T, G.OP_T, M, N, K, 2) == 0
    assert G.batched_workspace_size(G.OP_T, G.OP_N, M, N, 0, 1) == 0
    with pytest.raises(G.GemmError):
        G.batched_workspace_size(2, 0, M, N, K, 1)
    with pytest.raises(G.GemmError):
        G.batched_workspace_size(0, 0, -1, N, K, 1)


def test_batched_broadcast_operand():
    As, Bs, Cs, _, _, _ = _batched_case("NT", 200, 150, 96, 5, seed=1,
                                        broadcast_b=True)
    for i in range(5):
        check_full(As[i], Bs[i], Cs[i][:, :150], what=f"broadcast {i}")


def test_batched_binding_and_empty_batch():
    a = torch.from_numpy(np.stack([synth.make_operands(70, 40, 50, seed=i)[0]
                                   for i in range(3)])).to(DEV)
    b = torch.from_numpy(synth.make_operands(1, 60, 50, seed=9)[1].T.copy()
                         ).to(DEV)                      # 60 x 50, used as B^T
    c = G.gemm_f32_batched(a, b, trans_b=True)
    torch.cuda.synchronize()
    bt = b.cpu().numpy().T.copy()
    for i in range(3):
        check_full(a[i].cpu().numpy(), bt, c[i].cpu().numpy(), what=f"bind {i}")
    G.gemm_f32_batched_ptr(0, 0, 4, 4, 4, 8, 4, 16, 8, 4, 16, 8, 4, 16, 0)
    with pytest.raises(G.GemmError):
        G.gemm_f32_batched_ptr(2, 0, 4, 4, 4, 8, 4, 16, 8, 4, 16, 8, 4, 16, 1)
    with pytest.raises(G.GemmError):                   # lda < M for op T
        G.gemm_f32_batched_ptr(1, 0, 8, 4, 4, 8, 4, 32, 8, 4, 16, 8, 4, 32, 1)


@pytest.mark.parametrize("form", ["NN", "NT", "TN", "TT"])
def test_batched_forms_forced_simt(form):
    """The FFMA path for every form (the tensor path takes every form when
    the layouts allow; here every form runs on the FFMA kernel)."""
    with _env("GEMM_F32_AUTO_SIMT", 1):
        As, Bs, Cs, _, _, _ = _batched_case(form, 300, 260, 77, 3, seed=11,
                                            gap=0)
    for i in range(3):
        check_full(As[i], Bs[i], Cs[i][:, :260], what=f"simt {form} b{i}")


@pytest.mark.parametrize("form,ws,shape", [
    ("NT", None, (2048, 1536, 1024)), ("TT", None, (2048, 1536, 1024)),
    ("TN", None, (2048, 1536, 1024)), ("TN", "full", (2048, 1536, 1024)),
    # K >= 2048 and a 256-row tile per SM: the 256 × 128 configurations
    ("NT", None, (2560, 2048, 2048)), ("TT", None, (2048, 2560, 2048)),
    ("TN", "full", (2560, 2048, 2048))])
def test_transposed_forms_large_full(form, ws, shape):
    """op forms on large shapes, every element against the oracle."""
    M, N, K = shape
    As, Bs, Cs, _, _, _ = _batched_case(form, M, N, K, 1, seed=5, ws=ws)
    check_full(As[0], Bs[0], np.ascontiguousarray(Cs[0][:, :N]),
               what=f"{form} large")


# ------------------------------------------------------------- epilogue
def _check_epilogue(a, b, bias, act, c, what):
    """|C - act(C_ref + bias)| within GELU's slope (< 1.2) times the
    product's tolerance plus a few float32 ulps of the epilogue itself."""
    ref, bound, _ = oracle.gemm(a, b)
    want = oracle.epilogue(ref, bias, act)
    z = oracle.epilogue(ref, bias, 0)
    K = a.shape[1]
    tol = 1.2 * (1e-5 * np.sqrt(K) * bound + 1e-30) + \
        4 * 2.0**-24 * (np.abs(z) + np.abs(want)) + 1e-30
    err = np.abs(c.astype(np.float64) - want)
    assert (err <= tol).all(), \
        f"{what}: {int((err > tol).sum())} outside, worst {err.max():.3e}"


@pytest.mark.parametrize("shape,pad,use_ws", [
    ((1024, 1024, 1024), False, True),     # tensor path, split-K reduction
    ((2048, 768, 512), False, False),      # tensor path, epilogue in kernel
    ((300, 260, 77), True, False),         # unaligned: FFMA kernel
    ((129, 65, 33), False, True)])
@pytest.mark.parametrize("with_bias,act", [(True, 1), (False, 1), (True, 0)])
def test_bias_act(shape, pad, use_ws, with_bias, act):
    M, N, K = shape
    a, b = synth.make_operands(M, N, K, seed=M + N, dist_a="normal",
                               dist_b="normal")
    bias = synth.make_operands(1, N, 1, seed=3)[1][0] if with_bias else None
    if pad:  # odd leading dimensions force the FFMA kernel
        ta = torch.zeros(M, K + 1, device=DEV)[:, :K]
        ta.copy_(torch.from_numpy(a))
        tb = torch.zeros(K, N + 1, device=DEV)[:, :N]
        tb.copy_(torch.from_numpy(b))
    else:
        ta, tb = torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV)
    tbias = torch.from_numpy(bias).to(DEV) if with_bias else None
    need = G.workspace_size(M, N, K) if use_ws else 0
    ws = torch.empty(max(need // 4, 1), device=DEV) if use_ws else None
    c = G.gemm_f32_bias_act(ta, tb, tbias, act, workspace=ws)
    torch.cuda.synchronize()
    _check_epilogue(a, b, bias, act, c.cpu().numpy(),
                    f"{shape} bias={with_bias} act={act}")
    assert G.device_status() == 0


def test_bias_exact_on_integers():
    a, b = synth.make_operands(300, 200, 120, seed=4, dist_a="int",
                               dist_b="int")
    bias = np.arange(200, dtype=np.float32) - 100
    c = G.gemm_f32_bias_act(torch.from_numpy(a).to(DEV),
                            torch.from_numpy(b).to(DEV),
                            torch.from_numpy(bias).to(DEV), G.ACT_NONE)
    torch.cuda.synchronize()
    ref, _, _ = oracle.gemm(a, b)
    assert_bitexact(c.cpu().numpy(), oracle.epilogue(ref, bias, 0), "bias int")


def test_bias_act_rejects_bad_activation():
    t = torch.zeros(8, 8, device=DEV)
    with pytest.raises(G.GemmError):
        G.gemm_f32_bias_act(t, t, None, 7)
