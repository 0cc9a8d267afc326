"""GPU parity of the mixed-precision products against the float64 oracle.

"Rendre le GPU rapide", "Les Tensor Cores": only the operands of the
multiply are 16-bit (bfloat16, or binary16); products and sums are fp32.
The oracle of such a product is the float64 product of the rounded operands
(``oracle.gemm_mixed``).  Acceptance: the rounding kernel bit for bit; the
products bit for bit on integers in [-8, 8] (the pages' exactness test) and
within |C - C_ref| <= 1e-5·sqrt(K)·(|A|·|B|)_ij + 1e-30 (A, B the rounded
operands) otherwise.
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
TYPES = [G.MIXED_BF16, G.MIXED_F16]
TYPE_IDS = ["bf16", "f16"]
DTYPE = {G.MIXED_BF16: torch.bfloat16, G.MIXED_F16: torch.float16}


def _dev16(h, t, ld=None):
    """Device 16-bit matrix holding the patterns h (uint16), row stride ld
    (default: the width rounded up to a multiple of 8)."""
    rows, cols = h.shape
    ld = ld or max(8, (cols + 7) // 8 * 8)
    store = torch.zeros(max(rows, 1), ld, dtype=torch.int16, device=DEV)
    store[:rows, :cols] = torch.from_numpy(
        np.ascontiguousarray(h).view(np.int16)).to(DEV)
    return store.view(DTYPE[t])[:rows, :cols]


def run_mixed16(a, b, t):
    """Rounds a, b with the oracle, multiplies the 16-bit copies on the GPU."""
    ah, bh = oracle.round_half(a, t), oracle.round_half(b, t)
    c = torch.full((a.shape[0], b.shape[1]), float("nan"), device=DEV)
    G.gemm_f32_mixed16(_dev16(ah, t), _dev16(bh, t), c)
    torch.cuda.synchronize()
    return c.cpu().numpy()


def run_mixed(a, b, t):
    """fp32 operands in, rounded and multiplied by the library."""
    c = torch.full((a.shape[0], b.shape[1]), float("nan"), device=DEV)
    G.gemm_f32_mixed(torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV),
                     t, c)
    torch.cuda.synchronize()
    return c.cpu().numpy()


# ------------------------------------------------------------- rounding
def _round_sample(rows, cols, seed):
    """fp32 values over every finite exponent with exact ties of both
    formats, overflow candidates and signed zeros, no NaN."""
    rng = np.random.default_rng(seed)
    n = rows * cols
    bits = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
    kind = rng.integers(0, 4, n)
    bits = np.where(kind == 1, (bits & 0xFFFF0000) | 0x8000, bits)
    bits = np.where(kind == 2, (bits & 0xFFFFE000) | 0x1000, bits)
    x = bits.view(np.float32).copy()
    fin = np.isfinite(x)
    x[~fin] = np.float32(1.5)
    small = kind == 3
    e = rng.integers(-30, 17, n)
    x[small] = np.ldexp(1 + rng.random(n) * 0.999, e)[small].astype(np.float32)
    special = np.array([0.0, -0.0, 65520.0, 3.4028234663852886e38],
                       np.float32)
    k = min(n, special.size)
    x[:k] = special[:k]
    return x.reshape(rows, cols)


@pytest.mark.parametrize("t", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("shape", [(123, 457), (256, 512), (1, 3), (9, 8)])
def test_round16_bitexact(t, shape):
    x = _round_sample(*shape, seed=shape[0] + 7 * t)
    got = G.round16(torch.from_numpy(x).to(DEV), t)
    torch.cuda.synchronize()
    got = got.view(torch.int16).cpu().numpy().view(np.uint16)
    assert_bitexact(got.astype(np.float64),
                    oracle.round_half(x, t).astype(np.float64),
                    what=f"round16 {TYPE_IDS[t]} {shape}")


@pytest.mark.parametrize("t", TYPES, ids=TYPE_IDS)
def test_round16_nan_and_strided(t):
    """NaN stays NaN; a strided source and destination are honoured."""
    x = _round_sample(40, 60, seed=3)
    x[5, 7] = np.nan
    src = torch.zeros(40, 70, device=DEV)
    src[:, :60] = torch.from_numpy(x).to(DEV)
    dst = torch.zeros(40, 64, dtype=DTYPE[t], device=DEV)
    G.round16(src[:, :60], t, out=dst[:, :60])
    torch.cuda.synchronize()
    h = dst.view(torch.int16).cpu().numpy().view(np.uint16)
    assert not h[:, 60:].any()
    back = oracle.widen_half(h[:, :60], t)
    assert np.isnan(back[5, 7])
    x[5, 7] = 0.0
    h[5, 7] = 0
    assert np.array_equal(h[:, :60], oracle.round_half(x, t))


# ------------------------------------------------------------- exactness
INT_SHAPES = [(128, 256, 64), (1, 1, 8), (64, 64, 64), (300, 520, 136),
              (257, 255, 1000), (2048, 4096, 256), (4096, 4096, 128)]


@pytest.mark.parametrize("t", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("shape", INT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_mixed16_small_integers_exact(t, shape):
    """The pages' test: integers in [-8, 8] are exact in 16 bits and every
    sum is exact in fp32, so C equals the oracle bit for bit.  The larger
    shapes give every persistent CTA several tiles (both accumulators)."""
    M, N, K = shape
    a, b = synth.make_operands(M, N, K, seed=M + N + K, dist_a="int8")
    want, _, _ = oracle.gemm_mixed(a, b, t)
    assert_bitexact(run_mixed16(a, b, t), want, what=f"mixed16 {shape}")


@pytest.mark.parametrize("t", TYPES, ids=TYPE_IDS)
def test_mixed_small_integers_exact(t):
    a, b = synth.make_operands(300, 520, 137, seed=5, dist_a="int8")
    want, _, _ = oracle.gemm_mixed(a, b, t)
    assert_bitexact(run_mixed(a, b, t), want, what="mixed ints")


# ------------------------------------------------------------- tolerance
@pytest.mark.parametrize("t", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("shape", [(128, 256, 64), (333, 700, 264),
                                   (1024, 2048, 1024)],
                         ids=lambda s: "x".join(map(str, s)))
def test_mixed16_normal_within_tolerance(t, shape):
    M, N, K = shape
    a, b = synth.make_operands(M, N, K, seed=11, dist_a="normal")
    want, bound, _ = oracle.gemm_mixed(a, b, t)
    assert_within_tolerance(run_mixed16(a, b, t), want, bound, K,
                            what=f"mixed16 {shape}")


@pytest.mark.parametrize("t", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("shape", [(100, 130, 77), (512, 1024, 333),
                                   (1000, 1000, 1000), (8192, 64, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_mixed_fp32_operands_within_tolerance(t, shape):
    """fp32 operands of any width (lda = 77 included): the library rounds
    them into its workspace with padded rows, then multiplies."""
    M, N, K = shape
    a, b = synth.make_operands(M, N, K, seed=13)
    want, bound, _ = oracle.gemm_mixed(a, b, t)
    assert_within_tolerance(run_mixed(a, b, t), want, bound, K,
                            what=f"mixed {shape}")


def test_mixed_equals_mixed16_on_the_rounded_operands():
    a, b = synth.make_operands(700, 900, 500, seed=17, dist_a="normal")
    for t in TYPES:
        assert np.array_equal(run_mixed(a, b, t), run_mixed16(a, b, t))


@pytest.mark.parametrize("t", TYPES, ids=TYPE_IDS)
def test_mixed16_large_sampled(t):
    """4096^3: sampled elements against the oracle one by one."""
    M = N = K = 4096
    a, b = synth.make_operands(M, N, K, seed=2, dist_a="normal")
    ar = oracle.widen_half(oracle.round_half(a, t), t)
    br = oracle.widen_half(oracle.round_half(b, t), t)
    c = run_mixed16(a, b, t)
    rng = np.random.default_rng(1)
    rows = rng.integers(0, M, 3000)
    cols = rng.integers(0, N, 3000)
    rows[:4], cols[:4] = [0, M - 1, 0, M - 1], [0, N - 1, N - 1, 0]
    want, bound, _ = oracle.entries(ar, br, rows, cols)
    assert_within_tolerance(c[rows, cols], want, bound, K, what="sampled")


# ------------------------------------------------------------- work units
def _sms():
    return torch.cuda.get_device_properties(DEV).multi_processor_count


def _split_cases():
    """Shapes that reach each way the 16-bit kernel cuts C, for this GPU's
    SM count g: (M, N, K, expected plan)."""
    g = _sms()
    half_tail = g // 2 - 3        # 2 strips fit, 4 do not
    return [
        # one round and a tail of g/2 - 3 tiles: 128-column strips
        ((g + half_tail) * 128 - 5, 256, 72,
         dict(width=256, whole=g, parts=2)),
        # one round and a tail of 8 tiles: 64-column strips
        ((g + 8) * 128 - 77, 256, 40, dict(width=256, whole=g, parts=4)),
        # fewer tiles than SMs: every tile cut in four
        (300, 520, 136, dict(width=256, whole=0, parts=4)),
        # N <= 128: 128-wide tiles, cut in two
        (1000, 100, 200, dict(width=128, whole=0, parts=2)),
        # N <= 64: 64-wide tiles, never cut
        (g * 128 + 1, 40, 64, dict(width=64, whole=g + 1, parts=1)),
        # N = 257: a second column of tiles holding one column of C
        (640, 257, 96, dict(width=256, whole=0, parts=4)),
        # whole rounds only: nothing to cut
        (2 * g * 128, 256, 64, dict(width=256, whole=2 * g, parts=1)),
    ]


def test_mixed_tile_rows_rule():
    """256-row tiles for K >= 2048, N > 128 and a 256 × 256 tile per SM."""
    g = _sms()
    assert G.mixed_plan(4096, 4096, 4096)["rows"] == 256
    assert G.mixed_plan(4096, 4096, 1024)["rows"] == 128
    assert G.mixed_plan(1024, 1024, 4096)["rows"] == 128      # 16 tiles
    assert G.mixed_plan(65536, 64, 4096)["rows"] == 128       # narrow N
    p = G.mixed_plan(256 * g, 256, 2048)                       # one wave
    assert p["rows"] == 256 and p["whole"] == g and p["parts"] == 1


@pytest.mark.parametrize("t", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("shape", [(300, 520, 136), (600, 1000, 2064),
                                   (257, 255, 1000), (1000, 100, 200)],
                         ids=lambda s: "x".join(map(str, s)))
def test_mixed16_256_row_tiles_exact(t, shape, monkeypatch):
    """The 256-row tiles (two MMAs of M = 128 per k-step into one
    accumulator that fills TMEM), forced: ragged rows and columns, strips
    and narrow tiles, integers bit for bit; normal operands within the
    tolerance."""
    monkeypatch.setenv("GEMM_F32_MIXED_BM", "256")
    M, N, K = shape
    assert G.mixed_plan(M, N, K)["rows"] == 256
    a, b = synth.make_operands(M, N, K, seed=M + 1, dist_a="int8")
    want, _, _ = oracle.gemm_mixed(a, b, t)
    assert_bitexact(run_mixed16(a, b, t), want, what=f"mixed16 256 {shape}")
    a, b = synth.make_operands(M, N, K, seed=M + 2, dist_a="normal")
    want, bound, _ = oracle.gemm_mixed(a, b, t)
    assert_within_tolerance(run_mixed16(a, b, t), want, bound, K,
                            what=f"mixed16 256 normal {shape}")


def test_mixed_plan_cases():
    for M, N, _, want in _split_cases():
        got = G.mixed_plan(M, N)
        assert {k: got[k] for k in want} == want, (M, N, got)
        assert 1 <= got["grid"] <= _sms()


@pytest.mark.parametrize("t", TYPES, ids=TYPE_IDS)
@pytest.mark.parametrize("case", range(7))
def test_mixed16_work_units_exact(t, case):
    """Every cut (strips of the last round, narrow tiles, a ragged last
    column of tiles) covers C exactly once: bit for bit on integers."""
    M, N, K, plan = _split_cases()[case]
    a, b = synth.make_operands(M, N, K, seed=100 + case, dist_a="int8")
    want, _, _ = oracle.gemm_mixed(a, b, t)
    assert_bitexact(run_mixed16(a, b, t), want, what=f"mixed16 {plan}")


@pytest.mark.parametrize("case", [0, 1, 3])
def test_mixed16_work_units_normal(case, monkeypatch):
    """Normal operands through the cut and the uncut plan
    (GEMM_F32_MIXED_NARROW=0): both within the tolerance."""
    M, N, K, _ = _split_cases()[case]
    a, b = synth.make_operands(M, N, K, seed=200 + case, dist_a="normal")
    want, bound, _ = oracle.gemm_mixed(a, b, G.MIXED_BF16)
    cut = run_mixed16(a, b, G.MIXED_BF16)
    monkeypatch.setenv("GEMM_F32_MIXED_NARROW", "0")
    assert G.mixed_plan(M, N)["parts"] == 1
    assert G.mixed_plan(M, N)["width"] == 256
    whole = run_mixed16(a, b, G.MIXED_BF16)
    assert_within_tolerance(cut, want, bound, K, what="cut")
    assert_within_tolerance(whole, want, bound, K, what="whole")


# ------------------------------------------------------------- edges, errors
def test_mixed_k_zero_and_empty():
    c = torch.full((5, 7), float("nan"), device=DEV)
    G.gemm_f32_mixed16(torch.zeros(5, 0, dtype=torch.bfloat16, device=DEV),
                       torch.zeros(0, 7, dtype=torch.bfloat16, device=DEV), c)
    torch.cuda.synchronize()
    assert not c.cpu().numpy().any()
    c.fill_(float("nan"))
    G.gemm_f32_mixed(torch.zeros(5, 0, device=DEV),
                     torch.zeros(0, 7, device=DEV), G.MIXED_F16, c)
    torch.cuda.synchronize()
    assert not c.cpu().numpy().any()
    G.gemm_f32_mixed16(torch.zeros(0, 8, dtype=torch.bfloat16, device=DEV),
                       torch.zeros(8, 7, dtype=torch.bfloat16, device=DEV),
                       torch.zeros(0, 7, device=DEV))


def test_mixed16_rejects_unaligned_and_bad_type():
    a = torch.zeros(64, 60, dtype=torch.bfloat16, device=DEV)  # lda = 60
    b = torch.zeros(60, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(G.GemmError) as e:
        G.gemm_f32_mixed16(a, b)
    assert e.value.status == 2
    c = torch.zeros(8, 8, device=DEV)
    x = torch.zeros(8, 8, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(G.GemmError) as e:
        G.gemm_f32_mixed16_ptr(7, 8, 8, 8, x.data_ptr(), 8, x.data_ptr(), 8,
                               c.data_ptr(), 8)
    assert e.value.status == 1
    with pytest.raises(TypeError):
        G.gemm_f32_mixed16(x, x.to(torch.float16))


def test_mixed_rejects_small_workspace():
    a = torch.zeros(64, 64, device=DEV)
    need = G.mixed_workspace_size(64, 64, 64)
    assert need == 64 * 64 * 2 * 2
    ws = torch.zeros(need - 1, dtype=torch.uint8, device=DEV)
    with pytest.raises(G.GemmError) as e:
        G.gemm_f32_mixed(a, a, G.MIXED_BF16, workspace=ws)
    assert e.value.status == 1


def test_mixed16_timeout_path_reports_and_recovers():
    """A producer that issues no copies: every wait runs out, the kernel
    frees TMEM and leaves, the status word says TIMEOUT; the next call
    works."""
    a, b = synth.make_operands(300, 520, 136, seed=4, dist_a="int8")
    old_t = G.set_wait_timeout_ns(2_000_000)
    old_f = G.set_debug_flags(G.DEBUG_STALL_PRODUCER)
    try:
        run_mixed16(a, b, G.MIXED_BF16)
        assert G.device_status() == 4
    finally:
        G.set_debug_flags(old_f)
        G.set_wait_timeout_ns(old_t)
    want, _, _ = oracle.gemm_mixed(a, b, G.MIXED_BF16)
    assert_bitexact(run_mixed16(a, b, G.MIXED_BF16), want, what="after")
    assert G.device_status() == 0


@pytest.mark.parametrize("t", TYPES, ids=TYPE_IDS)
def test_mixed16_unaligned_c_direct_stores(t):
    """C that no tensor map can describe (offset by one element, odd
    leading dimension): the epilogue stores lane by lane, guarded."""
    M, N, K = 300, 520, 136
    a, b = synth.make_operands(M, N, K, seed=41, dist_a="int8")
    ah, bh = oracle.round_half(a, t), oracle.round_half(b, t)
    store = torch.full((M * (N + 3) + 1,), float("nan"), device=DEV)
    c = store[1:].view(M, N + 3)[:, :N]  # 4-byte aligned only, ldc = N + 3
    G.gemm_f32_mixed16(_dev16(ah, t), _dev16(bh, t), c)
    torch.cuda.synchronize()
    want, _, _ = oracle.gemm_mixed(a, b, t)
    assert_bitexact(c.cpu().numpy(), want, what="unaligned C")
    pad = store[1:].view(M, N + 3)[:, N:]
    assert torch.isnan(pad).all()  # the padding is left alone


def test_f16_rounding_overflows_to_inf():
    """fp32 values beyond binary16's range round to ±Inf, as the oracle's
    IEEE rounding says; bfloat16 keeps them finite."""
    x = np.array([[7.0e4, -7.0e4, 65519.0, 65520.0, 1e38, -1e-8]], np.float32)
    for t in TYPES:
        got = G.round16(torch.from_numpy(x).to(DEV), t)
        torch.cuda.synchronize()
        bits = got.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(bits, oracle.round_half(x, t))
