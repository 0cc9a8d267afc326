"""The planner on the CPU: which kernel, tile, split and chunking the library
picks, through the device-free entry points (gemm_f32_plan_sms,
gemm_f32_mixed_plan_sms, gemm_f32_host_chunks), which make no CUDA call.

The decisions at 152 SMs are the ones the GB300 measurements and profiles
describe (4096^3: 456 whole 256 x 128 tiles and the last 56 split two ways;
the transformer-MLP shape: 1520 whole 128 x 128 tiles and 16 split six
ways; 1024^3: every tile split four ways; 65536 x 64 x 64: the streaming
kernel).  The invariants below hold for any SM count."""

from __future__ import annotations

import itertools

import pytest

from dense_fp32_matrix_02_gb300 import gemm as G

SMS = 152  # GB300
KNOBS = ["GEMM_F32_TC_CFG", "GEMM_F32_SPLITS", "GEMM_F32_TAIL_SPLIT",
         "GEMM_F32_CLUSTER_REDUCE",
         "GEMM_F32_STREAM", "GEMM_F32_AUTO_SIMT", "GEMM_F32_SIMT_CFG",
         "GEMM_F32_MIXED_NARROW", "GEMM_F32_MIXED_BM"]


@pytest.fixture(scope="module")
def built_lib():
    from dense_fp32_matrix_02_gb300 import build
    return build.build()


@pytest.fixture(autouse=True)
def default_knobs(built_lib, monkeypatch):
    for k in KNOBS:
        monkeypatch.delenv(k, raising=False)


@pytest.mark.parametrize("shape,want", [
    ((4096, 4096, 4096), (3, "tiled", 2, 456, 256)),
    ((8192, 3072, 768), (3, "tiled", 6, 1520, 128)),
    ((1024, 1024, 1024), (3, "tiled", 4, 0, 128)),
    ((1000, 1000, 1000), (3, "tiled", 4, 0, 128)),
    ((65536, 64, 64), (3, "streaming", 1, 0, 128)),
    ((64, 64, 64), (3, "tiled", 1, 1, 128)),
])
def test_plans_of_the_measured_workloads(shape, want):
    p = G.plan(*shape, sm_count=SMS)
    got = (p["algo"], p["variant"], p["splits"], p["whole_tiles"],
           p["tile_rows"])
    assert got == want


def test_ffma_kernels_when_the_tensor_path_cannot_run():
    # not the tcgen05 family
    assert G.plan(4096, 4096, 4096, sm_count=SMS, cc_major=9)["algo"] == 1
    # an operand not 16-byte aligned, or a leading dimension not a
    # multiple of 4: the SIMT kernel with scalar copies
    assert G.plan(512, 512, 512, a_ptr=20, sm_count=SMS)["algo"] == 1
    assert G.plan(512, 512, 513, lda=513, sm_count=SMS)["algo"] == 1
    assert G.plan(512, 512, 512, sm_count=SMS)["algo"] == 3


def test_knobs_reach_the_planner(monkeypatch):
    monkeypatch.setenv("GEMM_F32_AUTO_SIMT", "1")
    assert G.plan(4096, 4096, 4096, sm_count=SMS)["algo"] == 1
    monkeypatch.delenv("GEMM_F32_AUTO_SIMT")
    monkeypatch.setenv("GEMM_F32_TAIL_SPLIT", "0")
    p = G.plan(4096, 4096, 4096, sm_count=SMS)
    assert p["splits"] == 1 and p["whole_tiles"] == 512
    monkeypatch.delenv("GEMM_F32_TAIL_SPLIT")
    monkeypatch.setenv("GEMM_F32_STREAM", "0")
    assert G.plan(65536, 64, 64, sm_count=SMS)["variant"] == "tiled"


SHAPES = [(m, n, k) for m, n, k in itertools.product(
    [1, 100, 128, 1000, 4096, 8192, 65536], [1, 64, 128, 129, 1000, 3072],
    [1, 16, 64, 128, 129, 768, 2047, 2048, 4096])]


@pytest.mark.parametrize("sms", [132, 148, 152, 160])
def test_tensor_plan_invariants(sms):
    for M, N, K in SHAPES:
        p = G.plan(M, N, K, sm_count=sms)
        assert p["algo"] == 3, (M, N, K)
        rows = p["tile_rows"]
        if p["variant"] == "streaming":
            assert N <= 128 and K <= 128 and (M + 127) // 128 >= sms
            assert p["splits"] == 1
            continue
        assert rows == (256 if K >= 2048 else 128), (M, N, K)
        tiles = -(-M // rows) * -(-N // 128)
        slots = (2 if rows == 128 else 1) * sms
        nk = -(-K // 16)
        s, whole = p["splits"], p["whole_tiles"]
        assert 1 <= s <= 16 and 0 <= whole <= tiles
        if s == 1:
            assert whole == tiles
        else:
            split = tiles - whole
            assert split * s <= slots          # the split CTAs fit a round
            assert s <= nk // 8                # >= 8 k-stages per split
            assert whole % slots == 0          # whole rounds before them


@pytest.mark.parametrize("shape,want", [
    ((4096, 4096, 4096), (256, 256, 1, 152, 256)),
    ((8192, 3072, 768), (256, 760, 4, 152, 128)),
    ((1024, 1024, 1024), (256, 0, 4, 128, 128)),
    ((65536, 64, 64), (64, 512, 1, 152, 128)),
])
def test_mixed_plans_of_the_measured_workloads(shape, want):
    p = G.mixed_plan(*shape, sm_count=SMS)
    assert (p["width"], p["whole"], p["parts"], p["grid"], p["rows"]) == want


@pytest.mark.parametrize("sms", [132, 152])
def test_mixed_plan_invariants(sms):
    for M, N, K in SHAPES:
        p = G.mixed_plan(M, N, K, sm_count=sms)
        w, rows = p["width"], p["rows"]
        assert w == (256 if N > 128 else 128 if N > 64 else 64)
        tiles256 = -(-M // 256) * -(-N // 256)
        assert rows == (256 if K >= 2048 and N > 128 and tiles256 >= sms
                        else 128), (M, N, K)
        total = -(-M // rows) * -(-N // w)
        parts, whole = p["parts"], p["whole"]
        assert parts in (1, 2, 4) and parts * 64 <= w
        if parts == 1:
            assert whole == total
        else:
            tail = total - whole
            assert tail == total % sms and tail * parts <= sms
        units = whole + (total - whole) * parts
        assert p["grid"] == min(units, sms)


def test_host_chunks_of_the_measured_workloads():
    assert G.host_chunks(4096, 4096, SMS) == [0, 512, 1536, 2560, 3584, 4096]
    assert G.host_chunks(1024, 1024, SMS) == [0, 1024]


@pytest.mark.parametrize("sms", [132, 152])
def test_host_chunk_invariants(sms):
    for M, N in itertools.product([1, 127, 128, 1000, 4096, 8192, 65536,
                                   1 << 20], [1, 64, 1000, 4096, 30000]):
        b = G.host_chunks(M, N, sms)
        assert b[0] == 0 and b[-1] == M and 1 <= len(b) - 1 <= 16
        assert all(x < y for x, y in zip(b, b[1:])), (M, N, b)
        assert all(x % 128 == 0 for x in b[:-1]), (M, N, b)
        per_rb = -(-N // 128)
        wave = max(1, 2 * sms // per_rb) * 128      # rows in one wave
        if M >= 2 * wave and wave >= 256:
            sizes = [y - x for x, y in zip(b, b[1:])]
            assert sizes[0] == wave // 256 * 128    # half a wave first
            assert sizes[-1] <= sizes[0]            # and at most that last
            if len(b) - 1 < 16:
                assert max(sizes[1:-1]) <= wave     # at most a wave between


def test_device_free_queries_reject_bad_arguments():
    lib = G.lib()
    import ctypes
    out = (ctypes.c_int64 * 5)()
    assert lib.gemm_f32_plan_sms(4, 4, 4, 16, 4, 16, 4, 16, 4, 0, 10,
                                 out) == 1
    assert lib.gemm_f32_plan_sms(4, 4, 4, 16, 4, 16, 4, 16, 4, 152, 10,
                                 None) == 1
    assert lib.gemm_f32_plan_sms(-1, 4, 4, 16, 4, 16, 4, 16, 4, 152, 10,
                                 out) == 1
    assert lib.gemm_f32_mixed_plan_sms(4, 4, 4, 0, out) == 1
    assert lib.gemm_f32_mixed_plan_sms(0, 4, 4, 152, out) == 1
    bounds = (ctypes.c_int64 * 17)()
    assert lib.gemm_f32_host_chunks(0, 4, 152, bounds) == -1
    assert lib.gemm_f32_host_chunks(4, 4, 0, bounds) == -1
    assert lib.gemm_f32_host_chunks(4, 4, 152, None) == -1
