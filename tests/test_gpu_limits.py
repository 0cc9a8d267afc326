"""Limits: products whose C has more than 2^31 elements (64-bit index
arithmetic in every store path), and concurrent calls from several host
threads on their own streams (the header's thread-safety claim)."""

from __future__ import annotations

import threading

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

# 65536 x 40000 = 2.62e9 elements of C (10.5 GB), K short so it stays quick
BIG_M, BIG_N, BIG_K = 65536, 40000, 8


def _sample(M, N, seed=0, count=4096):
    rng = np.random.default_rng(seed)
    rows = rng.integers(0, M, count)
    cols = rng.integers(0, N, count)
    # the far corner, where m·ldc + n is largest
    rows[:4] = [M - 1, M - 1, M - 2, 0]
    cols[:4] = [N - 1, N - 2, N - 1, N - 1]
    return rows, cols


@pytest.mark.parametrize("algo", [G.ALGO_AUTO, G.ALGO_SIMT])
def test_c_beyond_2_31_elements(algo):
    a, b = synth.make_operands(BIG_M, BIG_N, BIG_K, seed=31, dist_a="int",
                               dist_b="int")
    ta = torch.from_numpy(a).to(DEV)
    tb = torch.from_numpy(b).to(DEV)
    tc = torch.full((BIG_M, BIG_N), float("nan"), device=DEV)
    G.gemm_f32_ex(ta, tb, tc, algo=algo)
    rows, cols = _sample(BIG_M, BIG_N)
    got = tc[torch.from_numpy(rows).to(DEV),
             torch.from_numpy(cols).to(DEV)].cpu().numpy()
    del tc
    torch.cuda.empty_cache()
    want, _, _ = oracle.entries(a, b, rows, cols)
    assert_bitexact(got, want, what=f"2^31+ elements, algo {algo}")
    assert G.device_status() == 0


def test_mixed_c_beyond_2_31_elements():
    a, b = synth.make_operands(BIG_M, BIG_N, BIG_K, seed=32, dist_a="int8")
    ta = torch.from_numpy(a).to(DEV).to(torch.bfloat16)  # exact: integers
    tb = torch.from_numpy(b).to(DEV).to(torch.bfloat16)
    tc = torch.full((BIG_M, BIG_N), float("nan"), device=DEV)
    G.gemm_f32_mixed16(ta, tb, tc)
    rows, cols = _sample(BIG_M, BIG_N, seed=1)
    got = tc[torch.from_numpy(rows).to(DEV),
             torch.from_numpy(cols).to(DEV)].cpu().numpy()
    del tc
    torch.cuda.empty_cache()
    want, _, _ = oracle.entries(a, b, rows, cols)
    assert_bitexact(got, want, what="bf16, 2^31+ elements")
    assert G.device_status() == 0


def test_concurrent_host_threads():
    """Eight host threads, each with its own stream and operands, call the
    library at once (ctypes releases the GIL) for several rounds."""
    shapes = [(1024, 1024, 1024), (1000, 1000, 1000), (300, 260, 77),
              (129, 65, 33), (2048, 512, 256), (64, 64, 64), (700, 520, 300),
              (4096, 64, 64)]
    cases = []
    for i, (M, N, K) in enumerate(shapes):
        a, b = synth.make_operands(M, N, K, seed=100 + i)
        ref, bound, _ = oracle.gemm(a, b)
        cases.append((a, b, ref, bound, K))
    errors = []
    barrier = threading.Barrier(len(cases))

    def worker(i):
        try:
            a, b, ref, bound, K = cases[i]
            s = torch.cuda.Stream(DEV)
            with torch.cuda.stream(s):
                ta = torch.from_numpy(a).to(DEV, non_blocking=False)
                tb = torch.from_numpy(b).to(DEV, non_blocking=False)
                tc = torch.empty(a.shape[0], b.shape[1], device=DEV)
                need = G.workspace_size(a.shape[0], b.shape[1], K)
                ws = torch.empty(max(need // 4, 1), device=DEV)
            s.synchronize()
            barrier.wait()
            for _ in range(5):
                G.gemm_f32(ta, tb, tc, stream=s, workspace=ws)
                s.synchronize()
                assert_within_tolerance(tc.cpu().numpy(), ref, bound, K,
                                        what=f"thread {i}")
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(f"thread {i}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,))
               for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert G.device_status() == 0
