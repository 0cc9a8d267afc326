"""gemm_f32_noalloc: the split-K product whose scratch is a static buffer
inside the library, for callers that must not allocate device memory (code
whose device memory all comes from a framework's own pool, or paths where
an allocation's synchronisation and latency are not acceptable).

The entry point is called through the C ABI, twice in a row, and its
output is checked three ways: against the float64 oracle within the
tolerance the other tests use (bit for bit on small-integer inputs), and
bit for bit against gemm_f32_ws (the same product with caller-owned
scratch, which runs the same deterministic split).  The shapes used are
ones whose plan splits over K, so the static buffer is really written and
read.  This file sorts last so that a run stopping at the first failure
has already run every other test; it also passes on its own in a fresh
process.
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


def _noalloc(ta, tb, tc):
    M, K = ta.shape
    N = tb.shape[1]
    G.gemm_f32_noalloc_ptr(M, N, K, ta.data_ptr(), K, tb.data_ptr(), N,
                           tc.data_ptr(), N,
                           torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name", ["sq1024", "rag1000", "rag1000_int",
                                  "sq64"])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(name):
    w = (synth.WORKLOADS[name[:-4]].integer_variant() if name.endswith("_int")
         else synth.WORKLOADS[name])
    a, b = w.operands()
    need = G.workspace_size(w.M, w.N, w.K)
    # 1024^3 and 1000^3 are split over K: the static scratch is used
    assert (need > 0) == (name != "sq64")
    assert need <= G.noalloc_scratch_bytes()
    ta = torch.from_numpy(a).to(DEV)
    tb = torch.from_numpy(b).to(DEV)
    # the existing entry point, with scratch the caller allocates
    ws = torch.empty(max(need // 4, 1), device=DEV)
    c_ws = G.gemm_f32(ta, tb, workspace=ws)
    torch.cuda.synchronize()
    c_ws = c_ws.cpu().numpy()
    ref, bound, _ = oracle.gemm(a, b)
    tc = torch.empty(w.M, w.N, device=DEV)
    free_after = []
    for call in range(2):
        tc.fill_(float("nan"))
        _noalloc(ta, tb, tc)
        torch.cuda.synchronize()
        free_after.append(torch.cuda.mem_get_info(DEV)[0])
        c = tc.cpu().numpy()
        what = f"{w.name} call {call}"
        if w.dist_a == "int":
            assert_bitexact(c, ref, what)
        else:
            assert_within_tolerance(c, ref, bound, w.K, what)
        # same plan, same split, same summation order as gemm_f32_ws
        assert np.array_equal(c.view(np.uint32), c_ws.view(np.uint32)), what
    # the second call took no device memory
    assert free_after[1] == free_after[0]
    assert G.device_status() == 0


def test_noalloc_rejects_products_beyond_its_scratch():
    cap = G.noalloc_scratch_bytes()
    shape = None
    for n in (1536, 1600, 1700, 1800, 1900):
        need = G.workspace_size(n, n, 4096)
        if need > cap:
            shape = (n, n, 4096)
            break
    if shape is None:
        pytest.skip("no candidate shape needs more scratch on this GPU")
    M, N, K = shape
    ta = torch.zeros(M, K, device=DEV)
    tb = torch.zeros(K, N, device=DEV)
    tc = torch.full((M, N), 3.0, device=DEV)
    with pytest.raises(G.GemmError) as e:
        _noalloc(ta, tb, tc)
    assert e.value.status == 5
    torch.cuda.synchronize()
    assert (tc == 3.0).all()  # nothing was launched
