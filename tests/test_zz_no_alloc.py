"""gemm_f32_noalloc: the split-K product whose scratch is a static buffer
inside the library, for callers that must not allocate device memory (code
whose device memory all comes from a framework's own pool, or paths where
an allocation's synchronisation and latency are not acceptable).

The entry point is called through the C ABI, twice in a row, and its
output is checked three ways: against the float64 oracle within the
tolerance the other tests use (bit for bit on small-integer inputs), and
bit for bit against gemm_f32_ws (the same product with caller-owned
scratch, which runs the same deterministic split).  Most shapes used are
ones whose plan splits the last round of tiles over K, so the static
buffer is really written and read.  This file sorts last so that a run stopping at the first failure
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


# (name, M, N, K, integer): products whose tiles split more than 8 ways
# (few 256 x 128 tiles, long K), the one case a plan still needs scratch,
# one of them ragged and one integer-valued; the transformer-MLP workload
# (its last round split 6 ways), 1024^3 (every tile split 4 ways) and 64^3
# (no split) need none: their splits reduce within thread-block clusters
CASES = [("split16", 256, 256, 4096, False),
         ("split16_ragged", 300, 260, 2100, False),
         ("split16_int", 512, 384, 2048, True),
         ("mlp", 8192, 3072, 768, False),
         ("sq1024", 1024, 1024, 1024, False),
         ("sq64", 64, 64, 64, False)]


@pytest.mark.parametrize("name,M,N,K,integer", CASES,
                         ids=[c[0] for c in CASES])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(
        name, M, N, K, integer):
    if name == "mlp":
        a, b = synth.WORKLOADS["mlp"].operands()
    else:
        dist = "int" if integer else "uniform"
        a, b = synth.make_operands(M, N, K, seed=M + K, dist_a=dist,
                                   dist_b=dist)
    need = G.workspace_size(M, N, K)
    p = G.plan(M, N, K)
    # the static scratch is used where a tile splits more than 8 ways
    assert (need > 0) == (p["splits"] > 8)
    if name.startswith("split16"):
        assert need > 0, p
    assert need <= G.noalloc_scratch_bytes()
    ta = torch.from_numpy(a).to(DEV)
    tb = torch.from_numpy(b).to(DEV)
    # the existing entry point, with scratch the caller allocates
    ws = torch.empty(max(need // 4, 1), device=DEV)
    c_ws = G.gemm_f32(ta, tb, workspace=ws)
    torch.cuda.synchronize()
    c_ws = c_ws.cpu().numpy()
    ref, bound, _ = oracle.gemm(a, b)
    tc = torch.empty(M, N, device=DEV)
    free_after = []
    for call in range(2):
        tc.fill_(float("nan"))
        _noalloc(ta, tb, tc)
        torch.cuda.synchronize()
        free_after.append(torch.cuda.mem_get_info(DEV)[0])
        c = tc.cpu().numpy()
        what = f"{name} call {call}"
        if integer:
            assert_bitexact(c, ref, what)
        else:
            assert_within_tolerance(c, ref, bound, K, what)
        # same plan, same split, same summation order as gemm_f32_ws
        assert np.array_equal(c.view(np.uint32), c_ws.view(np.uint32)), what
    # the second call took no device memory
    assert free_after[1] == free_after[0]
    assert G.device_status() == 0


def test_noalloc_rejects_products_beyond_its_scratch():
    """A split whose partial tiles need more than the static buffer holds
    is refused with GEMM_F32_ERR_SCRATCH_LIMIT and nothing runs (nine
    256 x 128 tiles split 16 ways: about 19 MB on 152 SMs)."""
    cap = G.noalloc_scratch_bytes()
    shape = None
    for rows in range(1, 9):
        for cols in range(1, 9):
            need = G.workspace_size(256 * rows, 128 * cols, 4096)
            if need > cap:
                shape = (256 * rows, 128 * cols, 4096)
                break
        if shape:
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
