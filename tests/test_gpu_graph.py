"""The entry points inside CUDA graphs: captured once on a stream, replayed
with new data in the same buffers, each replay checked against the oracle.
Graph replay is how a caller removes per-call launch overhead from small
products; the library's one-time set-up happens on the first eager call."""

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


def _capture(fn):
    """fn(stream) run once eagerly (set-up), then captured into a graph."""
    s = torch.cuda.Stream(DEV)
    fn(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn(s)
    return g


@pytest.mark.parametrize("shape", [(64, 64, 64), (1024, 1024, 1024),
                                   (1000, 1000, 1000), (700, 520, 300)],
                         ids=lambda s: "x".join(map(str, s)))
def test_gemm_f32_graph_replay(shape):
    """AUTO product (split-K with scratch where it applies) in a graph."""
    M, N, K = shape
    ops = [synth.make_operands(M, N, K, seed=s) for s in (1, 2)]
    ta = torch.from_numpy(ops[0][0]).to(DEV)
    tb = torch.from_numpy(ops[0][1]).to(DEV)
    tc = torch.empty(M, N, device=DEV)
    need = G.workspace_size(M, N, K)
    ws = torch.empty(max(need // 4, 1), device=DEV)
    g = _capture(lambda s: G.gemm_f32(ta, tb, tc, stream=s, workspace=ws))
    for a, b in ops + ops[:1]:
        ta.copy_(torch.from_numpy(a))
        tb.copy_(torch.from_numpy(b))
        tc.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref, bound, _ = oracle.gemm(a, b)
        assert_within_tolerance(tc.cpu().numpy(), ref, bound, K,
                                what=f"graph {shape}")
    assert G.device_status() == 0


def test_many_products_in_one_graph():
    """Thirty-two small products captured back to back: one replay runs
    them all, each into its own C."""
    M = N = K = 128
    pairs = [synth.make_operands(M, N, K, seed=10 + i, dist_a="int",
                                 dist_b="int") for i in range(32)]
    tas = [torch.from_numpy(a).to(DEV) for a, _ in pairs]
    tbs = [torch.from_numpy(b).to(DEV) for _, b in pairs]
    tcs = [torch.empty(M, N, device=DEV) for _ in pairs]

    def run(s):
        for ta, tb, tc in zip(tas, tbs, tcs):
            G.gemm_f32(ta, tb, tc, stream=s)

    g = _capture(run)
    for tc in tcs:
        tc.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    for (a, b), tc in zip(pairs, tcs):
        ref, _, _ = oracle.gemm(a, b)
        assert_bitexact(tc.cpu().numpy(), ref, what="graph batch")


def test_fused_epilogue_and_batched_in_a_graph():
    a, b = synth.make_operands(512, 384, 256, seed=3, dist_a="normal")
    bias = synth.make_operands(1, 384, 1, seed=4)[1][0]
    ta, tb = torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV)
    tbias = torch.from_numpy(bias).to(DEV)
    tc = torch.empty(512, 384, device=DEV)
    # batched NT: four copies of Aᵀ-free products with B stored transposed
    bt = torch.from_numpy(np.ascontiguousarray(b.T)).to(DEV)
    ba = ta.unsqueeze(0).repeat(4, 1, 1)
    bb = bt.unsqueeze(0).repeat(4, 1, 1)
    bc = torch.empty(4, 512, 384, device=DEV)

    def run(s):
        G.gemm_f32_bias_act(ta, tb, tbias, G.ACT_GELU, tc, stream=s)
        G.gemm_f32_batched(ba, bb, bc, trans_b=True, stream=s)

    g = _capture(run)
    tc.fill_(float("nan"))
    bc.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    ref, bound, _ = oracle.gemm(a, b)
    want = oracle.epilogue(ref, bias, G.ACT_GELU)
    tol = 1.2 * oracle.tolerance(bound, 256) + 4 * 2.0**-24 * (
        np.abs(oracle.epilogue(ref, bias, 0)) + np.abs(want))
    assert (np.abs(tc.cpu().numpy() - want) <= tol).all()
    for i in range(4):
        assert_within_tolerance(bc[i].cpu().numpy(), ref, bound, 256,
                                what=f"graph batched {i}")


def test_mixed_precision_in_a_graph():
    a, b = synth.make_operands(1000, 1300, 520, seed=5, dist_a="int8")
    ta, tb = torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV)
    tc = torch.empty(1000, 1300, device=DEV)
    ws = torch.empty(G.mixed_workspace_size(1000, 1300, 520),
                     dtype=torch.uint8, device=DEV)
    g = _capture(lambda s: G.gemm_f32_mixed(ta, tb, G.MIXED_BF16, tc,
                                            workspace=ws, stream=s))
    tc.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    want, _, _ = oracle.gemm_mixed(a, b, 0)
    assert_bitexact(tc.cpu().numpy(), want, what="graph mixed")
