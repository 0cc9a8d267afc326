"""matmul(): operands as PyTorch hands them over -- row-major, transposed
views (w.t()), batched with a shared operand -- read in place and checked
against the oracle on the logical matrices."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_02_gb300 import synth
from helpers import assert_within_tolerance

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from dense_fp32_matrix_02_gb300 import gemm as G  # noqa: E402

DEV = torch.device("cuda:0")


def _dev(x, transposed):
    """Device tensor with the values of x; as a transposed view when asked
    (storage holds xᵀ row-major)."""
    if transposed:
        return torch.from_numpy(np.ascontiguousarray(x.T)).to(DEV).t()
    return torch.from_numpy(x).to(DEV)


@pytest.mark.parametrize("ta,tb", [(False, False), (False, True),
                                   (True, False), (True, True)])
@pytest.mark.parametrize("shape", [(512, 384, 256), (333, 257, 129),
                                   (1, 65, 17), (64, 1, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_matmul_views(shape, ta, tb):
    M, N, K = shape
    a, b = synth.make_operands(M, N, K, seed=M + N, dist_a="normal")
    A, B = _dev(a, ta), _dev(b, tb)
    assert A.shape == (M, K) and B.shape == (K, N)
    c = G.matmul(A, B)
    torch.cuda.synchronize()
    ref, bound, _ = oracle.gemm(a, b)
    assert_within_tolerance(c.cpu().numpy(), ref, bound, K,
                            what=f"matmul {shape} {ta} {tb}")


def test_matmul_batched_with_shared_weight():
    """x (batch × M × K) @ w.t() with w stored N × K, as a linear layer."""
    batch, M, N, K = 6, 200, 96, 160
    xs = [synth.make_operands(M, N, K, seed=50 + i)[0] for i in range(batch)]
    w = synth.make_operands(N, 1, K, seed=60)[0]  # N × K
    X = torch.from_numpy(np.stack(xs)).to(DEV)
    W = torch.from_numpy(w).to(DEV)
    c = G.matmul(X, W.t())
    torch.cuda.synchronize()
    for i in range(batch):
        ref, bound, _ = oracle.gemm(xs[i], np.ascontiguousarray(w.T))
        assert_within_tolerance(c[i].cpu().numpy(), ref, bound, K,
                                what=f"linear {i}")


def test_matmul_rejects_other_layouts():
    x = torch.zeros(8, 8, 2, device=DEV)[:, :, 0]  # both strides > 1
    with pytest.raises(ValueError):
        G.matmul(x, torch.zeros(8, 8, device=DEV))
    with pytest.raises(ValueError):
        G.matmul(torch.zeros(4, 5, device=DEV), torch.zeros(6, 7, device=DEV))


def test_matmul_transposed_a_on_a_side_stream():
    """Aᵀ·B through a transposed copy in scratch the binding allocates: on
    a stream other than the current one, repeated with fresh allocations in
    between, every result stays right (the scratch is not handed out again
    while the side stream may still use it)."""
    M, N, K = 640, 512, 384
    side = torch.cuda.Stream(DEV)
    outs, wants = [], []
    for i in range(4):
        a, b = synth.make_operands(M, N, K, seed=60 + i, dist_a="normal")
        at = _dev(a, True)
        bt = _dev(b, False)
        side.wait_stream(torch.cuda.current_stream(DEV))
        with torch.cuda.stream(side):
            c = torch.empty(M, N, device=DEV)
        G.matmul(at, bt, out=c, stream=side)
        # allocations on the current stream while the side stream runs
        junk = torch.full((M * K,), float("nan"), device=DEV)
        del junk
        outs.append((c, a, b, at, bt))  # inputs stay alive until the end
    side.synchronize()
    for c, a, b, _, _ in outs:
        want, bound, _ = oracle.gemm(a, b)
        assert_within_tolerance(c.cpu().numpy(), want, bound, K,
                                what="side-stream matmul")
    assert G.device_status() == 0
