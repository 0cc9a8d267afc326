"""Runs the FFMA and tensor kernels of the checked build on the sweep and
the ragged, split, streaming and transposed shapes; every result against
the oracle, and no index check may fire.

Run by tests/test_gpu_checked.py in a process of its own, with
GEMM_F32_LIBRARY pointing at libgemm_f32_debug.so (the library a process
loads is fixed at its first call).  Prints "checked run ok" at the end.
"""

from __future__ import annotations

import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
from dense_fp32_matrix_02_gb300 import gemm as G  # noqa: E402
from dense_fp32_matrix_02_gb300 import synth  # noqa: E402
from helpers import assert_bitexact, assert_within_tolerance  # noqa: E402

DEV = torch.device("cuda:0")


def padded(x):
    rows, cols = x.shape
    ld = max(4, (cols + 3) // 4 * 4)
    store = torch.zeros(max(rows, 1), ld, device=DEV)
    store[:rows, :cols] = torch.from_numpy(x).to(DEV)
    return store[:rows, :cols]


def run(a, b, algo=G.ALGO_AUTO, pad=False, ws=False):
    M, K = a.shape
    N = b.shape[1]
    if pad or ws:
        ta, tb = padded(a), padded(b)
        tc = padded(np.full((M, N), np.nan, np.float32))
    else:
        ta = torch.from_numpy(a).to(DEV)
        tb = torch.from_numpy(b).to(DEV)
        tc = torch.full((M, N), float("nan"), device=DEV)
    if ws:
        need = G.workspace_size(M, N, K)
        w = torch.empty(max(need // 4, 1), device=DEV)
        G.gemm_f32(ta, tb, tc, workspace=w)
    else:
        G.gemm_f32_ex(ta, tb, tc, algo=algo)
    torch.cuda.synchronize()
    return tc.cpu().numpy()


def check(a, b, c, what):
    ref, bound, _ = oracle.gemm(a, b)
    if np.all(np.round(a) == a) and np.all(np.round(b) == b) and \
            np.abs(a).max(initial=0) <= 2 and np.abs(b).max(initial=0) <= 2:
        assert_bitexact(c, ref, what)
    else:
        assert_within_tolerance(c, ref, bound, a.shape[1], what)


def status_clean(what):
    st = G.device_status()
    assert st == 0, f"{what}: device status {st} ({G.status_string(st)})"


def main():
    assert G.bounds_checked(), "not the checked build"
    # the check reports (nothing is accessed through the probed index)
    G.bounds_probe()
    assert G.device_status() == 6, "the probe's index check did not report"
    status_clean("after the probe")

    # the sweep, on every kernel family
    paths = [("simt-unpadded", G.ALGO_AUTO, False),
             ("tensor", G.ALGO_TF32X3, True), ("tma", G.ALGO_TMA, True),
             ("simt", G.ALGO_SIMT, True)]
    for M in (1, 5, 16, 17):
        for N in range(1, 18):
            for K in (1, 4, 7, 16, 17):
                a, b = synth.make_operands(M, N, K, seed=M * 1000 + N * 10 + K,
                                           dist_a="int", dist_b="int")
                for name, algo, pad in paths:
                    check(a, b, run(a, b, algo, pad), f"{name} {M}x{N}x{K}")
    status_clean("sweep")

    # ragged shapes on every family, every SIMT tile configuration
    for shape in ((1000, 1000, 1000), (300, 260, 77), (129, 65, 33),
                  (64, 64, 64)):
        a, b = synth.make_operands(*shape, seed=sum(shape))
        for name, algo, pad in paths:
            check(a, b, run(a, b, algo, pad), f"{name} {shape}")
        for cfg in range(6):
            os.environ["GEMM_F32_SIMT_CFG"] = str(cfg)
            check(a, b, run(a, b, G.ALGO_SIMT, True), f"simt{cfg} {shape}")
        os.environ.pop("GEMM_F32_SIMT_CFG")
    status_clean("ragged")

    # split-K (128- and 256-row tiles), a split tail, the streaming kernel
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    for shape in ((300, 260, 1000), (512, 384, 2048), (2100, 2420, 1000),
                  (1000, 1000, 2100), (128 * sms + 77, 64, 64),
                  (-(-(sms + 16) // 8) * 256 - 77, 974, 2061)):
        a, b = synth.make_operands(*shape, seed=shape[2], dist_a="normal")
        check(a, b, run(a, b, ws=True), f"split {shape}")
    status_clean("split")

    # transposed forms, in place (no scratch) and through the copy
    M, N, K = 300, 260, 520
    a, b = synth.make_operands(M, N, K, seed=3)
    for ta in (False, True):
        for tb in (False, True):
            sa = torch.from_numpy(a.T.copy() if ta else a).to(DEV)
            sb = torch.from_numpy(b.T.copy() if tb else b).to(DEV)
            c = torch.full((M, N), -7.0, device=DEV)
            G.gemm_f32_batched_ptr(int(ta), int(tb), M, N, K, sa.data_ptr(),
                                   sa.shape[1], 0, sb.data_ptr(), sb.shape[1],
                                   0, c.data_ptr(), N, 0, 1,
                                   torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            check(a, b, c.cpu().numpy(), f"op {int(ta)}{int(tb)}")
            if ta and not tb:
                c2 = G.gemm_f32_batched(sa, sb, trans_a=True)
                torch.cuda.synchronize()
                check(a, b, c2[0].cpu().numpy(), "op TN copy")
    status_clean("transposed")

    # fused bias + GELU, NaN / Inf inputs (the repair path)
    a, b = synth.make_operands(300, 260, 1000, seed=5, dist_b="int")
    a[5, 7] = np.inf
    b[9, 11] = -np.inf
    c = run(a, b, G.ALGO_TF32X3, True)
    ref, _, _ = oracle.gemm(a, b)
    assert np.array_equal(np.isnan(c), np.isnan(ref))
    assert np.array_equal(np.isinf(c), np.isinf(ref))
    bias = synth.make_operands(1, 260, 1, seed=6)[1][0]
    a, b = synth.make_operands(300, 260, 1000, seed=5)
    G.gemm_f32_bias_act(torch.from_numpy(a).to(DEV),
                        torch.from_numpy(b).to(DEV),
                        torch.from_numpy(bias).to(DEV), G.ACT_GELU)
    torch.cuda.synchronize()
    status_clean("epilogue and repair")
    print("checked run ok", flush=True)


if __name__ == "__main__":
    main()
