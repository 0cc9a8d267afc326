"""The checked build (libgemm_f32_debug.so): the FFMA and tensor kernels
test every shared-memory, tensor-memory and global index they compute
against its extent, report a failure through the status word and skip the
access.  It stands in for a memory checker: a run of the sweep and of the
ragged, split, streaming and transposed shapes under it must give the
oracle's results with no check firing, and the probe shows that a check
does report.  Runs in a process of its own (tests/checked_run.py), since
the library a process loads is fixed at its first call.
"""

from __future__ import annotations

import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_runs_clean():
    from dense_fp32_matrix_02_gb300 import build
    path = build.build(checked=True)
    env = dict(os.environ, GEMM_F32_LIBRARY=path)
    env.pop("GEMM_F32_SIMT_CFG", None)
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_run.py")],
                       env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "checked run ok" in r.stdout
