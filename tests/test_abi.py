"""The C-ABI library without a GPU: it loads, exports every declared symbol,
and its host-side argument checks answer before any CUDA call."""

import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "gemm_f32.h")


@pytest.fixture(scope="module")
def built_lib():
    from dense_fp32_matrix_02_gb300 import build
    path = build.build()
    return path


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_f32\w*)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("gemm_f32", "gemm_f32_ex", "gemm_f32_status_string",
                 "gemm_f32_last_cuda_error", "gemm_f32_device_status"):
        assert must in names


def test_library_exports_every_declared_symbol(built_lib):
    lib = ctypes.CDLL(built_lib)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"
    out = subprocess.run(["nm", "-D", "--defined-only", built_lib],
                         capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert set(declared_functions()) <= exported
    # nothing else from the implementation leaks into the dynamic table
    ours = {s for s in exported if "gemm" in s.lower()}
    assert ours == set(declared_functions())


def test_status_strings_and_version(built_lib):
    from dense_fp32_matrix_02_gb300 import gemm
    assert gemm.status_string(0) == "ok"
    assert "invalid" in gemm.status_string(1)
    assert gemm.status_string(99) == "unknown status"
    assert gemm.version() >= 100


def _call(lib, M, N, K, A=8, lda=None, B=8, ldb=None, C=8, ldc=None, algo=0):
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    return lib.gemm_f32_ex(M, N, K, A, lda, B, ldb, C, ldc, None, algo)


def test_argument_checks_need_no_gpu(built_lib):
    from dense_fp32_matrix_02_gb300 import gemm
    lib = gemm.lib()
    bad = gemm.GemmError
    assert _call(lib, -1, 4, 4) == 1
    assert _call(lib, 4, -1, 4) == 1
    assert _call(lib, 4, 4, -1) == 1
    assert _call(lib, 4, 4, 8, lda=7) == 1          # lda < K
    assert _call(lib, 4, 8, 4, ldb=7) == 1          # ldb < N
    assert _call(lib, 4, 8, 4, ldc=7) == 1          # ldc < N
    assert _call(lib, 4, 4, 4, A=None) == 1         # null A, non-empty
    assert _call(lib, 4, 4, 4, B=None) == 1
    assert _call(lib, 4, 4, 4, C=None) == 1
    assert _call(lib, 4, 4, 4, algo=9) == 1         # unknown algorithm
    assert _call(lib, 4, 4, 4, algo=-1) == 1
    assert _call(lib, 2**31, 4, 4, lda=4) == 2      # beyond 32-bit sizes
    # empty C: nothing to do, no CUDA call, no pointer needed
    assert _call(lib, 0, 4, 4, A=None, C=None) == 0
    assert _call(lib, 4, 0, 4, B=None, C=None) == 0
    # K == 0 still needs C (it is zero-filled) but not A or B
    assert _call(lib, 4, 4, 0, A=None, B=None, C=None) == 1
    with pytest.raises(bad):
        gemm.gemm_f32_ptr(-1, 1, 1, 8, 1, 8, 1, 8, 1)


def test_query_argument_checks_need_no_gpu(built_lib):
    """The plan and workspace queries reject bad arguments before any
    device call (status 1 = invalid argument)."""
    from dense_fp32_matrix_02_gb300 import gemm
    lib = gemm.lib()
    i64 = ctypes.c_int64
    out = (i64 * 5)()
    # gemm_f32_plan: NULL out, negative sizes, leading dimensions too small
    assert lib.gemm_f32_plan(4, 4, 4, 16, 4, 16, 4, 16, 4, None) == 1
    assert lib.gemm_f32_plan(-1, 4, 4, 16, 4, 16, 4, 16, 4, out) == 1
    assert lib.gemm_f32_plan(4, 4, 8, 16, 7, 16, 4, 16, 4, out) == 1
    # gemm_f32_mixed_plan: M or N < 1, K < 0, NULL out
    assert lib.gemm_f32_mixed_plan(0, 4, 4, out) == 1
    assert lib.gemm_f32_mixed_plan(4, 0, 4, out) == 1
    assert lib.gemm_f32_mixed_plan(4, 4, -1, out) == 1
    assert lib.gemm_f32_mixed_plan(4, 4, 4, None) == 1
    # gemm_f32_batched_workspace_size: unknown form or negative size
    assert lib.gemm_f32_batched_workspace_size(2, 0, 4, 4, 4, 1) == -1
    assert lib.gemm_f32_batched_workspace_size(0, 0, -1, 4, 4, 1) == -1
    assert lib.gemm_f32_batched_workspace_size(0, 0, 4, 4, 4, -1) == -1
    # nothing to do: no scratch, no device call
    assert lib.gemm_f32_batched_workspace_size(1, 0, 4, 4, 0, 1) == 0
    assert lib.gemm_f32_batched_workspace_size(1, 0, 4, 4, 4, 0) == 0
    # gemm_f32_batched_ws: negative scratch or NULL scratch with bytes
    args = (1, 0, 4, 4, 4, 16, 4, 16, 16, 4, 16, 16, 4, 16, 1)
    assert lib.gemm_f32_batched_ws(*args, None, -1, None) == 1
    assert lib.gemm_f32_batched_ws(*args, None, 64, None) == 1


def test_test_hooks_roundtrip(built_lib):
    from dense_fp32_matrix_02_gb300 import gemm
    old = gemm.set_wait_timeout_ns(1000)
    assert gemm.set_wait_timeout_ns(0) == 1000
    assert gemm.set_wait_timeout_ns(old) == 2_000_000_000
    assert gemm.set_debug_flags(1) == 0
    assert gemm.set_debug_flags(0) == 1


def test_binding_rejects_bad_tensors(built_lib):
    torch = pytest.importorskip("torch")
    from dense_fp32_matrix_02_gb300 import gemm
    a = torch.zeros(4, 4)
    with pytest.raises(ValueError):          # host tensor
        gemm.gemm_f32(a, a)
    with pytest.raises(TypeError):
        gemm.gemm_f32(a.double(), a.double())


def test_product_has_no_oracle_or_cpu_fallback():
    """The package neither imports the oracle nor computes on the CPU."""
    pkg = os.path.join(ROOT, "dense_fp32_matrix_02_gb300")
    for name in os.listdir(pkg):
        if not name.endswith(".py"):
            continue
        text = open(os.path.join(pkg, name), encoding="utf-8").read()
        assert "oracle" not in text.replace("float64 oracle", ""), name
        assert "torch.matmul" not in text and "np.matmul" not in text, name
        assert " @ " not in text, name


C_PROGRAM = r"""
/* A plain C99 caller of the library: only the public header, no CUDA
   headers, no C++.  Every call below is answered by the host-side checks,
   before any CUDA call, so no GPU is needed. */
#include <stdio.h>
#include <string.h>
#include "gemm_f32.h"

static int fails = 0;
#define EXPECT(cond) do { if (!(cond)) { printf("FAIL %s\n", #cond); ++fails; } } while (0)

int main(void) {
    float a[4] = {0}, b[4] = {0}, c[4] = {0};
    EXPECT(gemm_f32_version() >= 100);
    EXPECT(strcmp(gemm_f32_status_string(GEMM_F32_OK), "ok") == 0);
    EXPECT(gemm_f32(-1, 2, 2, a, 2, b, 2, c, 2, NULL) == GEMM_F32_ERR_INVALID_ARG);
    EXPECT(gemm_f32(2, 2, 2, a, 1, b, 2, c, 2, NULL) == GEMM_F32_ERR_INVALID_ARG);
    EXPECT(gemm_f32(2, 2, 2, NULL, 2, b, 2, c, 2, NULL) == GEMM_F32_ERR_INVALID_ARG);
    EXPECT(gemm_f32(0, 2, 2, NULL, 2, NULL, 2, NULL, 2, NULL) == GEMM_F32_OK);
    EXPECT(gemm_f32_ex(2, 2, 2, a, 2, b, 2, c, 2, NULL, 99) == GEMM_F32_ERR_INVALID_ARG);
    EXPECT(gemm_f32_batched(GEMM_F32_OP_N, 7, 2, 2, 2, a, 2, 0, b, 2, 0, c, 2, 0, 1, NULL)
           == GEMM_F32_ERR_INVALID_ARG);
    EXPECT(gemm_f32_bias_act(2, 2, 2, a, 2, b, 2, NULL, 5, c, 2, NULL, 0, NULL)
           == GEMM_F32_ERR_INVALID_ARG);
    EXPECT(gemm_f32_mixed16(7, 2, 2, 2, a, 8, b, 8, c, 2, NULL) == GEMM_F32_ERR_INVALID_ARG);
    EXPECT(gemm_f32_round16(GEMM_F32_MIXED_BF16, 2, 4, a, 2, b, 4, NULL)
           == GEMM_F32_ERR_INVALID_ARG);
    EXPECT(gemm_f32_mixed_workspace_size(-1, 1, 1) < 0);
    EXPECT(gemm_f32_host(2, 2, 2, a, 1, b, 2, c, 2, NULL, NULL, NULL, NULL, 0, NULL)
           == GEMM_F32_ERR_INVALID_ARG);
    printf("%s\n", fails ? "C caller: failures" : "C caller: ok");
    return fails != 0;
}
"""


def test_plain_c_caller(built_lib, tmp_path):
    """The header compiles as C99 and a C program linked against the
    library gets the documented status codes."""
    src = tmp_path / "caller.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(built_lib)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o",
                    str(exe), "-L", libdir, "-l:" + os.path.basename(built_lib),
                    "-Wl,-rpath," + libdir], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "C caller: ok" in out.stdout
