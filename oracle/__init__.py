"""Float64 CPU oracle for C = A·B (row-major float32 operands).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only users.  The product path
(``dense_fp32_matrix_02_gb300``) never imports this package, and this package
never imports the product: the two share nothing but the seeded input
generator, which holds none of the multiply's arithmetic.

The arithmetic lives in ``gemm_ref.c`` (plain C, float64 accumulation,
ascending k, no fused multiply-add); this module compiles it with gcc and
calls it through ctypes.  Source of the definition: "3 · La mémoire
partagée", §3.1 (C[lig][col] = sum over k of A[lig][k]·B[k][col], 2N³
operations) and "共享内存与同步", section "SharedArray —— 静态共享内存"
(the general m, n, k row-major indexing of tiled_sgemm).

Every function here is pinned by ``tests/test_oracle.py`` against things the
pages and the mathematics fix (identities, exact integer products, exact
rational brute force, a naive float32 loop, the 2MNK operation count and
metamorphic relations; for the epilogue, tabulated values of the normal
distribution function and the identity GELU(x) - GELU(-x) = x; for the
16-bit operand rounding, hand-worked ties and boundaries of both formats and
the conversions of torch and numpy); no function here is "parity unpinned".

The mixed-precision product ("Rendre le GPU rapide", "Les Tensor Cores")
rounds only the operands to 16 bits: ``gemm_mixed`` is ``gemm`` on the
rounded-and-widened operands.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "gemm_ref.c")
CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
          "-fopenmp", "-std=c11"]

_lock = threading.Lock()
_libs: dict = {}


def library_path(mutant: int = 0, outdir: str | None = None) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so"
    return os.path.join(outdir or _HERE, name)


def build(mutant: int = 0, outdir: str | None = None, force: bool = False) -> str:
    """Compile gemm_ref.c into a shared library; returns its path.

    ``mutant`` > 0 builds a copy with one planted mistake (see the C file);
    tests use those to show that the pins catch such mistakes.
    """
    out = library_path(mutant, outdir)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(SOURCE)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, f"-DORACLE_MUTANT={int(mutant)}", SOURCE, "-o", tmp,
           "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, dp, fp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
        lib.oracle_gemm_f64.restype = i64
        lib.oracle_gemm_f64.argtypes = [i64, i64, i64, fp, i64, fp, i64, dp,
                                        i64, dp, ctypes.c_int]
        lib.oracle_gemm_f64_entries.restype = i64
        lib.oracle_gemm_f64_entries.argtypes = [i64, i64, i64, fp, i64, fp,
                                                i64, i64, dp, dp, dp, dp]
        lib.oracle_epilogue_f64.restype = ctypes.c_int
        lib.oracle_epilogue_f64.argtypes = [i64, i64, dp, i64, fp, ctypes.c_int,
                                            dp, i64]
        lib.oracle_round_half.restype = ctypes.c_int
        lib.oracle_round_half.argtypes = [ctypes.c_int, i64, i64, fp, i64, dp,
                                          i64]
        lib.oracle_widen_half.restype = ctypes.c_int
        lib.oracle_widen_half.argtypes = [ctypes.c_int, i64, fp, dp]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        self._lib = lib
        self.path = path

    @staticmethod
    def _as_f32(x, name):
        x = np.asarray(x)
        if x.dtype != np.float32 or x.ndim != 2:
            raise TypeError(f"{name} must be a 2-D float32 array")
        if x.size == 0 or x.shape[1] == 1:
            return np.ascontiguousarray(x)
        if x.strides[1] != 4 or x.strides[0] % 4 or x.strides[0] < 0:
            raise ValueError(f"{name} must be row-major with unit column stride")
        return x

    def gemm(self, a, b, threads: int = 0, with_bound: bool = True):
        """(C_ref, bound, fmas) as float64 arrays for row-major float32 a, b."""
        a = self._as_f32(a, "a")
        b = self._as_f32(b, "b")
        M, K = a.shape
        K2, N = b.shape
        if K != K2:
            raise ValueError(f"inner sizes differ: {a.shape} x {b.shape}")
        lda = a.strides[0] // 4 if M > 1 else max(K, 1)
        ldb = b.strides[0] // 4 if K > 1 else max(N, 1)
        c = np.zeros((M, N), dtype=np.float64)
        bound = np.zeros((M, N), dtype=np.float64) if with_bound else None
        fmas = self._lib.oracle_gemm_f64(
            M, N, K, a.ctypes.data, max(lda, K), b.ctypes.data, max(ldb, N),
            c.ctypes.data, max(N, 1),
            bound.ctypes.data if with_bound else None, int(threads))
        if fmas < 0:
            raise ValueError("oracle rejected its arguments")
        return c, bound, fmas

    def entries(self, a, b, rows, cols):
        """C_ref and bound at the (rows[t], cols[t]) positions only."""
        a = self._as_f32(a, "a")
        b = self._as_f32(b, "b")
        M, K = a.shape
        _, N = b.shape
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        out = np.zeros(rows.shape[0], dtype=np.float64)
        bound = np.zeros(rows.shape[0], dtype=np.float64)
        lda = a.strides[0] // 4 if M > 1 else max(K, 1)
        ldb = b.strides[0] // 4 if K > 1 else max(N, 1)
        fmas = self._lib.oracle_gemm_f64_entries(
            M, N, K, a.ctypes.data, max(lda, K), b.ctypes.data, max(ldb, N),
            rows.shape[0], rows.ctypes.data, cols.ctypes.data, out.ctypes.data,
            bound.ctypes.data)
        if fmas < 0:
            raise ValueError("oracle rejected its arguments")
        return out, bound, fmas

    def epilogue(self, c, bias=None, act=0):
        """act(c + bias) in float64 for an oracle product c (M×N)."""
        c = np.ascontiguousarray(c, dtype=np.float64)
        M, N = c.shape
        out = np.empty_like(c)
        b = None
        if bias is not None:
            b = np.ascontiguousarray(bias, dtype=np.float32)
            if b.shape != (N,):
                raise ValueError("bias must have N elements")
        st = self._lib.oracle_epilogue_f64(
            M, N, c.ctypes.data, max(N, 1),
            b.ctypes.data if b is not None else None, int(act),
            out.ctypes.data, max(N, 1))
        if st != 0:
            raise ValueError("oracle rejected its arguments")
        return out

    def round_half(self, x, half_type: int):
        """The 16-bit patterns (uint16) of float32 x rounded to bfloat16
        (half_type 0) or IEEE binary16 (1), nearest with ties to even."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        flat = x.reshape(1, -1) if x.ndim != 2 else x
        out = np.empty(flat.shape, dtype=np.uint16)
        rows, cols = flat.shape
        st = self._lib.oracle_round_half(int(half_type), rows, cols,
                                         flat.ctypes.data, max(cols, 1),
                                         out.ctypes.data, max(cols, 1))
        if st != 0:
            raise ValueError("oracle rejected its arguments")
        return out.reshape(x.shape)

    def widen_half(self, h, half_type: int):
        """float32 values of 16-bit patterns h (exact)."""
        h = np.ascontiguousarray(h, dtype=np.uint16)
        out = np.empty(h.shape, dtype=np.float32)
        st = self._lib.oracle_widen_half(int(half_type), h.size, h.ctypes.data,
                                         out.ctypes.data)
        if st != 0:
            raise ValueError("oracle rejected its arguments")
        return out

    def gemm_mixed(self, a, b, half_type: int, threads: int = 0):
        """(C_ref, bound, fmas) of the mixed-precision product: a and b
        rounded to 16 bits, then the float64 product of the rounded values."""
        ar = self.widen_half(self.round_half(a, half_type), half_type)
        br = self.widen_half(self.round_half(b, half_type), half_type)
        return self.gemm(ar, br, threads)

    def max_threads(self) -> int:
        return int(self._lib.oracle_max_threads())


def load(mutant: int = 0, outdir: str | None = None) -> Oracle:
    """The oracle (mutant 0), compiled on first use."""
    key = (mutant, outdir)
    with _lock:
        if key not in _libs:
            _libs[key] = Oracle(build(mutant, outdir))
        return _libs[key]


def gemm(a, b, threads: int = 0, with_bound: bool = True):
    return load().gemm(a, b, threads, with_bound)


def entries(a, b, rows, cols):
    return load().entries(a, b, rows, cols)


def epilogue(c, bias=None, act=0):
    return load().epilogue(c, bias, act)


def round_half(x, half_type: int):
    return load().round_half(x, half_type)


def widen_half(h, half_type: int):
    return load().widen_half(h, half_type)


def gemm_mixed(a, b, half_type: int, threads: int = 0):
    return load().gemm_mixed(a, b, half_type, threads)


def tolerance(bound, K: int):
    """Per-element acceptance: 1e-5 * sqrt(K) * (|A|·|B|)_ij + 1e-30."""
    return 1e-5 * np.sqrt(max(K, 0)) * bound + 1e-30


if __name__ == "__main__":  # pragma: no cover - manual build helper
    print(build(force="--force" in sys.argv))
