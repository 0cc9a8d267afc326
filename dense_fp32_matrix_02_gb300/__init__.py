"""GB300-native single-precision matrix multiply, C = A·B, row-major.

The computation runs in hand-written CUDA kernels for sm_103a, built into
``libgemm_f32.so`` and reached through its C ABI (``include/gemm_f32.h``).
This package is the thin Python binding over that ABI (``gemm``) plus the
seeded input generator (``synth``).  Importing it does not load the shared
library; the first call does, and it raises if the library is missing.
"""

from .gemm import (ALGO_AUTO, ALGO_SIMT, ALGO_TMA, ALGO_TF32X3, GemmError,
                   gemm_f32, gemm_f32_ex, gemm_f32_ptr, library_path, lib)

__all__ = ["ALGO_AUTO", "ALGO_SIMT", "ALGO_TMA", "ALGO_TF32X3", "GemmError",
           "gemm_f32", "gemm_f32_ex", "gemm_f32_ptr", "library_path", "lib"]
