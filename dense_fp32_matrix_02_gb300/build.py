"""Builds libgemm_f32.so in-tree with nvcc for sm_103a.

Each CUDA translation unit compiles in parallel to an object file under
``_build/``; the objects link into ``libgemm_f32.so`` next to this file.
``python -m dense_fp32_matrix_02_gb300.build [--verbose-ptxas] [--checked]``.

``--checked`` (``build(checked=True)``) builds ``libgemm_f32_debug.so``
instead, with GEMM_F32_BOUNDS_CHECK=1: the FFMA and tensor kernels then test
every shared-memory, tensor-memory and global index against its extent and
report a failure through the kernel status word, skipping the access.
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
OUTPUT = os.path.join(HERE, "libgemm_f32.so")
OUTPUT_CHECKED = os.path.join(HERE, "libgemm_f32_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]


def _compile(src: str, ptxas_verbose: bool, checked: bool = False) -> str:
    bdir = os.path.join(BUILD_DIR, "checked") if checked else BUILD_DIR
    obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
    if checked:
        cmd.append("-DGEMM_F32_BOUNDS_CHECK=1")
    if ptxas_verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if ptxas_verbose:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, ptxas_verbose: bool = False,
          checked: bool = False) -> str:
    """Compiles the library (the checked one with `checked`) if any source
    is newer than it; returns its path."""
    output = OUTPUT_CHECKED if checked else OUTPUT
    if (not force and not ptxas_verbose and os.path.exists(output)
            and os.path.getmtime(output) >= max(os.path.getmtime(p)
                                                 for p in _deps())):
        return output
    os.makedirs(os.path.join(BUILD_DIR, "checked") if checked else BUILD_DIR,
                exist_ok=True)
    srcs = sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, ptxas_verbose, checked),
                           srcs))
    tmp = output + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, output)
    return output


if __name__ == "__main__":
    print(build(force=True, ptxas_verbose="--verbose-ptxas" in sys.argv,
                checked="--checked" in sys.argv))
