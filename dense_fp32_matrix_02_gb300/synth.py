"""Seeded synthetic operands for the FP32 GEMM C = A·B.

This module only draws numbers. It holds none of the multiply's arithmetic,
so the CUDA path and the float64 oracle can both take their inputs from it
without sharing any of the computation they are checked on.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), written here from its published
definition: the state advances by the golden-ratio increment and each output
is the state passed through the variant-13 mixing function (shifts 30, 27, 31
and the two odd multipliers below).  Output number ``i`` (0-based) of the
stream for ``seed`` is ``mix(seed + (i + 1) * GOLDEN)``, so any slice of the
stream can be produced without running through the ones before it.

A stream feeds one (A, B) pair: A's elements first, in row-major order, then
B's, also row-major.  Each element takes one draw (uniform, small integers) or
two (normal, Box-Muller).

Distributions (each maps draws to float32 exactly as written):

* ``uniform``  in [-1, 1): ``u = (x >> 40) * 2**-24``, value ``2u - 1``, which
  float32 represents exactly (a multiple of 2**-23 in [-1, 1)).
* ``normal``   N(0, sigma^2): Box-Muller in float64 on the draws x1, x2:
  ``u1 = ((x1 >> 11) + 1) * 2**-53`` in (0, 1], ``u2 = (x2 >> 11) * 2**-53``,
  ``z = sqrt(-2 ln u1) * cos(2 pi u2)``, value ``float32(sigma * z)``.
* ``int``      small integers in {-2, ..., 2}: ``((x >> 32) * 5) >> 32`` minus
  2, computed in unsigned 64-bit integers.  Float32 holds these exactly, and
  any sum of at most 2**22 products of them stays an exact float32 integer.
* ``int8``     integers in {-8, ..., 8}: ``((x >> 32) * 17) >> 32`` minus 8,
  the inputs of the mixed-precision exactness test ("Rendre le GPU rapide",
  "Les Tensor Cores"): exact in bfloat16 and binary16, and sums of at most
  2**18 products of them stay exact float32 integers.

The workloads (sizes, distributions and seeds) are the five dense FP32 GEMM
cases of this library's test and benchmark plan; ``WORKLOADS`` lists them.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
MUL1 = np.uint64(0xBF58476D1CE4E5B9)
MUL2 = np.uint64(0x94D049BB133111EB)

_CHUNK = 1 << 22  # draws per vectorised block, bounds temporary memory


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of the SplitMix64 stream for ``seed``."""
    out = np.empty(count, dtype=np.uint64)
    s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        for lo in range(0, count, _CHUNK):
            hi = min(count, lo + _CHUNK)
            idx = np.arange(start + lo + 1, start + hi + 1, dtype=np.uint64)
            z = s + idx * GOLDEN
            z = (z ^ (z >> np.uint64(30))) * MUL1
            z = (z ^ (z >> np.uint64(27))) * MUL2
            out[lo:hi] = z ^ (z >> np.uint64(31))
    return out


def _draws_per_element(dist: str) -> int:
    if dist == "normal":
        return 2
    if dist in ("uniform", "int", "int8"):
        return 1
    raise ValueError(f"unknown distribution {dist!r}")


def _fill(seed: int, start: int, n: int, dist: str, sigma: float) -> np.ndarray:
    if dist == "uniform":
        x = splitmix64(seed, start, n)
        u = (x >> np.uint64(40)).astype(np.float64) * 2.0**-24
        return (2.0 * u - 1.0).astype(np.float32)
    if dist == "int":
        x = splitmix64(seed, start, n)
        with np.errstate(over="ignore"):
            v = ((x >> np.uint64(32)) * np.uint64(5)) >> np.uint64(32)
        return (v.astype(np.int64) - 2).astype(np.float32)
    if dist == "int8":
        x = splitmix64(seed, start, n)
        with np.errstate(over="ignore"):
            v = ((x >> np.uint64(32)) * np.uint64(17)) >> np.uint64(32)
        return (v.astype(np.int64) - 8).astype(np.float32)
    if dist == "normal":
        x = splitmix64(seed, start, 2 * n)
        x1 = x[0::2]
        x2 = x[1::2]
        u1 = ((x1 >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0**-53
        u2 = (x2 >> np.uint64(11)).astype(np.float64) * 2.0**-53
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        return (sigma * z).astype(np.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def make_operands(M: int, N: int, K: int, seed: int, dist_a: str = "uniform",
                  dist_b: Optional[str] = None, sigma_a: float = 1.0,
                  sigma_b: float = 1.0):
    """Row-major float32 A (M×K) and B (K×N) drawn from one seeded stream."""
    dist_b = dist_a if dist_b is None else dist_b
    na, nb = M * K, K * N
    a = _fill(seed, 0, na, dist_a, sigma_a).reshape(M, K)
    b = _fill(seed, na * _draws_per_element(dist_a), nb, dist_b,
              sigma_b).reshape(K, N)
    return a, b


@dataclasses.dataclass(frozen=True)
class Workload:
    """One GEMM case: sizes, the seed and the operand distributions."""
    name: str
    M: int
    N: int
    K: int
    seed: int
    dist_a: str = "uniform"
    dist_b: str = "uniform"
    sigma_a: float = 1.0
    sigma_b: float = 1.0

    def operands(self):
        return make_operands(self.M, self.N, self.K, self.seed, self.dist_a,
                             self.dist_b, self.sigma_a, self.sigma_b)

    def integer_variant(self) -> "Workload":
        """Same sizes and seed, entries in {-2..2} (exact in float32)."""
        return dataclasses.replace(self, name=self.name + "_int",
                                   dist_a="int", dist_b="int")

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def bytes(self) -> int:
        return 4 * (self.M * self.K + self.K * self.N + self.M * self.N)


WORKLOADS = {
    # 64^3, uniform [-1, 1), seed 0 (also run with small integers)
    "sq64": Workload("sq64", 64, 64, 64, 0),
    # 1024^3, N(0, 1), seed 1
    "sq1024": Workload("sq1024", 1024, 1024, 1024, 1, "normal", "normal"),
    # 4096^3, uniform [-1, 1), seed 2: the headline size
    "sq4096": Workload("sq4096", 4096, 4096, 4096, 2),
    # transformer MLP up-projection: 8192 tokens x 768 -> 3072,
    # activations N(0, 1), weights N(0, 0.02^2), seed 3
    "mlp": Workload("mlp", 8192, 3072, 768, 3, "normal", "normal", 1.0, 0.02),
    # ragged 1000^3, uniform, seed 4 (edge tiles in M, N and K)
    "rag1000": Workload("rag1000", 1000, 1000, 1000, 4),
    # skinny 65536 x 64 x 64, uniform, seed 4 (near the memory roof)
    "skinny": Workload("skinny", 65536, 64, 64, 4),
}
