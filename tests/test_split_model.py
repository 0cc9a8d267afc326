"""The 3xTF32 split's error bound, on the CPU, from the definitions alone.

The tensor path reads each fp32 operand x as TF32 by truncation (the 13 low
mantissa bits dropped), computes small = x - trunc(x) exactly in fp32, and
forms a·b ≈ a_big·b_big + a_big·b_small + a_small·b_big, where the tensor
core again truncates the small parts it reads.  Every term it drops is at
most 2^-20·|a·b|, so the product is within 3·2^-20·|a·b| of the exact one
before the fp32 accumulation rounds it.  This model checks that bound on
random and extreme fp32 pairs (products evaluated exactly in float64); it
shares nothing with the GPU code and stands beside its parity tests."""

from __future__ import annotations

import numpy as np


def trunc_tf32(x: np.ndarray) -> np.ndarray:
    """fp32 -> TF32 by dropping the 13 low mantissa bits (sign, exponent
    and 10 mantissa bits kept)."""
    bits = np.asarray(x, np.float32).view(np.uint32)
    return (bits & np.uint32(0xFFFFE000)).view(np.float32)


def split_product(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """The three-term product as the tensor path forms it, each term exact
    in float64 (11-bit by 11-bit significands)."""
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    ab, bb = trunc_tf32(a), trunc_tf32(b)
    a_s = (a - ab).astype(np.float32)    # exact in fp32
    b_s = (b - bb).astype(np.float32)
    a_s, b_s = trunc_tf32(a_s), trunc_tf32(b_s)   # read as TF32 again
    f = np.float64
    return (ab.astype(f) * bb.astype(f) + ab.astype(f) * b_s.astype(f)
            + a_s.astype(f) * bb.astype(f))


def _samples(n, rng):
    u = rng.uniform(-1.0, 1.0, n).astype(np.float32)
    g = rng.standard_normal(n).astype(np.float32)
    wide = (rng.uniform(1, 2, n) * 2.0 ** rng.integers(-60, 60, n)
            * rng.choice([-1, 1], n)).astype(np.float32)
    raw = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
    raw = raw.view(np.float32)
    raw = raw[np.isfinite(raw) & (np.abs(raw) < 1e18) & (np.abs(raw) > 1e-18)]
    return np.concatenate([u, g, wide, raw])


def test_small_part_is_exact_in_fp32():
    rng = np.random.default_rng(0)
    x = _samples(100000, rng)
    big = trunc_tf32(x)
    small = (x - big).astype(np.float32)
    assert np.array_equal(big.astype(np.float64) + small.astype(np.float64),
                          x.astype(np.float64))
    # the truncation error is below one TF32 ulp of x
    assert np.all(np.abs(small.astype(np.float64))
                  <= 2.0 ** -10 * np.abs(x.astype(np.float64)))


def test_three_term_product_within_3_ulp20():
    rng = np.random.default_rng(1)
    a = _samples(200000, rng)
    b = rng.permutation(_samples(200000, rng))[: a.size]
    a = a[: b.size]
    exact = a.astype(np.float64) * b.astype(np.float64)
    err = np.abs(split_product(a, b) - exact)
    assert np.all(err <= 3 * 2.0 ** -20 * np.abs(exact))


def test_bound_is_reached_within_a_factor():
    """The bound is not loose by orders of magnitude: operands whose
    truncated bits are all ones come close to it."""
    a = np.array([np.uint32(0x3FFFFFFF)], np.uint32).view(np.float32)
    exact = a.astype(np.float64) ** 2
    err = np.abs(split_product(a, a) - exact)
    assert err[0] > 0.25 * 2.0 ** -20 * exact[0]
    assert err[0] <= 3 * 2.0 ** -20 * exact[0]


def test_integers_of_eleven_bits_are_exact():
    """Small integers split with small == 0: the product is exact, which is
    why the GPU's integer cases are bit-exact."""
    v = np.arange(-2048, 2049, dtype=np.float32)
    a, b = np.meshgrid(v[::37], v[::41])
    assert np.array_equal(split_product(a, b),
                          a.astype(np.float64) * b.astype(np.float64))
