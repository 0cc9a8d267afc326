"""Pins for the float64 oracle, against facts that do not come from it.

Each pin checks the oracle against something the pages or mathematics fix:
hand-worked products (tests/golden), closed forms (identity, all-ones,
index products, permutations), exact integer arithmetic, exact rational
brute force, a naive float32 loop inside its rounding-error bound, the
pages' operation count 2MNK ("3 · La mémoire partagée", §3.1) and
metamorphic relations.  ``test_mutant_is_caught`` builds oracle copies with
one planted mistake each (dropped term, transposed operand, wrong sign,
wrong row, float32 accumulation; truncating bfloat16 rounding, binary16
ties away from zero, binary16 without subnormals) and checks that some pin
fails on each.
"""

from __future__ import annotations

import fractions
import itertools

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_02_gb300 import synth
from helpers import load_golden_cases

U64 = 2.0**-53  # float64 unit roundoff
U32 = 2.0**-24  # float32 unit roundoff


def _gamma(n, u):
    return n * u / (1.0 - n * u)


# --------------------------------------------------------------------- pins
def pin_golden(orc):
    """Hand-worked products: exact, bit for bit."""
    for name, m in load_golden_cases():
        c, _, _ = orc.gemm(m["A"], m["B"])
        assert np.array_equal(c, m["C"]), f"golden case {name}: {c} != {m['C']}"


def pin_identity(orc):
    """A·I = A and I·B = B exactly (one non-zero term per sum)."""
    a, b = synth.make_operands(37, 29, 23, seed=11)
    c, _, _ = orc.gemm(a, np.eye(23, dtype=np.float32))
    assert np.array_equal(c, a.astype(np.float64)), "A·I != A"
    c, _, _ = orc.gemm(np.eye(23, dtype=np.float32), b)
    assert np.array_equal(c, b.astype(np.float64)), "I·B != B"


def pin_all_ones(orc):
    """All-ones A (M×K) and B (K×N) give C = K everywhere."""
    for (M, N, K) in [(5, 7, 1), (9, 4, 13), (16, 16, 64)]:
        c, bound, _ = orc.gemm(np.ones((M, K), np.float32),
                               np.ones((K, N), np.float32))
        assert np.array_equal(c, np.full((M, N), float(K))), "ones·ones != K"
        assert np.array_equal(bound, np.full((M, N), float(K)))


def pin_index_product(orc):
    """A[i][k] = i, B[k][j] = j gives C[i][j] = K·i·j exactly."""
    M, N, K = 12, 10, 9
    a = np.repeat(np.arange(M, dtype=np.float32)[:, None], K, axis=1)
    b = np.repeat(np.arange(N, dtype=np.float32)[None, :], K, axis=0)
    c, _, _ = orc.gemm(a, b)
    want = K * np.outer(np.arange(M), np.arange(N)).astype(np.float64)
    assert np.array_equal(c, want), "index product wrong"


def pin_permutation(orc):
    """P·B permutes B's rows and B·P permutes its columns, exactly."""
    rng = np.random.default_rng(5)
    _, b = synth.make_operands(1, 11, 11, seed=12)
    perm = rng.permutation(11)
    p = np.eye(11, dtype=np.float32)[perm]  # row i of P is e_{perm[i]}
    c, _, _ = orc.gemm(p, b)
    assert np.array_equal(c, b[perm].astype(np.float64)), "P·B wrong"
    c, _, _ = orc.gemm(b, p)
    inv = np.argsort(perm)
    assert np.array_equal(c, b[:, inv].astype(np.float64)), "B·P wrong"


def pin_integer_exact(orc):
    """Small-integer inputs: equal to exact int64 arithmetic."""
    for (M, N, K, seed) in [(17, 23, 31, 0), (64, 64, 64, 0), (3, 130, 257, 4)]:
        a, b = synth.make_operands(M, N, K, seed, "int", "int")
        c, _, _ = orc.gemm(a, b)
        exact = a.astype(np.int64) @ b.astype(np.int64)
        assert np.array_equal(c, exact.astype(np.float64)), "integer product"


def pin_exact_rational(orc):
    """Brute force in exact rationals: within the float64 summation bound.

    The product of two float32 values is exact in float64, so the oracle's
    only rounding is in its K-1 additions: |C_ref - C| <= gamma_{K-1}·sum|ab|.
    Includes a case (1 + 2**-30) that a float32 accumulator gets wrong.
    """
    cases = [synth.make_operands(M, N, K, seed=21 + M)
             for (M, N, K) in [(1, 1, 1), (2, 3, 5), (4, 4, 7), (3, 5, 16)]]
    cases.append((np.array([[1.0, 2.0**-30, -3.0]], np.float32),
                  np.array([[1.0], [1.0], [2.0**-40]], np.float32)))
    for a, b in cases:
        c, bound, _ = orc.gemm(a, b)
        M, K = a.shape
        N = b.shape[1]
        for i, j in itertools.product(range(M), range(N)):
            exact = sum(fractions.Fraction(float(a[i, k])) *
                        fractions.Fraction(float(b[k, j])) for k in range(K))
            err = abs(fractions.Fraction(c[i, j]) - exact)
            mag = sum(abs(fractions.Fraction(float(a[i, k])) *
                          fractions.Fraction(float(b[k, j]))) for k in range(K))
            assert err <= fractions.Fraction(_gamma(max(K - 1, 0), U64)) * mag, \
                f"rational check at {(i, j)}: {c[i, j]!r} vs {float(exact)!r}"
            assert bound[i, j] == float(mag) or abs(
                fractions.Fraction(bound[i, j]) - mag) <= \
                fractions.Fraction(_gamma(K, U64)) * mag, "bound wrong"


def pin_naive_float32(orc):
    """A naive float32 loop (k ascending) agrees within its error bound.

    For every M, N, K in 1..16: |C32 - C_ref| <= gamma_K(2**-24)·sum|ab|
    plus the oracle's own float64 bound.
    """
    for M, N, K in itertools.product(range(1, 17), repeat=3):
        if (M * 7 + N * 3 + K) % 5:  # every fifth shape keeps this quick
            continue
        a, b = synth.make_operands(M, N, K, seed=1000 + M * 289 + N * 17 + K)
        c32 = np.zeros((M, N), np.float32)
        for k in range(K):
            c32 = (c32 + (a[:, k:k + 1] * b[k:k + 1, :]).astype(np.float32)
                   ).astype(np.float32)
        c, bound, _ = orc.gemm(a, b)
        lim = (_gamma(K, U32) + _gamma(K, U64)) * bound
        assert (np.abs(c32.astype(np.float64) - c) <= lim).all(), \
            f"naive float32 loop disagrees at M,N,K={M},{N},{K}"


def pin_operation_count(orc):
    """2·(multiply-adds) = 2MNK, the pages' 2N³ for square N×N."""
    for (M, N, K) in [(64, 64, 64), (3, 5, 7), (10, 1, 33)]:
        a, b = synth.make_operands(M, N, K, seed=3)
        _, _, fmas = orc.gemm(a, b)
        assert 2 * fmas == 2 * M * N * K, f"op count {2 * fmas}"
    _, _, fmas = orc.gemm(*synth.make_operands(64, 64, 64, seed=0))
    assert 2 * fmas == 2 * 64**3


def pin_metamorphic(orc):
    """(AB)ᵀ = BᵀAᵀ bitwise; K-split additivity (exact on integers);
    scaling A by 2 scales C by 2 exactly; entries() equals gemm()."""
    a, b = synth.make_operands(19, 13, 21, seed=7)
    c, bound, _ = orc.gemm(a, b)
    ct, _, _ = orc.gemm(np.ascontiguousarray(b.T), np.ascontiguousarray(a.T))
    assert np.array_equal(c.T, ct), "(AB)^T != B^T A^T"
    c2, _, _ = orc.gemm(2 * a, b)
    assert np.array_equal(c2, 2 * c), "C(2A) != 2 C(A)"
    ai, bi = synth.make_operands(19, 13, 21, seed=7, dist_a="int", dist_b="int")
    ci, _, _ = orc.gemm(ai, bi)
    k1 = 8
    p1, _, _ = orc.gemm(np.ascontiguousarray(ai[:, :k1]), bi[:k1])
    p2, _, _ = orc.gemm(np.ascontiguousarray(ai[:, k1:]), bi[k1:])
    assert np.array_equal(ci, p1 + p2), "K-split additivity"
    rows = np.array([0, 5, 18, 7])
    cols = np.array([0, 12, 3, 7])
    e, eb, fm = orc.entries(a, b, rows, cols)
    assert np.array_equal(e, c[rows, cols]) and np.array_equal(
        eb, bound[rows, cols]) and fm == 4 * 21


def pin_bound(orc):
    """bound = oracle(|A|, |B|) and |C| <= bound."""
    a, b = synth.make_operands(9, 11, 40, seed=9, dist_a="normal",
                               dist_b="normal")
    c, bound, _ = orc.gemm(a, b)
    m, _, _ = orc.gemm(np.abs(a), np.abs(b))
    assert np.array_equal(m, bound)
    assert (np.abs(c) <= bound).all()


def pin_empty(orc):
    """K = 0 is the empty sum (zeros); M = 0 or N = 0 is an empty C."""
    c, bound, f = orc.gemm(np.zeros((4, 0), np.float32),
                           np.zeros((0, 5), np.float32))
    assert c.shape == (4, 5) and not c.any() and not bound.any() and f == 0
    c, _, _ = orc.gemm(np.zeros((0, 3), np.float32), np.ones((3, 5), np.float32))
    assert c.shape == (0, 5)
    c, _, _ = orc.gemm(np.ones((4, 3), np.float32), np.zeros((3, 0), np.float32))
    assert c.shape == (4, 0)


PINS = [pin_golden, pin_identity, pin_all_ones, pin_index_product,
        pin_permutation, pin_integer_exact, pin_exact_rational,
        pin_naive_float32, pin_operation_count, pin_metamorphic, pin_bound,
        pin_empty]


# ------------------------------------------------ 16-bit operand rounding
# Hand-worked values of both formats ("Rendre le GPU rapide", "Les Tensor
# Cores": operands rounded to nearest, ties to even).  bfloat16 keeps 7
# stored bits (quantum 2^-7 in [1, 2)); binary16 keeps 10 (quantum 2^-10 in
# [1, 2), 2^-24 below 2^-14) and overflows past 65504.
HALF_WORKED = [
    # (value, bfloat16 bits, binary16 bits)
    (1.0, 0x3F80, 0x3C00),
    (1 + 2**-8, 0x3F80, 0x3C04),           # bf16: halfway, even is 1.0
    (1 + 3 * 2**-8, 0x3F82, 0x3C0C),       # bf16: halfway, even is 1+2^-6
    (1 + 2**-8 + 2**-20, 0x3F81, 0x3C04),  # bf16: just above halfway
    (-(1 + 2**-7 + 2**-9), 0xBF81, 0xBC0A),
    (1 + 2**-11, 0x3F80, 0x3C00),          # f16: halfway, even is 1.0
    (1 + 3 * 2**-11, 0x3F80, 0x3C02),      # f16: halfway, even is 1+2^-9
    (65504.0, 0x4780, 0x7BFF),             # largest binary16
    (65519.0, 0x4780, 0x7BFF),
    (65520.0, 0x4780, 0x7C00),             # halfway to 2^16: ties to Inf
    (2.0**-14, 0x3880, 0x0400),            # smallest normal binary16
    (2.0**-24, 0x3380, 0x0001),            # smallest subnormal binary16
    (2.0**-25, 0x3300, 0x0000),            # halfway 0 .. 2^-24: even is 0
    (3 * 2.0**-25, 0x33C0, 0x0002),        # halfway 1 .. 2 quanta: even 2
    (2.0**-14 - 2.0**-25, 0x3880, 0x0400), # rounds up into the normals
    (3.0e38, 0x7F62, 0x7C00),
    (3.4028234663852886e38, 0x7F80, 0x7C00),  # FLT_MAX: bf16 overflows
    (-0.0, 0x8000, 0x8000),
    (float("inf"), 0x7F80, 0x7C00),
    (float("-inf"), 0xFF80, 0xFC00),
]


def pin_half_worked_values(orc):
    x = np.array([v for v, _, _ in HALF_WORKED], np.float32)
    assert orc.round_half(x, 0).tolist() == [b for _, b, _ in HALF_WORKED]
    assert orc.round_half(x, 1).tolist() == [h for _, _, h in HALF_WORKED]


def _float32_sample(n, seed):
    """Finite float32 values over every exponent, plus exact ties of both
    formats (low 16 bits 0x8000 for bfloat16; for binary16 values whose
    bits below the kept ones are exactly one half)."""
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
    bits = bits[(bits & 0x7F800000) != 0x7F800000]
    ties_bf = (bits & 0xFFFF0000) | 0x8000
    ties_f16 = (bits & 0xFFFFE000) | 0x1000
    # binary16 range: exponents -30 .. 16 with ties at the 13th bit
    e = rng.integers(-30, 17, n // 4)
    m = rng.integers(0, 2**23, n // 4)
    small = np.ldexp(1 + m / 2.0**23, e).astype(np.float32)
    return np.concatenate([bits.view(np.float32), ties_bf.view(np.float32),
                           ties_f16.view(np.float32), small,
                           -small]).astype(np.float32)


def pin_bf16_matches_torch(orc):
    """bfloat16 rounding equals torch's float32 -> bfloat16 conversion
    (round to nearest even) on every exponent, on ties, and keeps NaN."""
    torch = pytest.importorskip("torch")
    x = _float32_sample(40000, 11)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(orc.round_half(x, 0), want.view(np.uint16))
    nan = orc.round_half(np.array([np.nan], np.float32), 0)
    assert (nan[0] & 0x7F80) == 0x7F80 and (nan[0] & 0x7F) != 0


def pin_f16_matches_numpy(orc):
    """binary16 rounding equals numpy's float32 -> float16 conversion
    (IEEE round to nearest even, gradual underflow, overflow to Inf)."""
    x = _float32_sample(40000, 12)
    with np.errstate(over="ignore"):  # overflow to Inf is the point
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(orc.round_half(x, 1), want)
    nan = orc.round_half(np.array([np.nan], np.float32), 1)
    assert (nan[0] & 0x7C00) == 0x7C00 and (nan[0] & 0x3FF) != 0


def pin_widen_exact(orc):
    """Widening gives every 16-bit pattern's value: binary16 as numpy
    decodes it, bfloat16 as torch does; rounding a widened value gives the
    pattern back (every representable value rounds to itself)."""
    torch = pytest.importorskip("torch")
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f16 = orc.widen_half(h, 1)
    with np.errstate(invalid="ignore"):   # the NaN patterns widen to NaN
        ref16 = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref16)
    assert np.array_equal(np.isnan(f16), nan)
    assert np.array_equal(f16[~nan].view(np.uint32), ref16[~nan].view(np.uint32))
    bf = orc.widen_half(h, 0)
    refbf = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    nanb = np.isnan(refbf)
    assert np.array_equal(np.isnan(bf), nanb)
    assert np.array_equal(bf[~nanb].view(np.uint32), refbf[~nanb].view(np.uint32))
    assert np.array_equal(orc.round_half(f16[~nan], 1), h[~nan])
    assert np.array_equal(orc.round_half(bf[~nanb], 0), h[~nanb])


def pin_mixed_small_integers(orc):
    """The pages' test of the mixed-precision product: integers in [-8, 8]
    are exact in 16 bits and their sums exact in float32, so the result is
    the exact integer product."""
    rng = np.random.default_rng(5)
    a = rng.integers(-8, 9, (7, 300)).astype(np.float32)
    b = rng.integers(-8, 9, (300, 5)).astype(np.float32)
    exact = a.astype(np.int64) @ b.astype(np.int64)
    for t in (0, 1):
        c, _, _ = orc.gemm_mixed(a, b, t)
        assert np.array_equal(c, exact.astype(np.float64))


def pin_mixed_rounds_operands_only(orc):
    """The mixed product is the exact product of the rounded operands: with
    B = I it returns A rounded (worked values above), not A."""
    x = np.array([[v for v, _, _ in HALF_WORKED[:8]]], np.float32)
    for t in (0, 1):
        c, _, _ = orc.gemm_mixed(x, np.eye(8, dtype=np.float32), t)
        want = [w[1 + t] for w in HALF_WORKED[:8]]
        got = orc.round_half(c.astype(np.float32), t)[0].tolist()
        assert got == want


HALF_PINS = [pin_half_worked_values, pin_bf16_matches_torch,
             pin_f16_matches_numpy, pin_widen_exact, pin_mixed_small_integers,
             pin_mixed_rounds_operands_only]


@pytest.mark.parametrize("pin", PINS + HALF_PINS,
                         ids=[p.__name__ for p in PINS + HALF_PINS])
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6, 7, 8])
def test_mutant_is_caught(mutant, tmp_path):
    """Each planted mistake makes at least one pin fail."""
    orc = oracle.Oracle(oracle.build(mutant, outdir=str(tmp_path)))
    failed = []
    for pin in PINS + HALF_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} passed every pin"


def test_threads_do_not_change_bits(oracle_lib):
    a, b = synth.make_operands(33, 45, 70, seed=2)
    c1, b1, _ = oracle_lib.gemm(a, b, threads=1)
    c4, b4, _ = oracle_lib.gemm(a, b, threads=4)
    assert np.array_equal(c1, c4) and np.array_equal(b1, b4)


def test_strided_operands(oracle_lib):
    """Leading dimensions larger than the row width are honoured."""
    a, b = synth.make_operands(6, 5, 7, seed=8)
    big_a = np.zeros((6, 11), np.float32)
    big_a[:, :7] = a
    big_b = np.zeros((7, 9), np.float32)
    big_b[:, :5] = b
    c, _, _ = oracle_lib.gemm(a, b)
    cs, _, _ = oracle_lib.gemm(big_a[:, :7], big_b[:, :5])
    assert np.array_equal(c, cs)


# ------------------------------------------------------------- epilogue
def test_epilogue_gelu_tabulated_values(oracle_lib):
    """GELU(x) = x·Φ(x) at points where Φ is tabulated: Φ(0) = 1/2,
    Φ(1) = 0.8413447460685429, Φ(-1) = 0.15865525393145707,
    Φ(2) = 0.9772498680518208; far tails give x and 0."""
    x = np.array([[0.0, 1.0, -1.0, 2.0, 10.0, -10.0]])
    got = oracle_lib.epilogue(x, act=1)[0]
    want = [0.0, 0.8413447460685429, -0.15865525393145707,
            2 * 0.9772498680518208, 10.0, 0.0]
    assert np.allclose(got, want, rtol=1e-15, atol=1e-20)


def test_epilogue_gelu_odd_part_identity(oracle_lib):
    """Φ(x) + Φ(-x) = 1, so GELU(x) - GELU(-x) = x for every x."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((7, 9)) * 3
    g = oracle_lib.epilogue(x, act=1)
    gm = oracle_lib.epilogue(-x, act=1)
    assert np.allclose(g - gm, x, rtol=1e-14, atol=1e-15)


def test_epilogue_bias_broadcast_and_identity(oracle_lib):
    c = np.arange(12, dtype=np.float64).reshape(3, 4)
    bias = np.array([0.5, -1.0, 2.0, 0.0], np.float32)
    out = oracle_lib.epilogue(c, bias, act=0)
    assert np.array_equal(out, c + bias.astype(np.float64))
    assert np.array_equal(oracle_lib.epilogue(c), c)
    with pytest.raises(ValueError):
        oracle_lib.epilogue(c, bias, act=2)
