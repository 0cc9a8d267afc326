"""The seeded input generator: published SplitMix64 values, ranges, layout."""

import numpy as np

from dense_fp32_matrix_02_gb300 import synth


def _splitmix_reference(seed, n):
    """SplitMix64 written out with Python integers, one draw at a time."""
    mask = (1 << 64) - 1
    state = seed & mask
    out = []
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & mask
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & mask
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & mask
        out.append(z ^ (z >> 31))
    return out


def test_splitmix64_published_values():
    # first three outputs for seed 0, as published with the generator
    got = [int(x) for x in synth.splitmix64(0, 0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_splitmix64_matches_scalar_form_and_offsets():
    for seed in (0, 1, 2**63 + 5):
        ref = _splitmix_reference(seed, 40)
        assert [int(x) for x in synth.splitmix64(seed, 0, 40)] == ref
        assert [int(x) for x in synth.splitmix64(seed, 17, 23)] == ref[17:]


def test_distributions_and_layout():
    a, b = synth.make_operands(50, 40, 30, seed=2)
    assert a.shape == (50, 30) and b.shape == (30, 40)
    assert a.dtype == np.float32 and a.flags.c_contiguous
    assert a.min() >= -1.0 and a.max() < 1.0
    # A first, then B, one draw each
    x = synth.splitmix64(2, 0, 50 * 30 + 30 * 40)
    u = (x >> np.uint64(40)).astype(np.float64) * 2.0**-24
    v = (2 * u - 1).astype(np.float32)
    assert np.array_equal(a.ravel(), v[:1500]) and np.array_equal(
        b.ravel(), v[1500:])
    ai, bi = synth.make_operands(64, 64, 64, 0, "int", "int")
    assert set(np.unique(ai)) <= {-2.0, -1.0, 0.0, 1.0, 2.0}
    a8, _ = synth.make_operands(64, 64, 64, 0, "int8", "int8")
    assert set(np.unique(a8)) == {float(v) for v in range(-8, 9)}
    assert abs(a8.mean()) < 0.2
    an, bn = synth.WORKLOADS["mlp"].operands()
    assert abs(an.std() - 1.0) < 0.01 and abs(bn.std() - 0.02) < 0.0002
    assert abs(an.mean()) < 0.01


def test_deterministic():
    a1, b1 = synth.WORKLOADS["rag1000"].operands()
    a2, b2 = synth.WORKLOADS["rag1000"].operands()
    assert np.array_equal(a1, a2) and np.array_equal(b1, b2)
