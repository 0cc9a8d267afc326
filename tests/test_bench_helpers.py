"""Host-side helpers of bench.py: the timing arithmetic and the input
rotation, checked on the CPU (the GPU parts run under -m gpu)."""

from __future__ import annotations

import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location(
        "bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_sample_stats_orders_chunks():
    b = _bench()
    st = b.sample_stats(2e12, [2.0, 1.0, 4.0, 2.0, 1.0])  # ms per step
    assert st["n"] == 5
    assert st["max"] == pytest.approx(2000.0)   # 2e12 flop in 1 ms
    assert st["min"] == pytest.approx(500.0)
    assert st["median"] == pytest.approx(1000.0)
    assert b.sample_stats(1.0, []) is None


def test_rotating_sets_exceed_twice_l2():
    b = _bench()
    l2 = 129 * 2**20
    for set_bytes in (48 * 1024, 12 * 2**20, 33.6e6, 135e6, 201e6):
        n = b.rotating_sets(set_bytes, l2)
        assert n >= 3
        assert n * set_bytes > 2 * l2 or n == 8192
    assert b.rotating_sets(201e6, l2) == 3


def test_weak_scaling_value_counts_every_rank():
    b = _bench()
    # 4 ranks, 10 steps of 1e12 flop each, slowest rank 20 ms
    assert b.weak_scaling_value(1e12, 10, 4, 20.0) == pytest.approx(2000.0)
