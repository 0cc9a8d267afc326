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


def test_clock_record_keeps_the_timed_region():
    """Only samples taken inside the timed region enter the clock record:
    the idle clocks before and after it, and their reasons, do not."""
    b = _bench()
    samples = [(0.0, 2070.0, 150.0, []), (0.1, 2070.0, 160.0, []),
               (1.0, 1800.0, 1300.0, ["sw_power_cap"]),
               (1.5, 1700.0, 1400.0, ["sw_power_cap"]),
               (2.0, 1750.0, 1380.0, ["sw_power_cap"]),
               (3.0, 2070.0, 170.0, ["hw_slowdown"])]
    rec = b.summarize_clocks(samples, 0.9, 2.1, max_mhz=2070.0)
    assert rec["samples"] == 3 and rec["window"] == "timed region"
    assert rec["sm_mhz"] == 1750.0 and rec["sm_min_mhz"] == 1700.0
    assert rec["power_w_max"] == 1400.0 and rec["power_w_median"] == 1380.0
    assert rec["reasons"] == ["sw_power_cap"] and rec["sm_max_mhz"] == 2070.0


def test_clock_record_of_a_region_shorter_than_the_period():
    """A region between two samples takes the two nearest to its middle."""
    b = _bench()
    samples = [(0.0, 2070.0, 150.0, []), (1.0, 1900.0, 900.0, []),
               (1.2, 1850.0, 950.0, ["sw_power_cap"]),
               (5.0, 2070.0, 150.0, [])]
    rec = b.summarize_clocks(samples, 1.05, 1.1)
    assert rec["samples"] == 2 and rec["window"].startswith("nearest")
    assert rec["sm_mhz"] == 1875.0 and rec["reasons"] == ["sw_power_cap"]
    empty = b.summarize_clocks([], 0.0, 1.0)
    assert empty["samples"] == 0 and empty["sm_mhz"] is None


def test_clock_sampler_without_a_driver():
    """With neither NVML nor nvidia-smi reachable the record says so and
    carries no clocks; with either, a stop() returns a record."""
    b = _bench()
    s = b.ClockSampler("GPU-00000000-0000-0000-0000-000000000000")
    rec = s.stop(0.0, 1.0)
    assert "reasons" in rec and "sm_mhz" in rec
    if s.source is None:
        assert rec["sm_mhz"] is None and rec["error"]


def test_hbm_roofline_arithmetic():
    """Algorithmic bytes per launch over the launch time, against the
    measured copy bandwidth."""
    b = _bench()
    peaks = {"hbm_gbs": 6784.5}
    # 33,570,816 B (65536 x 64 x 64 fp32 A, B, C) in 12.5 us
    r = b.hbm_roofline(5.37e8, 33570816, 0.0125, peaks, "measured", 302.3,
                       42.9)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(33570816 / 12.5e-6 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6784.5)
    assert r["frac_tensor"] == pytest.approx(42.9 / 302.3)


def test_traffic_records_follow_the_sources(monkeypatch):
    """A DRAM-traffic record counts only while its kernel's sources hash to
    the value stored with it; every record names an existing summary."""
    import json
    b = _bench()
    path = os.path.join(ROOT, "profiles", "traffic.json")
    records = json.load(open(path))
    for key, rec in records.items():
        kernel, workload = key.split(":")
        assert kernel in b.KERNEL_SOURCES, key
        assert rec["dram_bytes_per_launch"] > 0
        assert os.path.exists(os.path.join(ROOT, rec["summary"])), key
        got = b.recorded_traffic(kernel, workload)
        if rec["source_hash"] == b.kernel_source_hash(kernel):
            assert got == rec["dram_bytes_per_launch"]
        else:
            assert got is None
    # a changed source invalidates the record
    monkeypatch.setattr(b, "kernel_source_hash", lambda k: "0" * 16)
    assert b.recorded_traffic("tf32x3", "sq4096") is None
    assert b.recorded_traffic("tf32x3", "no-such-workload") is None
