"""The multi-GPU path of bench.py on the CPU: two gloo ranks.

Each rank multiplies its own problem (no collective on the data path); the
only cross-rank steps are the barrier and the max-over-ranks reduction of
the timed region, from which the whole-job value is computed.  The
reference arm runs on rank 0 only.
"""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from conftest import ROOT  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r "measured" 10 + 5 r milliseconds for 3 steps of 2e9 flops
        ms = bench.reduce_max_over_ranks(10.0 + 5.0 * rank)
        value = bench.weak_scaling_value(2e9, 3, world, ms)
        dist.barrier()
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    # every process of the test (the ranks and the manager holding their
    # results) is spawned, never forked from this multi-threaded process
    with mp.get_context("spawn").Manager() as manager:
        out = manager.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world,
                           join=True, start_method="spawn")
        results = dict(out)
    assert set(results) == {0, 1}
    for rank in range(world):
        ms, value = results[rank]
        assert ms == 15.0                      # the slower rank's time
        # all ranks' flops (2 x 3 x 2e9) over 15 ms
        assert value == pytest.approx(2 * 3 * 2e9 / 15e-3 / 1e12)


def test_single_process_reduction_is_identity():
    import bench
    assert bench.reduce_max_over_ranks(7.5) == 7.5
    assert bench.weak_scaling_value(1e12, 2, 1, 1000.0) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import argparse
    import bench
    from dense_fp32_matrix_02_gb300 import synth
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = argparse.Namespace(steps=1, warmup=0)
    bench.run_reference(args, synth.WORKLOADS["sq64"], {"workload": "sq64"})
    assert capsys.readouterr().out == ""        # rank 1: no work, no line
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("LOCAL_RANK", "0")
    bench.run_reference(args, synth.WORKLOADS["sq64"], {"workload": "sq64"})
    import json
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
