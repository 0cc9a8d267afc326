"""The FP32 FMA throughput probe that bench.py times as the FFMA kernels'
measured ceiling: it must run, write nothing, count its work, and land in a
plausible band around the nameplate rate (2 flop x 128 FP32 lanes x SMs x
the clock)."""

from __future__ import annotations

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from dense_fp32_matrix_02_gb300 import gemm as G  # noqa: E402

DEV = torch.device("cuda:0")


def test_ffma_probe_rate_is_plausible():
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert G.ffma_peak_flops(10) == 2 * 8 * 16 * 10 * 256 * 8 * sms
    sink = torch.zeros(256, device=DEV)
    G.ffma_peak_launch(256, sink)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    iters = 8192
    s.record()
    G.ffma_peak_launch(iters, sink)
    e.record()
    torch.cuda.synchronize()
    rate = G.ffma_peak_flops(iters) / (s.elapsed_time(e) / 1e3) / 1e12
    nameplate_2100 = 2 * 128 * sms * 2.1e9 / 1e12
    assert 0.3 * nameplate_2100 < rate <= 1.02 * nameplate_2100
    assert not sink.any()
