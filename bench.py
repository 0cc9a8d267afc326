"""Benchmark of the FP32 GEMM C = A·B (libgemm_f32, one JSON line on stdout).

Default workload: M = N = K = 4096, row-major float32, entries uniform in
[-1, 1) from SplitMix64 seed 2.  A step is one gemm_f32 call over the whole
problem.  Inputs sit in HBM before the timed region; consecutive steps
rotate over three input/output sets (3 × 192 MB, well over the 129 MB L2),
so no step finds its operands left in L2 by the step before.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank multiplies its own full problem on its own
GPU (independent problems, no collective on the data path: weak scaling);
the value is all ranks' flops over the slowest rank's time.

``--impl reference`` times the float64 CPU oracle on this machine's host
cores instead (rank 0 only), each step a bounded block of rows of the same
workload.

The 3xTF32 kernel's roof is the TF32 tensor rate that cuBLAS reaches in the
same run (``tf32_probe``), divided by the three TF32 products per
multiply-add; the FFMA kernels' roof is the library's FMA-chain probe
(``ffma_probe``).  The default 4096^3 run also adds ``sub_records``:
secondary figures, each timed on its own with its own clock record (the
plain gemm_f32 call, the two FFMA kernels forced, and the other workloads
through gemm_f32_ws); none of them enters the headline value.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("FP32 GEMM TFLOPS at M=N=K=4096 and % of GB300 FP32 roofline, "
          "1 GPU")
ALGOS = {"auto": 0, "simt": 1, "tma": 2, "tf32x3": 3}
FP32_LANES_PER_SM = 128  # FFMA lanes per SM on GB300 (4 SMSPs x 32)


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="sq4096")
    p.add_argument("--algo", default="auto", choices=list(ALGOS))
    p.add_argument("--op", default="nn", choices=["nn", "nt", "tn", "tt"],
                   help="operand forms (gemm_f32_batched_ws); nn = plain")
    p.add_argument("--batch", type=int, default=1,
                   help="independent products per step (gemm_f32_batched)")
    p.add_argument("--epilogue", default="none",
                   choices=["none", "bias", "bias_gelu"],
                   help="fused epilogue C = act(A·B + bias) "
                        "(gemm_f32_bias_act)")
    p.add_argument("--precision", default="fp32",
                   choices=["fp32", "bf16", "f16"],
                   help="fp32: the FP32 product (default); bf16/f16: the "
                        "mixed-precision product gemm_f32_mixed16 on 16-bit "
                        "operands resident in HBM")
    p.add_argument("--from-f32", action="store_true",
                   help="with --precision bf16/f16: time gemm_f32_mixed "
                        "(fp32 operands rounded inside the step)")
    p.add_argument("--graph", action="store_true",
                   help="capture the timed steps in CUDA graphs (one per "
                        "timing chunk) and time their replay")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-sub-records", action="store_true",
                   help="skip the secondary timings the default run adds "
                        "(the plain call, the FFMA kernels, the other "
                        "workloads)")
    args = p.parse_args()
    if args.epilogue != "none" and (args.algo != "auto" or args.op != "nn"
                                    or args.batch != 1):
        p.error("--epilogue runs gemm_f32_bias_act, which picks its kernel "
                "itself: use it with --algo auto --op nn --batch 1")
    if args.precision != "fp32" and (args.algo != "auto" or args.op != "nn"
                                     or args.batch != 1
                                     or args.epilogue != "none"):
        p.error("--precision bf16/f16 runs the mixed-precision product alone")
    if args.from_f32 and args.precision == "fp32":
        p.error("--from-f32 goes with --precision bf16/f16")
    return args


# ------------------------------------------------------------------ helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
            "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}, "fallback"


# sources each kernel is built from (its counters go stale when one changes)
KERNEL_SOURCES = {
    "tf32x3": ["tf32x3_gemm.cu", "tcgen05.cuh", "common.cuh", "kernels.h"],
    "tf32x3_stream": ["tf32x3_stream.cu", "tcgen05.cuh", "common.cuh",
                      "kernels.h"],
    "simt": ["simt_gemm.cu", "ffma_tile.cuh", "common.cuh", "kernels.h"],
    "tma": ["tma_ffma_gemm.cu", "ffma_tile.cuh", "common.cuh", "kernels.h"],
    "mixed16": ["mixed_gemm.cu", "tcgen05.cuh", "common.cuh", "kernels.h"],
}
TF32_FLOP_PER_CLK_PER_SM = 4096  # tcgen05 kind::tf32 dense (ncu peak rate)


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_fp32_matrix_02_gb300", "csrc")
    for name in KERNEL_SOURCES.get(kernel, []):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def product_launches(plan, ws_bytes):
    """Kernel launches of one automatic product: a split plan adds the
    reduction kernel when the partial tiles go through scratch, or, when
    its split tiles reduce within clusters, a launch of their own after the
    whole tiles (if any)."""
    if plan["algo"] != 3 or plan["splits"] < 2:
        return 1
    if ws_bytes:
        return 2
    return 2 if plan["whole_tiles"] > 0 else 1


def hbm_roofline(flops, nbytes, kernel_ms, peaks, peaks_src, tensor_peak,
                 achieved):
    """Roofline entry of a memory-bound launch: algorithmic bytes per
    launch over its time against the measured copy bandwidth, the tensor
    figures beside it."""
    gbs = nbytes / (kernel_ms / 1e3) / 1e9
    return {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
            "peak_source": f"{peaks_src} HBM copy bandwidth",
            "tensor_peak_tflops": tensor_peak,
            "frac_tensor": achieved / tensor_peak}


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary of this kernel on
    this workload, if it was taken on the kernel's current sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            rec = json.load(f).get(f"{kernel}:{workload}")
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_hash") != kernel_source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


# clock-event reason bits of the NVML API (nvml.h, "ClocksEventReasons")
NVML_REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8,
                "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
                "hw_power_brake_slowdown": 0x80}
NVML_CLOCK_SM = 1


class _Nvml:
    """The few read-only NVML queries the clock record needs, through
    ctypes (libnvidia-ml ships with the driver).  Raises OSError when the
    library or the device is not there."""

    def __init__(self, uuid):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        for name, args in (
                ("nvmlInit_v2", []),
                ("nvmlShutdown", []),
                ("nvmlDeviceGetHandleByUUID",
                 [ctypes.c_char_p, ctypes.POINTER(ctypes.c_void_p)]),
                ("nvmlDeviceGetClockInfo",
                 [ctypes.c_void_p, ctypes.c_int,
                  ctypes.POINTER(ctypes.c_uint)]),
                ("nvmlDeviceGetMaxClockInfo",
                 [ctypes.c_void_p, ctypes.c_int,
                  ctypes.POINTER(ctypes.c_uint)]),
                ("nvmlDeviceGetPowerUsage",
                 [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint)]),
                ("nvmlDeviceGetCurrentClocksEventReasons",
                 [ctypes.c_void_p, ctypes.POINTER(ctypes.c_ulonglong)])):
            fn = getattr(self.lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        self.dev = ctypes.c_void_p()
        if not uuid or self.lib.nvmlDeviceGetHandleByUUID(
                uuid.encode(), ctypes.byref(self.dev)) != 0:
            self.lib.nvmlShutdown()
            raise OSError("no NVML handle for this device")
        v = ctypes.c_uint()
        self.max_mhz = (float(v.value) if self.lib.nvmlDeviceGetMaxClockInfo(
            self.dev, NVML_CLOCK_SM, ctypes.byref(v)) == 0 else None)

    def sample(self):
        """(SM MHz, watts, reason bits); None for a query that failed."""
        ct = self.ct
        mhz, mw, bits = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        ok1 = self.lib.nvmlDeviceGetClockInfo(
            self.dev, NVML_CLOCK_SM, ct.byref(mhz)) == 0
        ok2 = self.lib.nvmlDeviceGetPowerUsage(self.dev, ct.byref(mw)) == 0
        ok3 = self.lib.nvmlDeviceGetCurrentClocksEventReasons(
            self.dev, ct.byref(bits)) == 0
        return (float(mhz.value) if ok1 else None,
                mw.value / 1e3 if ok2 else None,
                int(bits.value) if ok3 else None)

    def close(self):
        self.lib.nvmlShutdown()


def summarize_clocks(samples, t0, t1, max_mhz=None):
    """Clock record of the samples (time, SM MHz, watts, reason names)
    taken between t0 and t1 (the timed region); when none fell inside
    (a region shorter than the sampling period), the ones nearest to it."""
    inside = [x for x in samples if t0 <= x[0] <= t1]
    where = "timed region"
    if not inside and samples:
        mid = 0.5 * (t0 + t1)
        inside = sorted(samples, key=lambda x: abs(x[0] - mid))[:2]
        where = "nearest to the timed region (shorter than the period)"
    sm = [x[1] for x in inside if x[1] is not None]
    power = [x[2] for x in inside if x[2] is not None]
    reasons = sorted({r for x in inside for r in x[3]})
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_min_mhz": min(sm) if sm else None,
            "sm_max_mhz": max_mhz,
            "power_w_median": statistics.median(power) if power else None,
            "power_w_max": max(power) if power else None,
            "samples": len(inside), "window": where,
            "reasons": reasons}


class ClockSampler:
    """SM clock, power and clock-event reasons, sampled while the timed
    region runs: NVML every 2 ms from a thread, else nvidia-smi every
    200 ms.  `stop(t0, t1)` keeps the samples taken between the
    time.perf_counter() stamps t0 and t1."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    PERIOD_S = 0.002

    def __init__(self, gpu_id=None):
        import threading
        self.proc = None
        self.nvml = None
        self.error = None
        self.samples = []
        self.smi_max = []
        self.source = None
        try:
            self.nvml = _Nvml(gpu_id)
        except (OSError, AttributeError) as e:
            self.error = f"NVML: {e}"
        if self.nvml is not None:
            self.source = "nvml, every 2 ms"
            self.done = threading.Event()
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}",
               "--format=csv,noheader,nounits", "-lms", "200"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi, every 200 ms"
            self.done = threading.Event()
            self.thread = threading.Thread(target=self._read_smi, daemon=True)
            self.thread.start()
        except OSError as e:
            self.error = f"{self.error}; nvidia-smi: {e}"

    def _poll(self):
        while not self.done.is_set():
            mhz, watts, bits = self.nvml.sample()
            names = ([n for n, b in NVML_REASONS.items() if bits & b]
                     if bits is not None else [])
            self.samples.append((time.perf_counter(), mhz, watts, names))
            self.done.wait(self.PERIOD_S)

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in self.proc.stdout:
            t = time.perf_counter()
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz, smax, watts = (float(parts[1]), float(parts[2]),
                                    float(parts[3]))
            except ValueError:
                continue
            self.smi_max.append(smax)
            active = [n for n, v in zip(names, parts[5:9])
                      if v.lower().startswith("active")]
            self.samples.append((t, mhz, watts, active))

    def stop(self, t0=None, t1=None):
        """The clock record of the samples between t0 and t1 (all of them
        when no window is given)."""
        if self.source is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "error": self.error or "no clock source"}
        if self.nvml is not None:
            self.done.set()
            self.thread.join(timeout=5)
            self.nvml.close()
            max_mhz = self.nvml.max_mhz
        else:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            self.thread.join(timeout=5)
            max_mhz = max(self.smi_max) if self.smi_max else None
        if t0 is None:
            t0, t1 = float("-inf"), float("inf")
        rec = summarize_clocks(list(self.samples), t0, t1, max_mhz)
        rec["source"] = self.source
        return rec


def reduce_max_over_ranks(value, device=None):
    """Largest `value` over all ranks of the process group (itself alone
    when there is no group)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and \
            dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(flops_per_rank, steps, world, ms_slowest):
    """Whole-job TFLOP/s: every rank's flops over the slowest rank's time."""
    return flops_per_rank * steps * world / (ms_slowest / 1e3) / 1e12


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------- reference (oracle)
def oracle_rows_timing(a, b, rows, threads=0):
    import oracle
    t = time.perf_counter()
    oracle.gemm(a[:rows], b, threads=threads)
    return time.perf_counter() - t


def calibrate_rows(a, b, target_s):
    """Rows of A whose oracle product takes about target_s seconds."""
    M = a.shape[0]
    rows = min(M, 8)
    t = oracle_rows_timing(a, b, rows)
    while t < 0.2 and rows < M:
        rows = min(M, rows * 4)
        t = oracle_rows_timing(a, b, rows)
    return max(1, min(M, int(rows * target_s / max(t, 1e-6))))


def cpu_baseline(w, a, b, target_s):
    import oracle
    rows = calibrate_rows(a, b, target_s)
    t = oracle_rows_timing(a, b, rows)
    flops = 2.0 * rows * w.N * w.K
    cores = oracle.load().max_threads()
    # and one thread alone, on a quarter of the per-core share of rows
    rows1 = max(1, rows // max(1, 4 * cores))
    t1 = oracle_rows_timing(a, b, rows1, threads=1)
    return {"value": flops / t / 1e12, "unit": "TFLOP/s",
            "cores": cores, "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of A times all of B "
                      f"({rows}x{w.N}x{w.K}, float64 accumulation, "
                      f"{t:.1f} s)",
            "single_thread": {
                "value": 2.0 * rows1 * w.N * w.K / t1 / 1e12,
                "unit": "TFLOP/s",
                "sample": f"rows 0..{rows1 - 1} ({rows1}x{w.N}x{w.K}, "
                          f"{t1:.1f} s, 1 thread)"}}


def run_reference(args, w, config):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    a, b = w.operands()
    nthreads = oracle.load().max_threads()
    per_step = max(0.05, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    rows = calibrate_rows(a, b, per_step)
    for _ in range(args.warmup):
        oracle_rows_timing(a, b, rows)
    times = [oracle_rows_timing(a, b, rows) for _ in range(args.steps)]
    total = sum(times)
    flops = 2.0 * rows * w.N * w.K
    value = flops * args.steps / total / 1e12
    sample = (f"rows 0..{rows - 1} of A times all of B per step "
              f"({rows}x{w.N}x{w.K}, float64 accumulation)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": config,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def timed_region(step, args, stream, dev, world):
    """W warm-up steps, then K steps between CUDA events on `stream`, with
    a barrier and a synchronize on both sides and SM clocks sampled
    meanwhile.  Returns (ms, max ms over ranks, clocks, wall seconds)."""
    import torch
    import torch.distributed as dist

    from dense_fp32_matrix_02_gb300 import gemm as G
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if G.device_status() != 0:
        raise SystemExit("kernel status word set during warm-up")
    try:
        gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:  # noqa: BLE001 - older torch
        gpu_uuid = None
    sampler = ClockSampler(gpu_uuid)
    if sampler.nvml is None:
        time.sleep(0.3)  # nvidia-smi's first sample
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # events at the edges of 5 equal chunks of the K steps: the whole
    # region is timed once, the chunks give the spread between samples
    nchunks = min(5, args.steps)
    edges = [round(c * args.steps / nchunks) for c in range(nchunks + 1)]
    events = [torch.cuda.Event(enable_timing=True) for _ in edges]
    graphs = None
    if getattr(args, "graph", False):
        # each chunk's steps captured once (the warm-up above did the
        # library's one-time set-up eagerly), replayed once untimed
        cap = torch.cuda.Stream(dev)
        graphs = []
        for c in range(nchunks):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                for i in range(edges[c], edges[c + 1]):
                    step(i, cap)
            graphs.append(g)
        with torch.cuda.stream(stream):
            for g in graphs:
                g.replay()
        torch.cuda.synchronize()
    wall0 = time.perf_counter()
    events[0].record(stream)
    for c in range(nchunks):
        if graphs is not None:
            with torch.cuda.stream(stream):
                graphs[c].replay()
        else:
            for i in range(edges[c], edges[c + 1]):
                step(i)
        events[c + 1].record(stream)
    torch.cuda.synchronize()
    wall1 = time.perf_counter()
    wall = wall1 - wall0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop(wall0, wall1)
    ms = events[0].elapsed_time(events[-1])
    ms_max = reduce_max_over_ranks(ms, dev)
    if G.device_status() != 0:
        raise SystemExit("kernel status word set during the timed region")
    chunk_ms = [events[c].elapsed_time(events[c + 1]) /
                max(1, edges[c + 1] - edges[c]) for c in range(nchunks)]
    clocks["chunk_ms_per_step"] = chunk_ms
    return ms, ms_max, clocks, wall


def sample_stats(flops_per_step, chunk_ms):
    """Median, worst and best TFLOP/s over the timed chunks."""
    v = sorted(flops_per_step / (m / 1e3) / 1e12 for m in chunk_ms if m > 0)
    if not v:
        return None
    return {"n": len(v), "median": statistics.median(v), "min": v[0],
            "max": v[-1], "unit": "TFLOP/s"}


def rotating_sets(set_bytes, l2_bytes):
    """Input/output sets to rotate between timed steps so that the ones a
    step touches were last used more than 2x the L2 size of traffic ago."""
    return max(3, min(8192, math.ceil(2.1 * l2_bytes / max(set_bytes, 1))))


def measure_ffma_peak(dev, stream, target_ms=60.0):
    """The FP32 pipe's rate from the library's FMA-chain probe (best of 3
    launches of about target_ms each), with the SM clocks seen meanwhile."""
    import torch

    from dense_fp32_matrix_02_gb300 import gemm as G
    sink = torch.zeros(256, device=dev)
    handle = stream.cuda_stream

    def run(iters):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        G.ffma_peak_launch(iters, sink, handle)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    iters = 256
    run(iters)
    t = run(iters)
    iters = max(256, int(iters * target_ms / max(t, 1e-3)))
    run(iters)
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:  # noqa: BLE001 - older torch
        uuid = None
    sampler = ClockSampler(uuid)
    if sampler.nvml is None:
        time.sleep(0.3)  # nvidia-smi's first sample
    t0 = time.perf_counter()
    best = min(run(iters) for _ in range(3))
    clocks = sampler.stop(t0, time.perf_counter())
    flops = G.ffma_peak_flops(iters)
    return {"tflops": flops / (best / 1e3) / 1e12, "ms": best,
            "iters": iters, "sm_mhz": clocks.get("sm_mhz"),
            "reasons": clocks.get("reasons")}


def _gpu_uuid(dev):
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:  # noqa: BLE001 - older torch
        return None


def measure_tf32_peak(dev, stream, n=8192, reps=10):
    """cuBLAS's dense TF32 tensor rate on this GPU, measured in this run:
    an n x n x n float32 torch.matmul with TF32 tensor math allowed (one
    TF32 product, fp32 accumulation), best of `reps` launches timed one
    at a time with CUDA events, with the SM clocks seen meanwhile.  It is
    the denominator of the 3xTF32 kernel (which does three TF32 products
    per multiply-add), the way the bf16 GEMM is for the 16-bit one."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        g = torch.Generator(device=dev)
        g.manual_seed(0)
        a = torch.rand(n, n, device=dev, generator=g)
        b = torch.rand(n, n, device=dev, generator=g)
        c = torch.empty(n, n, device=dev)
        with torch.cuda.stream(stream):
            for _ in range(3):
                torch.matmul(a, b, out=c)
        torch.cuda.synchronize()
        sampler = ClockSampler(_gpu_uuid(dev))
        if sampler.nvml is None:
            time.sleep(0.3)  # nvidia-smi's first sample
        t0 = time.perf_counter()
        times = []
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                torch.matmul(a, b, out=c)
                e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        clocks = sampler.stop(t0, time.perf_counter())
        del a, b, c
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    best = min(times)
    return {"tflops": 2.0 * n ** 3 / (best / 1e3) / 1e12, "ms": best,
            "n": n, "reps": reps, "sm_mhz": clocks.get("sm_mhz"),
            "reasons": clocks.get("reasons"),
            "how": f"cuBLAS float32 matmul {n}^3 with TF32 tensor math "
                   f"(torch allow_tf32), best of {reps}, CUDA events"}


def time_steps(step, stream, dev, warmup=5, target_ms=40.0, min_steps=20,
               max_steps=4000):
    """Secondary timing of one step function: `warmup` untimed steps, a
    short calibration, then enough steps for about target_ms (at least
    min_steps) between CUDA events on `stream`, with the SM clocks seen
    meanwhile.  Returns (ms per step, steps, clock record)."""
    import torch
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(5):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    est = max(e0.elapsed_time(e1) / 5, 1e-4)
    steps = int(min(max_steps, max(min_steps, target_ms / est)))
    sampler = ClockSampler(_gpu_uuid(dev))
    if sampler.nvml is None:
        time.sleep(0.3)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop(t0, time.perf_counter())
    return e0.elapsed_time(e1) / steps, steps, clocks


def sub_record(w, ms, steps, clocks, kernel, entry, peaks, tf32_peak,
               fp32_peak):
    """One secondary figure: TFLOP/s over the step time, with the roof that
    bounds the kernel (tensor/3 for 3xTF32, the FFMA probe for the FFMA
    kernels, the copy bandwidth where intensity x bandwidth is lower)."""
    tflops = w.flops / (ms / 1e3) / 1e12
    rec = {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
           "entry": entry, "kernel": kernel, "value": tflops,
           "unit": "TFLOP/s", "ms_per_step": ms, "steps": steps,
           "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_min_mhz",
                                                 "samples", "reasons")},
           "traffic": recorded_traffic(kernel, w.name),
           "algorithmic_bytes": w.bytes}
    bw_roof = w.flops / w.bytes * peaks["hbm_gbs"] / 1e3
    if kernel.startswith("tf32x3"):
        if bw_roof < tf32_peak / 3.0:
            gbs = w.bytes / (ms / 1e3) / 1e9
            rec["roofline"] = {"bound": "hbm", "achieved": gbs,
                               "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": gbs / peaks["hbm_gbs"]}
        else:
            rec["roofline"] = {"bound": "tensor", "achieved": tflops,
                               "peak": tf32_peak / 3.0, "unit": "TFLOP/s",
                               "frac": tflops / (tf32_peak / 3.0)}
    else:
        rec["roofline"] = {"bound": "alu", "achieved": tflops,
                           "peak": fp32_peak, "unit": "TFLOP/s",
                           "frac": tflops / fp32_peak}
    return rec


def run_sub_records(dev, stream, head_sets, peaks, tf32_peak, fp32_peak):
    """Secondary figures of the default run, each timed on its own (CUDA
    events, its own clock record), none of them part of the headline:

    * 4096^3 through gemm_f32 itself (no lent scratch: nothing split);
    * 4096^3 on the two FFMA kernels, forced (TMA-fed and cp.async);
    * the other workloads through gemm_f32_ws with the scratch it asks
      for, as the headline runs 4096^3.
    Inputs rotate over sets together larger than 2x the L2."""
    import torch

    from dense_fp32_matrix_02_gb300 import gemm as G
    from dense_fp32_matrix_02_gb300 import synth

    w = synth.WORKLOADS["sq4096"]
    h = stream.cuda_stream
    out = []

    def forced(algo):
        def step(i):
            ta, tb, tc = head_sets[i % len(head_sets)]
            G.gemm_f32_ptr(w.M, w.N, w.K, ta.data_ptr(), w.K, tb.data_ptr(),
                           w.N, tc.data_ptr(), w.N, h, algo)
        return step

    for algo, entry, kernel in ((0, "gemm_f32", "tf32x3"),
                                (2, "gemm_f32_ex(TMA)", "tma"),
                                (1, "gemm_f32_ex(SIMT)", "simt")):
        ms, steps, clocks = time_steps(forced(algo), stream, dev)
        out.append(sub_record(w, ms, steps, clocks, kernel, entry, peaks,
                              tf32_peak, fp32_peak))
        if algo == 0:
            out[-1]["note"] = "no scratch lent: the last round of tiles " \
                              "runs whole"
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    for name in ("mlp", "sq1024", "rag1000", "skinny", "sq64"):
        v = synth.WORKLOADS[name]
        a, b = v.operands()
        ta0 = torch.from_numpy(a).to(dev)
        tb0 = torch.from_numpy(b).to(dev)
        n = rotating_sets(v.bytes, l2)
        sets = [(ta0 if i == 0 else ta0.clone(),
                 tb0 if i == 0 else tb0.clone(),
                 torch.empty(v.M, v.N, device=dev)) for i in range(n)]
        need = G.workspace_size(v.M, v.N, v.K)
        ws = torch.empty(max(need // 4, 1), device=dev) if need else None
        p = G.plan(v.M, v.N, v.K)
        kernel = G.ALGO_NAMES.get(p["algo"], str(p["algo"]))
        if kernel == "tf32x3" and p["variant"] == "streaming":
            kernel = "tf32x3_stream"

        def step(i, v=v, sets=sets, ws=ws, need=need):
            ta, tb, tc = sets[i % len(sets)]
            G.gemm_f32_ws_ptr(v.M, v.N, v.K, ta.data_ptr(), v.K,
                              tb.data_ptr(), v.N, tc.data_ptr(), v.N,
                              ws.data_ptr() if ws is not None else 0, need, h)

        ms, steps, clocks = time_steps(step, stream, dev)
        rec = sub_record(v, ms, steps, clocks, kernel, "gemm_f32_ws", peaks,
                         tf32_peak, fp32_peak)
        rec["plan"] = p
        out.append(rec)
        del sets, ws
    if G.device_status() != 0:
        raise SystemExit("kernel status word set during the sub-records")
    return out


# ------------------------------------------------------------------ ours
def run_ours(args, w, config):
    import torch
    import torch.distributed as dist

    from dense_fp32_matrix_02_gb300 import gemm as G
    from dense_fp32_matrix_02_gb300 import synth

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    algo = ALGOS[args.algo]
    a, b = w.operands()
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    nsets = rotating_sets(w.bytes * args.batch, l2_bytes)
    ta0 = torch.from_numpy(a).to(dev)
    tb0 = torch.from_numpy(b).to(dev)
    sets = [(ta0, tb0, torch.empty(w.M, w.N, device=dev))]
    for _ in range(nsets - 1):
        sets.append((ta0.clone(), tb0.clone(), torch.empty(w.M, w.N,
                                                           device=dev)))
    stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream
    ran = G.select_algo(w.M, w.N, w.K, ta0.data_ptr(), w.K, tb0.data_ptr(),
                        w.N, sets[0][2].data_ptr(), w.N) if algo == 0 else algo

    # AUTO goes through gemm_f32_ws with the scratch it asks for (split-K
    # on grids too small to fill the GPU); a forced kernel through gemm_f32_ex
    ws_bytes = G.workspace_size(w.M, w.N, w.K) if algo == 0 else 0
    ws = torch.empty(max(ws_bytes // 4, 1), device=dev) if ws_bytes else None
    launches_per_step = product_launches(G.plan(w.M, w.N, w.K), ws_bytes) \
        if algo == 0 else 1

    batched = args.op != "nn" or args.batch > 1
    if batched:
        # stored operands: A as K x M when op(A) = T, B as N x K when
        # op(B) = T; `batch` copies laid out back to back
        ta_, tb_ = args.op[0] == "t", args.op[1] == "t"
        sa = torch.from_numpy(a.T.copy() if ta_ else a).to(dev)
        sb = torch.from_numpy(b.T.copy() if tb_ else b).to(dev)
        bA = sa.unsqueeze(0).repeat(args.batch, 1, 1)
        bB = sb.unsqueeze(0).repeat(args.batch, 1, 1)
        bsets = [(bA, bB, torch.empty(args.batch, w.M, w.N, device=dev))]
        for _ in range(nsets - 1):
            bsets.append((bA.clone(), bB.clone(),
                          torch.empty(args.batch, w.M, w.N, device=dev)))
        # scratch gemm_f32_batched_ws asks for: the transposed copy of A
        # for Aᵀ·B (one more launch), split-K scratch for a single product
        bws_bytes = G.batched_workspace_size(int(ta_), int(tb_), w.M, w.N,
                                             w.K, args.batch)
        bws = torch.empty(max(bws_bytes, 1), dtype=torch.uint8, device=dev)
        launches_per_step = 1
        if ta_ and not tb_:
            launches_per_step += 1
        if args.batch == 1 and not tb_ and G.workspace_size(w.M, w.N, w.K):
            launches_per_step += 1

    if batched:  # aligned operands: the tensor kernel takes every form
        ran = 3

    fused = args.epilogue != "none"
    if fused:
        ebias = torch.from_numpy(
            synth.make_operands(1, w.N, 1, seed=7)[1][0]).to(dev)
        eact = 1 if args.epilogue == "bias_gelu" else 0

    def step(i, on=None):
        # on: the stream to launch on (the capture stream in graph mode)
        s_obj = on if on is not None else stream
        h = s_obj.cuda_stream
        if fused:
            ta, tb, tc = sets[i % nsets]
            G.gemm_f32_bias_act_ptr(w.M, w.N, w.K, ta.data_ptr(), w.K,
                                    tb.data_ptr(), w.N, ebias.data_ptr(),
                                    eact, tc.data_ptr(), w.N,
                                    ws.data_ptr() if ws is not None else 0,
                                    ws_bytes, h)
            return
        if batched:
            xa, xb, xc = bsets[i % nsets]
            G.gemm_f32_batched(xa, xb, xc, trans_a=ta_, trans_b=tb_,
                               stream=s_obj, workspace=bws)
            return
        ta, tb, tc = sets[i % nsets]
        if algo == 0:
            G.gemm_f32_ws_ptr(w.M, w.N, w.K, ta.data_ptr(), w.K,
                              tb.data_ptr(), w.N, tc.data_ptr(), w.N,
                              ws.data_ptr() if ws is not None else 0,
                              ws_bytes, h)
        else:
            G.gemm_f32_ptr(w.M, w.N, w.K, ta.data_ptr(), w.K, tb.data_ptr(),
                           w.N, tc.data_ptr(), w.N, h, algo)

    ms, ms_max, clocks, wall = timed_region(step, args, stream, dev, world)

    flops = float(w.flops) * args.batch
    value = weak_scaling_value(flops, args.steps, world, ms_max)
    samples = sample_stats(flops, clocks.pop("chunk_ms_per_step"))
    # one GEMM launch per step (plus the split-K reduction when it splits);
    # launch gaps are included
    kernel_ms = ms / args.steps

    # ---- end to end: pinned host buffers through the public API
    # (gemm_f32_host: B, then row chunks of A copied in while earlier
    # chunks are multiplied and their C copied back; forced kernels go
    # through gemm_f32_ex between plain copies)
    if batched:
        hba = bsets[0][0].cpu().pin_memory()
        hbb = bsets[0][1].cpu().pin_memory()
        hbc = torch.empty(args.batch, w.M, w.N).pin_memory()
    ha = torch.from_numpy(a).pin_memory()
    hb = torch.from_numpy(b).pin_memory()
    hc = torch.empty(w.M, w.N, dtype=torch.float32).pin_memory()
    ea, eb, ec = sets[0]
    e_steps = max(1, args.e2e_steps)

    def e2e_step():
        if batched:  # host copies of every operand, then the batched call
            xa, xb, xc = bsets[0]
            xa.copy_(hba, non_blocking=True)
            xb.copy_(hbb, non_blocking=True)
            G.gemm_f32_batched(xa, xb, xc, trans_a=ta_, trans_b=tb_,
                               stream=stream, workspace=bws)
            hbc.copy_(xc, non_blocking=True)
            return
        if algo == 0:
            G.gemm_f32_host(ha, hb, hc, ea, eb, ec, workspace=ws,
                            stream=stream)
        else:
            ea.copy_(ha, non_blocking=True)
            eb.copy_(hb, non_blocking=True)
            G.gemm_f32_ex(ea, eb, ec, algo=algo, stream=stream)
            hc.copy_(ec, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    s2 = torch.cuda.Event(enable_timing=True)
    e2 = torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    for _ in range(e_steps):
        e2e_step()
    e2.record(stream)
    torch.cuda.synchronize()
    e2e_value = weak_scaling_value(
        flops, e_steps, world, reduce_max_over_ranks(s2.elapsed_time(e2), dev))

    # ---- roofline of the (only) kernel
    peaks, peaks_src = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    smax = clocks.get("sm_max_mhz") or peaks.get("sm_max_mhz", 2070.0)
    # FP32 pipe: measured by the FMA-chain probe (primary) and the nameplate
    # 2 flop x 128 lanes x SMs x maximum clock beside it
    probe = measure_ffma_peak(dev, stream)
    fp32_nameplate = 2.0 * sms * FP32_LANES_PER_SM * smax * 1e6 / 1e12
    fp32_peak = probe["tflops"]
    # the TF32 tensor rate, measured here (cuBLAS), for the 3xTF32 roof
    tf32_probe = measure_tf32_peak(dev, stream)
    tf32 = tf32_probe["tflops"]
    achieved = flops / (kernel_ms / 1e3) / 1e12
    algo_name = G.ALGO_NAMES.get(ran, str(ran))
    if algo_name == "tf32x3" and not batched and algo == 0:
        if G.plan(w.M, w.N, w.K)["variant"] == "streaming":
            algo_name = "tf32x3_stream"  # B held in tensor memory
    bw_roof = (flops / (w.bytes * args.batch)) * peaks["hbm_gbs"] / 1e3
    if algo_name in ("tf32x3", "tf32x3_stream") and bw_roof < tf32 / 3.0:
        # memory-bound shape: the copy bandwidth is the roof
        roof = hbm_roofline(flops, w.bytes * args.batch, kernel_ms, peaks,
                            peaks_src, tf32 / 3.0, achieved)
    elif algo_name in ("tf32x3", "tf32x3_stream"):
        # three TF32 tensor products per algorithmic multiply-add: the roof
        # is the TF32 rate cuBLAS reached in this run, / 3
        roof = {"bound": "tensor", "achieved": achieved, "peak": tf32 / 3.0,
                "unit": "TFLOP/s", "frac": achieved / (tf32 / 3.0),
                "peak_source": "measured in this run: cuBLAS TF32 burst "
                               f"{tf32:.1f} TFLOP/s at "
                               f"{tf32_probe['sm_mhz']} MHz median, / 3 "
                               "products"}
        # the earlier derived figure, for comparison: the driver's bf16
        # burst x the nominal TF32/bf16 ratio (1.1/2.25), / 3
        derived = peaks["bf16_tflops"] * (1.1 / 2.25) / 3.0
        roof["peak_derived_from_bf16"] = derived
        roof["frac_derived_from_bf16"] = achieved / derived
        # the sustained figure, for a timed region long enough to meet the
        # power cap: the TF32 burst x the measured bf16 sustained / burst
        # ratio (cuBLAS held for seconds against its best of ten), / 3
        if peaks.get("bf16_tflops_sustained") and peaks.get("bf16_tflops"):
            sus = tf32 * peaks["bf16_tflops_sustained"] \
                / peaks["bf16_tflops"] / 3.0
            roof["peak_sustained"] = sus
            roof["frac_sustained"] = achieved / sus
            roof["peak_sustained_source"] = (
                f"TF32 burst x {peaks_src} bf16 sustained / burst "
                f"({peaks['bf16_tflops_sustained']:.1f} / "
                f"{peaks['bf16_tflops']:.1f}), / 3 products")
        # the tensor pipe's own TF32 rate (ncu peak_sustained: 4096 flop per
        # clock per SM) at the run's maximum clock, / 3 products
        hw = TF32_FLOP_PER_CLK_PER_SM * sms * smax * 1e6 / 1e12 / 3.0
        roof["peak_tensor_pipe_at_clock"] = hw
        roof["frac_tensor_pipe_at_clock"] = achieved / hw
        if clocks.get("sm_mhz"):
            # the same at the median SM clock sampled in the timed region
            # (lower than the maximum once the power cap acts)
            run = TF32_FLOP_PER_CLK_PER_SM * sms * clocks["sm_mhz"] * 1e6 \
                / 1e12 / 3.0
            roof["peak_tensor_pipe_at_run_clock"] = run
            roof["frac_tensor_pipe_at_run_clock"] = achieved / run
    else:
        roof = {"bound": "alu", "achieved": achieved, "peak": fp32_peak,
                "unit": "TFLOP/s", "frac": achieved / fp32_peak,
                "peak_source": "measured: FMA-chain probe on every SM "
                               f"({probe['sm_mhz']} MHz median)",
                "peak_nameplate": fp32_nameplate,
                "frac_nameplate": achieved / fp32_nameplate,
                "nameplate_source": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 "
                                    f"lanes x 2 flop x {smax:.0f} MHz"}
    roof["traffic"] = recorded_traffic(algo_name, w.name)
    roof["algorithmic_bytes"] = w.bytes * args.batch
    roof["kernel_ms"] = kernel_ms

    fp32_roof = min(fp32_peak, bw_roof)
    fp32_roof_nameplate = min(fp32_nameplate, bw_roof)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": config,
        "kernel": algo_name,
        "pct_fp32_roofline": 100.0 * (value / world) / fp32_roof,
        "fp32_roofline_tflops": fp32_roof,
        "fp32_roofline_source": "min(measured FFMA probe, I x HBM)",
        "pct_fp32_roofline_nameplate":
            100.0 * (value / world) / fp32_roof_nameplate,
        "ffma_probe": probe,
        "tf32_probe": tf32_probe,
        "samples": samples,
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s",
                "h2d_bytes_per_step": 4 * (w.M * w.K + w.K * w.N) * args.batch,
                "d2h_bytes_per_step": 4 * w.M * w.N * args.batch},
        "gpu_launches": args.steps * launches_per_step,
        "split_k_workspace_bytes": ws_bytes,
        "clocks": clocks,
        "wall_s_timed": wall,
    }
    if (rank == 0 and world == 1 and not args.no_sub_records
            and w.name == "sq4096" and algo == 0 and not batched
            and not fused and not args.graph):
        line["sub_records"] = run_sub_records(dev, stream, sets, peaks, tf32,
                                              fp32_peak)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, a, b, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------ ours, mixed precision
def run_mixed(args, w, config):
    """The mixed-precision product ("Rendre le GPU rapide", "Les Tensor
    Cores"): 16-bit operands, fp32 accumulation, on the tensor cores."""
    import torch
    import torch.distributed as dist

    from dense_fp32_matrix_02_gb300 import gemm as G

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    if w.K % 8 or w.N % 8:
        raise SystemExit("16-bit operands need K and N multiples of 8")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    t = G.MIXED_BF16 if args.precision == "bf16" else G.MIXED_F16
    a, b = w.operands()
    nsets = rotating_sets(2 * (w.M * w.K + w.K * w.N) + 4 * w.M * w.N,
                          torch.cuda.get_device_properties(dev).L2_cache_size)
    f32 = [(torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev))]
    for _ in range(nsets - 1):
        f32.append((f32[0][0].clone(), f32[0][1].clone()))
    sets = [(G.round16(fa, t), G.round16(fb, t),
             torch.empty(w.M, w.N, device=dev)) for fa, fb in f32]
    if not args.from_f32:
        del f32
    stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream
    ws_bytes = G.mixed_workspace_size(w.M, w.N, w.K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def step(i, on=None):
        h = (on if on is not None else stream).cuda_stream
        xa, xb, xc = sets[i % nsets]
        if args.from_f32:
            fa, fb = f32[i % nsets]
            G.gemm_f32_mixed_ptr(t, w.M, w.N, w.K, fa.data_ptr(), w.K,
                                 fb.data_ptr(), w.N, xc.data_ptr(), w.N,
                                 ws.data_ptr(), ws_bytes, h)
        else:
            G.gemm_f32_mixed16_ptr(t, w.M, w.N, w.K, xa.data_ptr(), w.K,
                                   xb.data_ptr(), w.N, xc.data_ptr(), w.N,
                                   h)

    ms, ms_max, clocks, wall = timed_region(step, args, stream, dev, world)
    flops = float(w.flops)
    value = weak_scaling_value(flops, args.steps, world, ms_max)
    samples = sample_stats(flops, clocks.pop("chunk_ms_per_step"))
    kernel_ms = ms / args.steps

    # ---- end to end: fp32 operands from pinned host memory, the public
    # gemm_f32_mixed call (rounding + product), C back to the host
    ha = torch.from_numpy(a).pin_memory()
    hb = torch.from_numpy(b).pin_memory()
    hc = torch.empty(w.M, w.N, dtype=torch.float32).pin_memory()
    ea = torch.empty(w.M, w.K, device=dev)
    eb = torch.empty(w.K, w.N, device=dev)
    ec = sets[0][2]

    def e2e_step():
        ea.copy_(ha, non_blocking=True)
        eb.copy_(hb, non_blocking=True)
        G.gemm_f32_mixed(ea, eb, t, ec, workspace=ws, stream=stream)
        hc.copy_(ec, non_blocking=True)

    e_steps = max(1, args.e2e_steps)
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    s2 = torch.cuda.Event(enable_timing=True)
    e2 = torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    for _ in range(e_steps):
        e2e_step()
    e2.record(stream)
    torch.cuda.synchronize()
    e2e_value = weak_scaling_value(
        flops, e_steps, world, reduce_max_over_ranks(s2.elapsed_time(e2), dev))

    peaks, peaks_src = load_peaks()
    achieved = flops / (kernel_ms / 1e3) / 1e12
    peak = peaks["bf16_tflops"]  # binary16 has the same nominal dense rate
    nbytes = 2 * (w.M * w.K + w.K * w.N) + 4 * w.M * w.N
    if flops / nbytes * peaks["hbm_gbs"] / 1e3 < peak and not args.from_f32:
        roof = hbm_roofline(flops, nbytes, kernel_ms, peaks, peaks_src, peak,
                            achieved)
    else:
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{peaks_src} bf16 burst (cuBLAS bf16 GEMM)"}
    roof.update({"traffic": None if args.from_f32
                 else recorded_traffic("mixed16", w.name),
                 "algorithmic_bytes": nbytes, "kernel_ms": kernel_ms})
    if args.from_f32:
        roof["note"] = ("step = two rounding kernels + the product; "
                        "achieved is over the whole step")
    line = {
        "metric": f"mixed-precision GEMM TFLOPS ({args.precision} operands, "
                  "fp32 accumulation)",
        "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": args.precision,
        "data": "synthetic", "config": config, "kernel": "mixed16",
        "samples": samples,
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s",
                "h2d_bytes_per_step": 4 * (w.M * w.K + w.K * w.N),
                "d2h_bytes_per_step": 4 * w.M * w.N},
        "gpu_launches": args.steps * (3 if args.from_f32 else 1),
        "clocks": clocks,
        "wall_s_timed": wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        ar = oracle.widen_half(oracle.round_half(a, t), t)
        br = oracle.widen_half(oracle.round_half(b, t), t)
        line["cpu_baseline"] = cpu_baseline(w, ar, br, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse_args()
    from dense_fp32_matrix_02_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    dist_txt = {"uniform": "uniform [-1,1)", "normal": "normal",
                "int": "integers {-2..2}"}
    config = {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
              "op": args.op, "batch": args.batch,
              "epilogue": args.epilogue,
              "layout": "row-major, ld = row width",
              "inputs": f"A {dist_txt[w.dist_a]} (sigma {w.sigma_a}), "
                        f"B {dist_txt[w.dist_b]} (sigma {w.sigma_b}), "
                        f"SplitMix64 seed {w.seed}",
              "l2": "rotating input/output sets between timed steps, "
                    "together more than 2x the L2 size (at least 3 sets "
                    f"of {w.bytes / 2**20:.1f} MiB)",
              "parallelism": f"independent problem per GPU x {args.gpus}",
              "launch": "CUDA graph replay" if args.graph else "stream"}
    if args.precision != "fp32":
        config["precision"] = (f"{args.precision} operands, fp32 products, "
                               "sums and C")
        config["operands"] = ("fp32 in HBM, rounded inside each step"
                              if args.from_f32 else
                              f"{args.precision} in HBM (rounded once before "
                              "timing)")
    if args.impl == "reference":
        run_reference(args, w, config)
    elif args.precision != "fp32":
        run_mixed(args, w, config)
    else:
        run_ours(args, w, config)


if __name__ == "__main__":
    main()
