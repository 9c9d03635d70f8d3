#!/usr/bin/env python3
"""Benchmark of the fused fp16 GEMM + ReLU on GB300.

One "step" is one call of the hot path, C = ReLU(A @ B), on the headline
workload (default ``relu_8192``: M = N = K = 8192, fp16 inputs N(0,1)/sqrt(K),
seed 5).  The inputs (A, B: 256 MiB, C: 128 MiB) are larger than the 126 MB
L2, so no flush is needed between steps.

Prints ONE JSON line:
  value        TFLOP/s, 2*M*N*K*steps*ranks / max-over-ranks device time
               (CUDA events on the launching stream, inputs resident in HBM)
  e2e          the same metric through the C ABI's host-buffer call
               (gemm_f16_from_host: H2D copies of A and B, the GEMM, D2H of C
               every step, pinned host memory)
  roofline     tensor-core bound: achieved TFLOP/s per launch against the
               measured bf16 matmul peak of this machine (fp16 has the same rate)
  cpu_baseline the CPU oracle, as it stands, on a bounded sample of rows
  clocks       SM clock, power and throttle reasons polled through NVML
               (read-only, ~1 ms) inside the timed region
  sweep        every square configuration of the benchmark description
               (64^3 integers, 1000^3, 1024^3, n^3 for n = 512 .. 16384):
               TFLOP/s of single launches (L2 flushed where the operands fit)
               and of back-to-back launches replayed from a CUDA graph
  sustained    the headline workload back to back for a few seconds, with
               the clock samples inside that loop

``--impl reference`` times the CPU oracle instead (the reference arm: a
deliberately slow, obviously correct program on the host cores).

Multi-GPU: the method has no exchange step, so N GPUs run N independent
replicas of the step (weak scaling); torch.distributed is used only for the
barrier and the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM+ReLU TFLOP/s at 4096^3/8192^3 fp16 and % of GB300 dense FP16 peak"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
FP8_PER_BF16 = 2.0            # nominal dense fp8 / bf16 tensor rate (4.5 / 2.25 PFLOP/s)
TENSOR_FLOP_PER_CLK_PER_SM = 8192   # dense fp16/bf16 tcgen05 rate per SM per clock


# ---------------------------------------------------------------- helpers

def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (x itself when running alone)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: every rank does the same steps (replicas), timed by the slowest rank."""
    return world * flops_per_step * steps / (max_ms * 1e-3) / 1e12


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS, "hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


# Files that define the device code and its launch geometry.  Host-only files
# (argument checks, the tuned selection table) do not change what a launch
# does on the GPU, so recorded profiler counters stay valid across them.
KERNEL_FILES = ("gemm_kernel.cuh", "sm103_ptx.cuh", "gemm_launch.cuh", "relu_backward.cu")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_fp16_gemm_05_gb300", "csrc")
    for name in KERNEL_FILES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(workload)
    if not entry or entry.get("kernel_source_hash") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """Read-only NVML polling of the SM clock, the board power and the active
    clock-event (throttle) reasons, in a background thread about every
    millisecond, through the driver's own libnvidia-ml (ctypes; queries only,
    no setting is touched).  Each sample carries its host time, so a timed
    region -- host times taken right after the synchronisations that bracket
    it -- selects exactly the samples that fall inside it."""

    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, interval_s: float = 0.001):
        self.device_index = device_index
        self.interval_s = interval_s
        self.samples = []          # (host time, SM MHz, power W, reason bits)
        self.max_mhz = None
        self.error = None
        self._stop = False
        self._thread = None

    def _open(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        handle = ctypes.c_void_p()
        import torch
        uuid = str(torch.cuda.get_device_properties(self.device_index).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(handle)) != 0:
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.device_index), ctypes.byref(handle)) != 0:
                raise OSError("no NVML handle for the device")
        reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(handle, ctypes.c_int(1), ctypes.byref(mx)) == 0:   # NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
        return nv, handle, reasons_fn

    def _run(self, nv, handle, reasons_fn):
        import ctypes
        clk, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop:
            t = time.perf_counter()
            ok = nv.nvmlDeviceGetClockInfo(handle, ctypes.c_int(1), ctypes.byref(clk)) == 0
            pw = nv.nvmlDeviceGetPowerUsage(handle, ctypes.byref(mw)) == 0
            rr = reasons_fn(handle, ctypes.byref(rs)) == 0
            if ok:
                self.samples.append((t, float(clk.value), mw.value / 1000.0 if pw else float("nan"),
                                     int(rs.value) if rr else 0))
            time.sleep(self.interval_s)

    def start(self):
        import threading
        try:
            nv, handle, reasons_fn = self._open()
        except (OSError, AttributeError) as e:
            self.error = f"NVML unavailable: {e}"
            return self
        self._thread = threading.Thread(target=self._run, args=(nv, handle, reasons_fn), daemon=True)
        self._thread.start()
        time.sleep(0.05)
        return self

    def stop(self):
        self._stop = True
        if self._thread is not None:
            self._thread.join(timeout=5)

    def region(self, t0: float, t1: float, ms: float | None = None) -> dict:
        """Summary of the samples taken between host times t0 and t1."""
        if self.error:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [self.error], "samples": 0}
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        out = {"samples": len(inside), "sm_max_mhz": self.max_mhz, "source": "NVML, read-only, ~1 ms polling"}
        if not inside:
            out.update({"sm_mhz": None, "reasons": ["no sample inside the region"]})
            return out
        mhz = statistics.median(x[1] for x in inside)
        bits = 0
        for x in inside:
            bits |= x[3]
        powers = [x[2] for x in inside if x[2] == x[2]]
        out.update({"sm_mhz": mhz, "sm_mhz_min": min(x[1] for x in inside),
                    "power_w_max": max(powers) if powers else None,
                    "reasons": sorted(name for bit, name in self.REASON_BITS.items() if bits & bit)})
        if ms is not None:
            out["ms_x_median_mhz"] = ms * mhz   # clock-normalised duration (kilocycles at the median clock)
        return out


def oracle_cpu_baseline(A, B, relu: bool, budget_s: float, workload_name: str, M: int):
    """Times the CPU oracle on a bounded sample of full output rows."""
    import oracle
    N = B.shape[1]
    K = A.shape[1]
    # Probe with two rows per thread so that every core is busy, as in the run.
    rows_probe = max(1, min(M, 2 * oracle.num_threads()))
    _, t_probe = oracle.time_rows(A, B, relu, list(range(rows_probe)))
    per_row = max(t_probe / rows_probe, 1e-6)
    n_rows = int(max(1, min(M, budget_s / per_row)))
    step = max(1, M // n_rows)
    rows = list(range(0, M, step))[:n_rows]
    _, secs = oracle.time_rows(A, B, relu, rows)
    flops = 2.0 * len(rows) * N * K
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{len(rows)} of {M} output rows (all {N} columns, full K={K}) of {workload_name}, "
                      f"{secs:.1f} s"}, secs


VALUES_LABEL = {"normal_scaled": "N(0,1)/sqrt(K) fp16", "normal": "N(0,1) fp16", "integer": "integers -4..4 fp16"}


def workload_config(w) -> dict:
    """The `config` of the JSON line: the workload only, identical in both arms."""
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "relu": w.relu,
            "values": VALUES_LABEL.get(w.values, w.values), "seed": w.seed}


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from dense_fp16_gemm_05_gb300.inputs import WORKLOADS, draw_workload
    w = WORKLOADS[args.workload]
    A, B = draw_workload(w)
    # each step: a bounded sample of output rows, sized so the run ends within minutes
    probe_rows = list(range(min(2 * oracle.num_threads(), w.M)))
    _, t_probe = oracle.time_rows(A, B, w.relu, probe_rows)
    per_row = max(t_probe / len(probe_rows), 1e-6)
    per_step_budget = max(0.5, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    n_rows = int(max(1, min(w.M, per_step_budget / per_row)))
    rng_rows = [(i * 7919) % w.M for i in range(n_rows)]
    for _ in range(args.warmup):
        oracle.time_rows(A, B, w.relu, rng_rows)
    total = 0.0
    for _ in range(args.steps):
        _, s = oracle.time_rows(A, B, w.relu, rng_rows)
        total += s
    flops = 2.0 * n_rows * w.N * w.K * args.steps
    value = flops / total / 1e12
    cores = oracle.num_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "gpu_launches": 0,
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n_rows} of {w.M} output rows per step (all {w.N} columns, full K)",
                         "sample_rows_per_step": n_rows},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm

def time_device(g, A, B, C, relu, config, steps, warmup, stream, barrier=None):
    """Returns (total_ms over the timed steps, list of per-launch ms, host
    time right after the synchronisation before the steps, host time right
    after the one after them)."""
    import torch
    for _ in range(warmup):
        g.gemm_f16(A, B, C, relu=relu, stream=stream, config=config)
    (barrier or torch.cuda.synchronize)()
    h0 = time.perf_counter()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        starts[i].record(stream)
        g.gemm_f16(A, B, C, relu=relu, stream=stream, config=config)
        ends[i].record(stream)
    t1.record(stream)
    (barrier or torch.cuda.synchronize)()
    h1 = time.perf_counter()
    return t0.elapsed_time(t1), [s.elapsed_time(e) for s, e in zip(starts, ends)], h0, h1


SWEEP_WORKLOADS = ("int_64", "relu_ragged_1000", "relu_1024", "sweep_512", "sweep_1024", "sweep_2048",
                   "sweep_4096", "sweep_8192", "sweep_16384")


def run_sweep(g, dev, stream, peak, theoretical, sampler):
    """Every square configuration of the benchmark description, each in the
    automatic kernel configuration, timed two ways: single launches with L2
    flushed before each (where the operands fit in L2; median of the launches,
    all enqueued back to back), and back-to-back launches replayed from a CUDA
    graph (warm L2; the per-launch GPU time a chain of GEMMs sees)."""
    import torch
    from dense_fp16_gemm_05_gb300.inputs import WORKLOADS, draw_on_device, draw_workload
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 1000 * 1000))
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    out = []
    for name in SWEEP_WORKLOADS:
        w = WORKLOADS[name]
        if w.M * w.K <= 4096 * 4096:
            A, B = (t.to(dev) for t in draw_workload(w))
            drawn = "host generator (the parity tests' inputs)"
        else:
            A, B = draw_on_device(w.M, w.N, w.K, w.values, w.seed, dev)
            drawn = "seeded device generator (same distribution)"
        C = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
        cfg = g.auto_config(w.M, w.N, w.K)
        op_bytes = 2 * (w.M * w.K + w.K * w.N + w.M * w.N)
        fits = op_bytes < l2

        def call():
            g.gemm_f16(A, B, C, relu=w.relu, stream=stream)

        for _ in range(3):
            call()
        torch.cuda.synchronize()
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_ev.record(stream)
        call()
        e_ev.record(stream)
        e_ev.synchronize()
        one = max(s_ev.elapsed_time(e_ev), 1e-3)
        reps = int(min(50, max(7, 40.0 / one)))
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        h0 = time.perf_counter()
        for a_ev, b_ev in evs:
            if fits:
                flush.zero_()
            a_ev.record(stream)
            call()
            b_ev.record(stream)
        torch.cuda.synchronize()
        h1 = time.perf_counter()
        ms = statistics.median(a.elapsed_time(b) for a, b in evs)
        # back to back from a CUDA graph
        per_graph = int(min(200, max(1, 10.0 / one)))
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(torch.cuda.current_stream(dev))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for _ in range(per_graph):
                g.gemm_f16(A, B, C, relu=w.relu)
        replays = int(min(500, max(3, 30.0 / (one * per_graph))))
        graph.replay()
        torch.cuda.synchronize()
        s_ev.record()
        for _ in range(replays):
            graph.replay()
        e_ev.record()
        e_ev.synchronize()
        ms_graph = s_ev.elapsed_time(e_ev) / (replays * per_graph)
        del graph
        st = g.check(stream)
        if st != g.GEMM_OK:
            raise RuntimeError(f"{name}: device status {st}: {g.strerror(st)}")
        tf = w.flops / (ms * 1e-3) / 1e12
        tf_graph = w.flops / (ms_graph * 1e-3) / 1e12
        clk = sampler.region(h0, h1)
        out.append({"workload": name, "M": w.M, "N": w.N, "K": w.K, "relu": w.relu,
                    "values": VALUES_LABEL.get(w.values, w.values), "seed": w.seed, "inputs": drawn,
                    "kernel_config": g.config_label(cfg), "ms": ms, "TFLOP_s": tf,
                    "frac_of_measured_peak": tf / peak, "frac_of_theoretical_peak": tf / theoretical,
                    "l2": ("L2 flushed (a 2x-L2 buffer written) before each launch; median of launches"
                           if fits else "operands larger than L2, no flush; median of launches"),
                    "launches": reps, "sm_mhz": clk.get("sm_mhz"), "clock_samples": clk.get("samples"),
                    "graph_replay": {"us_per_launch": ms_graph * 1e3, "TFLOP_s": tf_graph,
                                     "frac_of_measured_peak": tf_graph / peak,
                                     "launches": replays * per_graph,
                                     "l2": "warm: back-to-back launches replayed from a CUDA graph"}})
        del A, B, C
    del flush
    torch.cuda.empty_cache()
    return out


def run_sustained(g, A, B, C, w, config, stream, sampler, seconds, peaks, peak_src, theoretical):
    """The headline workload back to back for `seconds` (the power-capped
    regime of a long run), with the clock samples taken inside the loop."""
    import torch
    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s_ev.record(stream)
    for _ in range(5):
        g.gemm_f16(A, B, C, relu=w.relu, stream=stream, config=config)
    e_ev.record(stream)
    e_ev.synchronize()
    one = s_ev.elapsed_time(e_ev) / 5
    n = int(max(10, seconds * 1e3 / one))
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    s_ev.record(stream)
    for _ in range(n):
        g.gemm_f16(A, B, C, relu=w.relu, stream=stream, config=config)
    e_ev.record(stream)
    torch.cuda.synchronize()
    h1 = time.perf_counter()
    ms = s_ev.elapsed_time(e_ev)
    st = g.check(stream)
    if st != g.GEMM_OK:
        raise RuntimeError(f"sustained loop: device status {st}: {g.strerror(st)}")
    tf = n * w.flops / (ms * 1e-3) / 1e12
    sus = peaks.get("bf16_tflops_sustained")
    return {"workload": w.name, "kernel_config": g.config_label(config), "launches": n, "seconds": ms / 1e3,
            "TFLOP_s": tf, "frac_of_theoretical_peak": tf / theoretical,
            "frac_of_measured_sustained_peak": tf / sus if sus else None, "peak_sustained": sus,
            "peak_source": f"{peak_src} bf16 matmul, back to back for seconds (fp16 has the same tensor rate)",
            "clocks": sampler.region(h0, h1, ms / n)}


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from dense_fp16_gemm_05_gb300 import gemm_f16 as g
    from dense_fp16_gemm_05_gb300.inputs import WORKLOADS, draw_workload
    g.lib()   # fails loudly if the CUDA library is missing

    w = WORKLOADS[args.workload]
    A_cpu, B_cpu = draw_workload(w)
    A = A_cpu.to(dev)
    B = B_cpu.to(dev)
    C = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
    stream = torch.cuda.current_stream(dev)
    config = args.config if args.config else g.auto_config(w.M, w.N, w.K)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()


    # ---- device-resident timing
    sampler = ClockSampler(local).start()
    total_ms, per_launch, h0, h1 = time_device(g, A, B, C, w.relu, config, args.steps, args.warmup, stream,
                                               barrier)
    clocks = sampler.region(h0, h1, total_ms / args.steps)
    st = g.check(stream)
    if st != g.GEMM_OK:
        raise RuntimeError(f"device status {st}: {g.strerror(st)}")
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(w.flops, args.steps, world, total_ms)

    avg_launch_ms = statistics.mean(per_launch)
    achieved = w.flops / (avg_launch_ms * 1e-3) / 1e12
    peaks, peak_src = measured_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    theoretical = sm_count * TENSOR_FLOP_PER_CLK_PER_SM * sm_max * 1e6 / 1e12

    # ---- secondary size of the metric: 4096^3 without ReLU
    secondary = None
    if args.workload == "relu_8192" and not args.no_secondary:
        w2 = WORKLOADS["plain_4096"]
        A2c, B2c = draw_workload(w2)
        A2, B2 = A2c.to(dev), B2c.to(dev)
        C2 = torch.empty((w2.M, w2.N), dtype=torch.float16, device=dev)
        cfg2 = args.config if args.config else g.auto_config(w2.M, w2.N, w2.K)
        # 96 MiB of inputs + 32 MiB output fit in L2: flush between launches
        flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
        for _ in range(3):
            g.gemm_f16(A2, B2, C2, relu=False, stream=stream, config=cfg2)
        # Everything is enqueued back to back (flush, event, GEMM, event) and
        # synchronised once, so host-side call overhead stays out of the timing.
        reps2 = max(5, min(args.steps, 50))
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps2)]
        for s_ev, e_ev in evs:
            flush.zero_()
            s_ev.record(stream)
            g.gemm_f16(A2, B2, C2, relu=False, stream=stream, config=cfg2)
            e_ev.record(stream)
        torch.cuda.synchronize()
        ms2 = statistics.median(s_ev.elapsed_time(e_ev) for s_ev, e_ev in evs)
        tf2 = w2.flops / (ms2 * 1e-3) / 1e12
        secondary = {"workload": w2.name, "M": w2.M, "N": w2.N, "K": w2.K, "relu": False,
                     "TFLOP_s": tf2, "ms": ms2, "frac_of_measured_peak": tf2 / peak,
                     "frac_of_theoretical_peak": tf2 / theoretical, "kernel_config": g.config_label(cfg2),
                     "l2": "256 MiB buffer written between launches (L2 flush); median of launches"}
        del A2, B2, C2, flush

    # ---- backward pair of the same workload (training use): the ReLU gradient
    # mask, dA = dZ @ B^T (NT layout) and dB = A^T @ dZ (TN layout)
    backward = None
    if not args.no_secondary:
        dC = torch.empty_like(C).normal_()
        dZ = torch.empty_like(C)
        dA = torch.empty_like(A)
        dB = torch.empty_like(B)
        hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))

        def timed(fn, reps):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s_ev.record(stream)
            for _ in range(reps):
                fn()
            e_ev.record(stream)
            e_ev.synchronize()
            return s_ev.elapsed_time(e_ev) / reps

        reps_b = args.steps   # as many launches as the forward loop (same power-capped regime)
        ms_mask = timed(lambda: g.relu_backward(dC, C, dZ, stream=stream), reps_b)
        ms_da = timed(lambda: g.gemm_f16_t(dZ, B, dA, transb=True, relu=False, stream=stream), reps_b)
        ms_db = timed(lambda: g.gemm_f16_t(A, dZ, dB, transa=True, relu=False, stream=stream), reps_b)
        mask_bytes = 3 * C.numel() * 2
        backward = {
            "relu_backward": {"ms": ms_mask, "GB_s": mask_bytes / (ms_mask * 1e-3) / 1e9,
                              "frac_of_measured_hbm": mask_bytes / (ms_mask * 1e-3) / 1e9 / hbm,
                              "bytes": mask_bytes, "bound": "hbm"},
            "dA_NT": {"ms": ms_da, "TFLOP_s": w.flops / (ms_da * 1e-3) / 1e12,
                      "kernel_config": g.config_label(g.auto_config(w.M, w.K, w.N))},
            "dB_TN": {"ms": ms_db, "TFLOP_s": w.flops / (ms_db * 1e-3) / 1e12,
                      "kernel_config": g.config_label(g.auto_config(w.K, w.N, w.M))},
            "note": "back-to-back launches on resident 8192^3 operands (larger than L2), as many as the timed forward steps",
        }
        del dC, dZ, dA, dB

    # ---- FP8 block-scaled GEMM (the next-row extension) at the same size:
    # E4M3 operands quantized per 128-blocks, fp32 scales, fp16 output
    fp8 = fp8_e8m0 = None
    if not args.no_secondary:
        from dense_fp16_gemm_05_gb300.inputs import FP8_WORKLOADS, draw_fp8_block_scaled
        w8 = FP8_WORKLOADS["fp8_8192"]
        A8c, SA8c, W8c, SW8c = draw_fp8_block_scaled(w8.M, w8.N, w8.K, w8.values, w8.seed)
        A8, SA8, W8, SW8 = A8c.to(dev), SA8c.to(dev), W8c.to(dev), SW8c.to(dev)
        C8 = torch.empty((w8.M, w8.N), dtype=torch.float16, device=dev)
        reps8 = args.steps
        for _ in range(3):
            g.gemm_fp8_block_scaled(A8, SA8, W8, SW8, C=C8, relu=w8.relu, stream=stream)
        torch.cuda.synchronize()
        s8, e8 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s8.record(stream)
        for _ in range(reps8):
            g.gemm_fp8_block_scaled(A8, SA8, W8, SW8, C=C8, relu=w8.relu, stream=stream)
        e8.record(stream)
        e8.synchronize()
        ms8 = s8.elapsed_time(e8) / reps8
        if g.check(stream) != g.GEMM_OK:
            raise SystemExit("FP8 kernel reported a device error")
        tf8 = w8.flops / (ms8 * 1e-3) / 1e12
        peak8 = peak * FP8_PER_BF16
        fp8 = {"workload": w8.name, "M": w8.M, "N": w8.N, "K": w8.K, "relu": w8.relu, "ms": ms8, "TFLOP_s": tf8,
               "roofline": {"bound": "tensor", "achieved": tf8, "peak": peak8, "unit": "TFLOP/s", "frac": tf8 / peak8,
                            "peak_source": f"{peak_src} bf16 matmul burst x {FP8_PER_BF16} (nominal fp8 / bf16 dense ratio)"},
               "values": "N(0,1) quantized per 128-block to E4M3, fp32 scales", "launches": reps8,
               "note": "back-to-back launches on resident operands"}
        del A8, SA8, W8, SW8
        # the same with power-of-two scales (E8M0 bytes), applied inside the MMA
        from dense_fp16_gemm_05_gb300.inputs import draw_mxfp8_block_scaled
        A8, SA8, W8, SW8 = (t.to(dev) for t in draw_mxfp8_block_scaled(w8.M, w8.N, w8.K, "normal", w8.seed))
        for _ in range(3):
            g.gemm_mxfp8_block_scaled(A8, SA8, W8, SW8, C=C8, relu=w8.relu, stream=stream)
        torch.cuda.synchronize()
        s8.record(stream)
        for _ in range(reps8):
            g.gemm_mxfp8_block_scaled(A8, SA8, W8, SW8, C=C8, relu=w8.relu, stream=stream)
        e8.record(stream)
        e8.synchronize()
        msx = s8.elapsed_time(e8) / reps8
        if g.check(stream) != g.GEMM_OK:
            raise SystemExit("FP8 (power-of-two scales) kernel reported a device error")
        tfx = w8.flops / (msx * 1e-3) / 1e12
        fp8_e8m0 = {
            "workload": w8.name, "M": w8.M, "N": w8.N, "K": w8.K, "relu": w8.relu, "ms": msx, "TFLOP_s": tfx,
            "roofline": {"bound": "tensor", "achieved": tfx, "peak": peak8, "unit": "TFLOP/s", "frac": tfx / peak8,
                         "peak_source": fp8["roofline"]["peak_source"]},
            "values": "N(0,1) quantized per 128-block to E4M3, scales rounded up to powers of two (E8M0 bytes)",
            "entry": "gemm_mxfp8_block_scaled", "launches": reps8,
            "note": "the same method with power-of-two scales, applied inside the tensor core"}
        fp8["power_of_two_scales"] = {"ms": msx, "TFLOP_s": tfx, "roofline": fp8_e8m0["roofline"],
                                      "see": "fp8_block_scaled_e8m0"}
        del A8, SA8, W8, SW8, C8

    # ---- attention forward (the next-row extension): 4096 tokens, batch 4,
    # 32 heads of dim 128 and 64 heads of dim 64, fp16, non-causal and causal
    attention = None
    if not args.no_secondary:
        from dense_fp16_gemm_05_gb300.inputs import ATTN_WORKLOADS, draw_attention_workload
        attention = {}
        for name in ("attn_4096_d128", "attn_4096_d128_causal", "attn_4096_d64", "attn_4096_d64_causal"):
            wa = ATTN_WORKLOADS[name]
            Qa, Ka, Va = (t.to(dev) for t in draw_attention_workload(wa))
            Oa = torch.empty_like(Qa)
            # causal: the work queue, zero before the first launch; each launch
            # leaves it zero, so one serves all launches on this stream
            with torch.cuda.stream(stream):
                qa = torch.zeros(2, dtype=torch.int32, device=dev)
            for _ in range(3):
                g.attention_fwd(Qa, Ka, Va, O=Oa, causal=wa.causal, stream=stream, queue=qa)
            torch.cuda.synchronize()
            sa, ea = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps_a = max(10, args.steps // 2)
            sa.record(stream)
            for _ in range(reps_a):
                g.attention_fwd(Qa, Ka, Va, O=Oa, causal=wa.causal, stream=stream, queue=qa)
            ea.record(stream)
            ea.synchronize()
            msa = sa.elapsed_time(ea) / reps_a
            if g.check(stream) != g.GEMM_OK:
                raise SystemExit("attention kernel reported a device error")
            tfa = wa.flops / (msa * 1e-3) / 1e12
            attention[name] = {"batch": wa.batch, "heads": wa.heads, "seq": wa.seq, "dim": wa.dim,
                               "causal": wa.causal, "ms": msa, "TFLOP_s": tfa,
                               "roofline": {"bound": "tensor", "achieved": tfa, "peak": peak, "unit": "TFLOP/s",
                                            "frac": tfa / peak,
                                            "peak_source": f"{peak_src} bf16 matmul burst (fp16 rate)"},
                               "flops_counted": "4 batch heads seq^2 dim (halved when causal)", "launches": reps_a,
                               "schedule": "work queue" if wa.causal else "fixed shares"}
            del Qa, Ka, Va, Oa, qa

    # ---- every configuration of the benchmark description (the shape sweep
    # and the named sizes) and a seconds-long loop of the headline workload
    sweep = sustained = None
    if not args.no_secondary and world == 1:
        sweep = run_sweep(g, dev, stream, peak, theoretical, sampler)
        sustained = run_sustained(g, A, B, C, w, config, stream, sampler, args.sustained_s, peaks, peak_src,
                                  theoretical)

    # ---- end to end through the host-buffer C call.  Steps alternate between
    # two streams, each with its own device buffers and host result buffer (a
    # caller streaming independent problems): a step's uploads start as soon
    # as the previous step's uploads are done, while its GEMMs and downloads
    # finish.  Every step copies its inputs up and its result down.
    A_h = A_cpu.pin_memory()
    B_h = B_cpu.pin_memory()
    stream2 = torch.cuda.Stream(device=dev)
    e2e_sets = [(stream, A, B, C, torch.empty((w.M, w.N), dtype=torch.float16).pin_memory()),
                (stream2, torch.empty_like(A), torch.empty_like(B), torch.empty_like(C),
                 torch.empty((w.M, w.N), dtype=torch.float16).pin_memory())]
    C_h = e2e_sets[0][4]
    e2e_steps = max(3, min(args.steps, 30))
    for i in range(2):
        st_, Ad_, Bd_, Cd_, Ch_ = e2e_sets[i]
        g.gemm_f16_from_host(A_h, B_h, Ch_, Ad_, Bd_, Cd_, relu=w.relu, stream=st_)
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2 = torch.cuda.Event()
    e0.record(stream)
    stream2.wait_event(e0)
    for i in range(e2e_steps):
        st_, Ad_, Bd_, Cd_, Ch_ = e2e_sets[i % 2]
        g.gemm_f16_from_host(A_h, B_h, Ch_, Ad_, Bd_, Cd_, relu=w.relu, stream=st_)
    e2.record(stream2)
    stream.wait_event(e2)
    e1.record(stream)
    barrier()
    for st_ in (stream, stream2):
        if g.check(stream=st_) != g.GEMM_OK:
            raise SystemExit("end-to-end call reported a device error")
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = whole_job_rate(w.flops, e2e_steps, world, e2e_ms)

    sampler.stop()
    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_baseline, _ = oracle_cpu_baseline(A_cpu, B_cpu, w.relu, args.cpu_budget, w.name, w.M)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": workload_config(w),
            "kernel": {"config": g.config_label(config), "accumulate": "f32",
                       "l2": "inputs 384 MiB > 126 MB L2, no flush",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "frac_of_theoretical_peak": value / world / theoretical,
            "theoretical_peak_tflops": theoretical,
            "theoretical_peak_basis": f"{sm_count} SMs x {TENSOR_FLOP_PER_CLK_PER_SM} FLOP/clk x {sm_max:.0f} MHz",
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": recorded_traffic(w.name),
                         "peak_source": f"{peak_src} bf16 matmul burst (fp16 has the same tensor rate)",
                         "avg_launch_ms": avg_launch_ms},
            "e2e": {"value": e2e_value, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": int(A_h.numel() * 2 + B_h.numel() * 2),
                    "d2h_bytes_per_step": int(C_h.numel() * 2), "steps": e2e_steps,
                    "pipelining": "steps alternate between two streams and two buffer sets"},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu_baseline,
        }
        if secondary is not None:
            line["secondary"] = secondary
        if backward is not None:
            line["backward"] = backward
        if fp8 is not None:
            line["fp8_block_scaled"] = fp8
        if fp8_e8m0 is not None:
            line["fp8_block_scaled_e8m0"] = fp8_e8m0
        if attention is not None:
            line["attention_fwd"] = attention
        if sweep is not None:
            line["sweep"] = sweep
        if sustained is not None:
            line["sustained"] = sustained
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="relu_8192")
    p.add_argument("--config", type=int, default=0, help="kernel configuration id (0 = automatic)")
    p.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-secondary", action="store_true")
    p.add_argument("--sustained-s", type=float, default=2.5, help="seconds of the sustained headline loop")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
