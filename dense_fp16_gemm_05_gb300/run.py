"""Runs one named workload through the C ABI a few times and prints the timings.

    python -m dense_fp16_gemm_05_gb300.run --workload relu_8192 --reps 4 [--config ID]

A minimal program around the library (no oracle, no other kernels besides the
input upload), suited as the target of a profiler capture: every GPU kernel it
launches after the upload is the GEMM.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import gemm_f16 as g
from .inputs import WORKLOADS, Workload, draw_workload


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--workload", default="relu_8192", help=f"one of {sorted(WORKLOADS)} or MxNxK")
    p.add_argument("--reps", type=int, default=4)
    p.add_argument("--config", type=int, default=0)
    p.add_argument("--relu", type=int, default=None, help="override the workload's ReLU flag")
    args = p.parse_args(argv)
    if args.workload in WORKLOADS:
        w = WORKLOADS[args.workload]
    else:
        M, N, K = (int(x) for x in args.workload.lower().split("x"))
        w = Workload(args.workload, M, N, K, True, "normal_scaled", 0)
    relu = w.relu if args.relu is None else bool(args.relu)
    dev = torch.device("cuda", 0)
    A_cpu, B_cpu = draw_workload(w)
    A, B = A_cpu.to(dev), B_cpu.to(dev)
    C = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
    cfg = args.config or g.auto_config(w.M, w.N, w.K)
    times = []
    for _ in range(args.reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        g.gemm_f16(A, B, C, relu=relu, config=cfg)
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    st = g.check()
    if st != g.GEMM_OK:
        raise SystemExit(f"device status {st}: {g.strerror(st)}")
    best = min(times)
    print(json.dumps({"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "relu": relu,
                      "config": g.config_name(cfg), "ms": times,
                      "best_tflops": w.flops / (best * 1e-3) / 1e12}))


if __name__ == "__main__":
    main()
