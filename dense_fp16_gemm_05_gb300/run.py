"""Runs one named workload through the C ABI a few times and prints the timings.

    python -m dense_fp16_gemm_05_gb300.run --workload relu_8192 --reps 4 [--config ID]
        [--op gemm|dA_nt|dB_tn|relu_backward|fp8|attn]

--op picks the kernel: the forward GEMM (default), the two backward GEMMs of
the workload (dA = dZ @ B^T in the NT layout, dB = A^T @ dZ in the TN layout)
or the ReLU-gradient mask over an (M,N) gradient; --op fp8 runs the FP8
block-scaled GEMM on the workload's sizes (E4M3 operands quantized per
128-block, fp32 scales), --op mxfp8 the same with power-of-two scales; --op attn runs the attention forward on an attention
workload (--workload attn_4096_d128, ...); causal attention takes work items
from one work queue made before the first launch (--attn-queue fixed: the
fixed shares instead).

A minimal program around the library (no oracle, no other kernels besides the
input upload), suited as the target of a profiler capture: every GPU kernel it
launches after the upload is the GEMM.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import gemm_f16 as g
from .inputs import (ATTN_WORKLOADS, WORKLOADS, Workload, draw_attention_workload, draw_fp8_block_scaled,
                     draw_mxfp8_block_scaled, draw_workload)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--workload", default="relu_8192", help=f"one of {sorted(WORKLOADS)} or MxNxK")
    p.add_argument("--reps", type=int, default=4)
    p.add_argument("--config", type=int, default=0)
    p.add_argument("--relu", type=int, default=None, help="override the workload's ReLU flag")
    p.add_argument("--op", default="gemm", choices=["gemm", "dA_nt", "dB_tn", "relu_backward", "fp8", "mxfp8", "attn"])
    p.add_argument("--attn-queue", default="reuse", choices=["reuse", "fixed"])
    args = p.parse_args(argv)
    if args.op == "attn":
        return run_attention(ATTN_WORKLOADS[args.workload], args.reps, torch.device("cuda", 0), args.attn_queue)
    if args.workload in WORKLOADS:
        w = WORKLOADS[args.workload]
    else:
        M, N, K = (int(x) for x in args.workload.lower().split("x"))
        w = Workload(args.workload, M, N, K, True, "normal_scaled", 0)
    relu = w.relu if args.relu is None else bool(args.relu)
    dev = torch.device("cuda", 0)
    if args.op in ("fp8", "mxfp8"):
        return run_fp8(w, relu, args.reps, dev, pow2=args.op == "mxfp8")
    A_cpu, B_cpu = draw_workload(w)
    A, B = A_cpu.to(dev), B_cpu.to(dev)
    C = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
    cfg = args.config or g.auto_config(w.M, w.N, w.K)
    dZ = dA = dB = None
    if args.op != "gemm":
        dZ = torch.empty((w.M, w.N), dtype=torch.float16, device=dev).normal_()
        g.gemm_f16(A, B, C, relu=True, config=cfg)
        dA = torch.empty_like(A) if args.op == "dA_nt" else None
        dB = torch.empty_like(B) if args.op == "dB_tn" else None

    def step():
        if args.op == "gemm":
            g.gemm_f16(A, B, C, relu=relu, config=cfg)
        elif args.op == "dA_nt":
            g.gemm_f16_t(dZ, B, dA, transb=True, relu=False, config=args.config)
        elif args.op == "dB_tn":
            g.gemm_f16_t(A, dZ, dB, transa=True, relu=False, config=args.config)
        else:
            g.relu_backward(dZ, C, dZ)

    times = []
    for _ in range(args.reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        step()
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    st = g.check()
    if st != g.GEMM_OK:
        raise SystemExit(f"device status {st}: {g.strerror(st)}")
    best = min(times)
    out = {"workload": w.name, "op": args.op, "M": w.M, "N": w.N, "K": w.K, "relu": relu,
           "config": g.config_label(cfg) if args.op == "gemm" else args.config, "ms": times}
    if args.op == "relu_backward":
        out["best_GBps"] = 3 * w.M * w.N * 2 / (best * 1e-3) / 1e9
    else:
        out["best_tflops"] = w.flops / (best * 1e-3) / 1e12
    print(json.dumps(out))


def run_fp8(w, relu, reps, dev, pow2=False):
    draw = draw_mxfp8_block_scaled if pow2 else draw_fp8_block_scaled
    fn = g.gemm_mxfp8_block_scaled if pow2 else g.gemm_fp8_block_scaled
    A8, SA, W8, SW = (t.to(dev) for t in draw(w.M, w.N, w.K, "normal", w.seed))
    C = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
    times = []
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn(A8, SA, W8, SW, C=C, relu=relu)
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    st = g.check()
    if st != g.GEMM_OK:
        raise SystemExit(f"device status {st}: {g.strerror(st)}")
    print(json.dumps({"workload": w.name, "op": "mxfp8" if pow2 else "fp8", "M": w.M, "N": w.N, "K": w.K, "relu": relu, "ms": times,
                      "best_tflops": w.flops / (min(times) * 1e-3) / 1e12}))


def run_attention(w, reps, dev, queue_mode="reuse"):
    Q, K, V = (t.to(dev) for t in draw_attention_workload(w))
    O = torch.empty_like(Q)
    # the kernel leaves the queue zero, so one serves every launch below
    queue = torch.zeros(2, dtype=torch.int32, device=dev) if queue_mode == "reuse" else False
    times = []
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        g.attention_fwd(Q, K, V, O=O, sm_scale=w.sm_scale, causal=w.causal, queue=queue)
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    st = g.check()
    if st != g.GEMM_OK:
        raise SystemExit(f"device status {st}: {g.strerror(st)}")
    print(json.dumps({"workload": w.name, "op": "attn", "causal": w.causal, "queue": queue_mode, "ms": times,
                      "best_tflops": w.flops / (min(times) * 1e-3) / 1e12}))


if __name__ == "__main__":
    main()
