"""Offline sweep for the automatic configuration choice.

    python -m dense_fp16_gemm_05_gb300.tune [--out PATH] [--rounds 3] [--quick]

Times every fixed configuration, with and without the tail split
(GEMM_F16_NO_SPLIT), and the cluster K split configuration at its rule-chosen
cluster size and at clusters of 2 and 4, on a grid of problem shapes (the
candidates of the automatic choice; none allocates memory), and writes the measured
throughputs as a C include (``csrc/gemm_f16_tuned.inc``) that the library
compiles in.  The tile GEMM lesson of the pages tunes its block sizes with a
JIT autotuner at run time ("Writing High-Performance Kernels in TileLang, from
GEMM to MLA", autotuning section); here the search is done once, offline, and
the run-time choice is a table lookup (see ``select_config`` in gemm_f16.cu).

Method: for each shape, every candidate runs ``rounds`` times in interleaved
order (so slow drift of the power-capped clock hits all candidates alike);
each round times about 150 ms of back-to-back launches on resident operands
with CUDA events (the sustained regime: short bursts run at a higher clock
than the power cap allows for long), replayed from a CUDA graph so that the
per-call host cost does not hide the kernels' differences on small problems,
and keeps the mean time per launch; a candidate's figure is the median over
rounds.  Needs one sm_103 GPU and the
built library.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import os
import statistics
import sys

import torch

from . import build as _build
from . import gemm_f16 as g

SQUARES = [512, 1024, 2048, 3072, 4096, 6144, 8192, 12288, 16384]
SIDES = [1024, 2048, 4096, 8192, 16384]
DEPTHS = [1024, 4096, 16384]
DEFAULT_OUT = os.path.join(_build.CSRC, "gemm_f16_tuned.inc")


def grid_shapes(quick: bool = False) -> list[tuple[int, int, int]]:
    if quick:
        return [(n, n, n) for n in (1024, 4096, 8192)]
    shapes = {(n, n, n) for n in SQUARES}
    shapes.update((m, n, k) for m in SIDES for n in SIDES for k in DEPTHS)
    return sorted(shapes)


def candidates() -> list[int]:
    """Every schedule the automatic choice may take: each configuration with
    and without the tail split, and the cluster K split at its rule-chosen
    size and at clusters of 2 and 4.  None of them allocates memory: the
    workspace K split stays an explicit request (gemm_f16_ex with the K-split
    bits), so gemm_f16 itself never allocates."""
    out = []
    for cfg in range(1, g.num_configs() + 1):
        if g.config_cluster_k(cfg):
            out += [cfg, cfg | g.ksplit(2), cfg | g.ksplit(4)]
        else:
            out += [cfg, cfg | g.GEMM_F16_NO_SPLIT]
    return out


def time_candidate(A, B, C, cfg: int, min_ms: float) -> float:
    """Mean ms per launch over back-to-back launches on resident operands,
    about ``min_ms`` of them: long enough for the power-capped clock to settle
    as it does in a sustained run.  The launches are captured once in a CUDA
    graph (up to 200 of them, every stream-ordered workspace allocation
    included) and the graph is replayed, so no host work sits between two
    launches: on small problems the per-call host cost would otherwise set
    the pace for every candidate alike and hide the kernels' differences."""
    def run():
        g.gemm_f16(A, B, C, relu=True, config=cfg)

    for _ in range(2):
        run()                      # the first calls also do the library's per-device set-up
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    run()
    e.record()
    e.synchronize()
    one = max(s.elapsed_time(e), 1e-3)
    per_graph = int(min(200, max(1, 20.0 / one)))
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(per_graph):
            run()
    replays = int(min(20000, max(2, min_ms / (one * per_graph))))
    graph.replay()
    torch.cuda.synchronize()
    s.record()
    for _ in range(replays):
        graph.replay()
    e.record()
    e.synchronize()
    st = g.check()
    if st != g.GEMM_OK:
        raise RuntimeError(f"config {cfg:#x}: device status {st} ({g.strerror(st)})")
    del graph
    return s.elapsed_time(e) / (replays * per_graph)


def sweep(shapes, rounds: int, min_ms: float, log=sys.stderr) -> list[dict]:
    dev = torch.device("cuda", 0)
    cands = candidates()
    rows = []
    for (M, N, K) in shapes:
        gen = torch.Generator(device=dev).manual_seed(M * 7 + N * 3 + K)
        A = (torch.randn(M, K, device=dev, generator=gen) / K ** 0.5).half()
        B = torch.randn(K, N, device=dev, generator=gen).half()
        C = torch.empty(M, N, device=dev, dtype=torch.float16)
        times = {c: [] for c in cands}
        for _ in range(rounds):
            for c in cands:
                times[c].append(time_candidate(A, B, C, c, min_ms))
        flops = 2.0 * M * N * K
        tf = {c: flops / (statistics.median(times[c]) * 1e-3) / 1e12 for c in cands}
        best = max(tf, key=tf.get)
        rows.append({"shape": (M, N, K), "tflops": tf})
        print(f"{M:6d} {N:6d} {K:6d}  best {g.config_label(best):28s} {tf[best]:7.1f} TF/s", file=log, flush=True)
        del A, B, C
        torch.cuda.empty_cache()
    return rows


def kernel_hash() -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(_build.CSRC)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(_build.CSRC, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def write_include(rows, path: str, rounds: int, min_ms: float):
    cands = candidates()
    props = torch.cuda.get_device_properties(0)
    lines = [
        "// Generated by `python -m dense_fp16_gemm_05_gb300.tune`; do not edit by hand.",
        f"// Device: {props.name}, {props.multi_processor_count} SMs; {datetime.date.today().isoformat()};",
        f"// kernel sources {kernel_hash()}; {rounds} interleaved rounds per shape, median;",
        f"// about {min_ms:.0f} ms of back-to-back launches (CUDA graph replays) per candidate and round.",
        "// Each row: M, N, K, then the measured TFLOP/s of every candidate in",
        "// kTunedCandidates order (ReLU on, N(0,1) operands, back-to-back launches).",
        f"#define GEMM_F16_TUNED_CANDIDATES {len(cands)}",
        "static const int kTunedCandidates[GEMM_F16_TUNED_CANDIDATES] = {" +
        ", ".join(f"0x{c:03x}" for c in cands) + "};",
        f"#define GEMM_F16_TUNED_ROWS {len(rows)}",
        "static const struct TunedRow { int M, N, K; float tflops[GEMM_F16_TUNED_CANDIDATES]; } "
        "kTunedRows[GEMM_F16_TUNED_ROWS] = {",
    ]
    for r in rows:
        M, N, K = r["shape"]
        vals = ", ".join(f"{r['tflops'][c]:.1f}f" for c in cands)
        lines.append(f"    {{{M}, {N}, {K}, {{{vals}}}}},")
    lines.append("};")
    tmp = path + ".tmp"
    with open(tmp, "w") as f:
        f.write("\n".join(lines) + "\n")
    os.replace(tmp, path)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--out", default=DEFAULT_OUT)
    p.add_argument("--rounds", type=int, default=2)
    p.add_argument("--ms", type=float, default=150.0, help="timed milliseconds per candidate and round")
    p.add_argument("--quick", action="store_true", help="three square shapes only (a smoke run)")
    args = p.parse_args(argv)
    if not torch.cuda.is_available():
        raise SystemExit("the sweep needs a GPU")
    g.lib()
    rows = sweep(grid_shapes(args.quick), args.rounds, args.ms)
    write_include(rows, args.out, args.rounds, args.ms)
    print(f"wrote {len(rows)} shapes x {len(candidates())} candidates to {args.out}", file=sys.stderr)


if __name__ == "__main__":
    main()
