"""Times every synthetic workload through the library and writes one JSON
record per workload (appended to --out; workloads already in the file are
skipped, so an interrupted sweep resumes) plus a Markdown table.

Per workload: 10 warm-up launches, then at least 50 timed launches (200 when
one takes under 100 µs) in back-to-back CUDA-event pairs on one stream, L2 not
flushed between them (the operands of the larger workloads exceed the L2
anyway); the median and mean; the device time per launch with no host time
between launches (20 launches, or 3 of the long ones, captured in one CUDA
graph and replayed: for the small products the event pairs above measure the
Python call, not the kernel); one cold launch after writing a 256 MiB buffer;
and ``torch.matmul`` on the same operands as context (TF32 allowed for fp32).
The records also carry the plan, the GPU name, SM count, driver and the SM
clocks sampled during the timed launches.

    python -m dense_gemm_tensor_gb300.sweep --out sweep.jsonl --md sweep.md
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess

import torch

from . import build, gemm, inputs

PEAK_NOTE = "of the measured bf16 cuBLAS burst rate (x 1.1/2.25 for TF32)"


def _clock_sample(gpu: int) -> dict:
    try:
        out = subprocess.run(["nvidia-smi", f"--id={gpu}", "--query-gpu=clocks.sm,clocks.max.sm,driver_version",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10).stdout
        sm, smax, drv = [x.strip() for x in out.strip().split(",")]
        return {"sm_mhz": float(sm), "sm_max_mhz": float(smax), "driver": drv}
    except (OSError, ValueError, subprocess.SubprocessError):
        return {}


def _time(fn, iters: int) -> list[float]:
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for e0, e1 in evs:
        e0.record()
        fn()
        e1.record()
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) * 1e3 for e0, e1 in evs]  # µs


def _time_graph(fn, per_graph: int, replays: int = 10) -> float:
    """Device time per launch with no host time between launches: `per_graph`
    launches captured in one CUDA graph (on a stream warmed up first, so the
    library's scratch already exists), replayed `replays` times; µs."""
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            fn()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(per_graph):
            fn()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(replays):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (replays * per_graph)


def run_one(name: str, peaks: dict, gpu: int) -> dict:
    p = inputs.workload(name)
    A, B = p.a.cuda(), p.b.cuda()
    a = A[:, :p.K]
    b = B[:, :p.N] if p.layout == 0 else B[:, :p.K]
    C = torch.empty((p.M, p.N), dtype=A.dtype, device="cuda")
    fn = lambda: gemm.matmul(a, b, C, layout=p.layout)  # noqa: E731
    for _ in range(10):
        fn()
    torch.cuda.synchronize()
    probe = _time(fn, 5)
    iters = 200 if statistics.median(probe) < 100 else 50
    clk0 = _clock_sample(gpu)
    ts = _time(fn, iters)
    clk1 = _clock_sample(gpu)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    flush.zero_()
    cold = _time(fn, 1)[0]
    del flush
    plan = gemm.last_plan()
    flops = 2.0 * p.M * p.N * p.K
    med = statistics.median(ts)
    graph_us = _time_graph(fn, 20 if med < 1000 else 3)
    rec = {"workload": name, "dtype": p.dtype, "M": p.M, "N": p.N, "K": p.K, "layout": p.layout,
           "lda": p.lda, "ldb": p.ldb, "seeds": [1000 + inputs.WORKLOADS[name]["n"], 2000 + inputs.WORKLOADS[name]["n"]],
           "iters": iters, "median_us": round(med, 2), "mean_us": round(statistics.mean(ts), 2),
           "cold_us": round(cold, 2), "tflops": round(flops / (med * 1e-6) / 1e12, 1), "plan": plan,
           "graph_us": round(graph_us, 2), "graph_tflops": round(flops / (graph_us * 1e-6) / 1e12, 1)}
    peak = peaks.get("bf16_tflops")
    if peak:
        if p.dtype == "tf32":
            peak = peak * 1.1 / 2.25
        rec["frac_of_peak"] = round(rec["tflops"] / peak, 4)
    # torch.matmul on the same operands, as context
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        bt = b if p.layout == 0 else b.t()
        tfn = lambda: torch.matmul(a, bt, out=C)  # noqa: E731
        for _ in range(5):
            tfn()
        torch.cuda.synchronize()
        tt = statistics.median(_time(tfn, min(iters, 50)))
        rec["torch_matmul_us"] = round(tt, 2)
    except RuntimeError as ex:  # e.g. an out= layout torch does not take
        rec["torch_matmul_us"] = None
        rec["torch_note"] = str(ex).splitlines()[0][:120]
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    rec["sm_mhz"] = [clk0.get("sm_mhz"), clk1.get("sm_mhz")]
    del A, B, C, a, b
    torch.cuda.empty_cache()
    return rec


def markdown(recs: list[dict]) -> str:
    lines = ["| workload | dtype | M x N x K | B | plan (kernel, tile, segs) | median µs | mean µs | cold µs | TFLOP/s | "
             f"fraction {PEAK_NOTE} | in a CUDA graph µs | TFLOP/s in a graph | torch.matmul µs |",
             "|---|---|---|---|---|---|---|---|---|---|---|---|---|"]
    for r in recs:
        pl = r["plan"]
        kern = {1: "single", 2: "pair", 3: "pair on C^T", 4: "2 pairs"}.get(pl["kernel"], str(pl["kernel"]))
        lines.append(f"| {r['workload']} | {r['dtype']} | {r['M']}x{r['N']}x{r['K']} | {'K-major' if r['layout'] else 'row'} "
                     f"| {kern}, {pl['tile_n']}, {pl['tail_segs']} | {r['median_us']} | {r['mean_us']} | {r['cold_us']} "
                     f"| {r['tflops']} | {r.get('frac_of_peak', '')} | {r.get('graph_us', '')} | {r.get('graph_tflops', '')} "
                     f"| {r.get('torch_matmul_us', '')} |")
    return "\n".join(lines) + "\n"


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description="time every workload")
    ap.add_argument("--out", default="sweep.jsonl")
    ap.add_argument("--md", default=None)
    ap.add_argument("--workloads", default=",".join(inputs.WORKLOADS))
    args = ap.parse_args(argv)
    build.build()
    gemm.load()
    gpu = torch.cuda.current_device()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    peaks = {}
    try:
        with open(os.path.join(root, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    done = {}
    if os.path.exists(args.out):
        with open(args.out) as f:
            for line in f:
                if line.strip():
                    r = json.loads(line)
                    done[r["workload"]] = r
    props = torch.cuda.get_device_properties(gpu)
    for name in args.workloads.split(","):
        if name in done:
            continue
        rec = run_one(name, peaks, gpu)
        rec["gpu"] = props.name
        rec["sms"] = props.multi_processor_count
        rec["driver"] = _clock_sample(gpu).get("driver")
        with open(args.out, "a") as f:
            f.write(json.dumps(rec) + "\n")
        done[name] = rec
        print(json.dumps(rec), flush=True)
    if args.md:
        order = [n for n in args.workloads.split(",") if n in done]
        with open(args.md, "w") as f:
            f.write(markdown([done[n] for n in order]))


if __name__ == "__main__":
    main()
