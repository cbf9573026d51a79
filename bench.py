"""Benchmark of the dense GEMM at M = N = K = 4096 in TF32, FP16 and BF16.

One step is one pass of the whole path over one batch of synthetic input:
the three 4096^3 products (TF32 with fp32 operands uniform in [-1, 1);
FP16 and BF16 with N(0, 1) operands), each one launch of the library's
kernel through its C interface. ``value`` is TFLOP/s (2MNK per product)
over the timed steps with the operands resident in device memory; ``e2e``
is the same metric through the host-memory call (pinned host operands copied
in, C copied out, every step). ``--impl reference`` times the CPU oracle on
the same workload instead (a bounded slice of rows per step).

Launch: ``python bench.py [--gpus N] [--steps K] [--warmup W]``; for N > 1
under torchrun each rank runs an independent replica on its own GPU (the
product does not shard), and ``value`` is the total over ranks divided by the
slowest rank's time.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

M = N = K = 4096
DTYPES = ("tf32", "f16", "bf16")
WORKLOAD = {"tf32": "tf32_4096", "f16": "f16_4096", "bf16": "bf16_4096"}
FLOP_PER_PRODUCT = 2.0 * M * N * K
METRIC = "TFLOP/s at M=N=K=4096 (bf16, fp16, tf32) and % of GB300 dense tensor peak"
# Dense tensor-core rates relative to BF16 (nominal: TF32 1.1, FP16/BF16 2.25 PFLOP/s)
NOMINAL_RATIO = {"bf16": 1.0, "f16": 1.0, "tf32": 1.1 / 2.25}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def peak_for(dtype: str, peaks: dict, sustained: bool = True) -> float:
    """Dense tensor peak for ``dtype`` in TFLOP/s: the measured BF16 figure times
    the nominal ratio. The sustained figure (a seconds-long loop under the power
    cap) is the one for kernels timed inside the long back-to-back loop here;
    the burst figure is for a kernel timed alone."""
    burst = peaks["bf16_tflops"]
    base = peaks.get("bf16_tflops_sustained", burst) if sustained else burst
    return base * NOMINAL_RATIO[dtype]


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over ranks (identity for one process)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while a region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.raw = out
        else:
            self.raw = ""

    def summary(self) -> dict:
        rows = []
        for line in self.raw.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


def make_inputs():
    from dense_gemm_tensor_gb300 import inputs
    return {dt: inputs.workload(WORKLOAD[dt]) for dt in DTYPES}


def run_ours(args, world, rank, local):
    import torch
    from dense_gemm_tensor_gb300 import build as libbuild
    from dense_gemm_tensor_gb300 import gemm

    libbuild.build()
    gemm.load()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(dev)
    probs = make_inputs()
    A = {dt: probs[dt].a.to(dev) for dt in DTYPES}
    B = {dt: probs[dt].b.to(dev) for dt in DTYPES}
    C = {dt: torch.empty((M, N), dtype=A[dt].dtype, device=dev) for dt in DTYPES}

    def step(ev=None):
        for i, dt in enumerate(DTYPES):
            if ev is not None:
                ev[dt][0].record(stream)
            gemm.matmul(A[dt], B[dt], C[dt], stream=stream)
            if ev is not None:
                ev[dt][1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    # the launch plan of each product (the same every step: it depends only on shape and alignment)
    plans = {}
    with torch.cuda.stream(stream):
        for dt in DTYPES:
            gemm.matmul(A[dt], B[dt], C[dt], stream=stream)
            plans[dt] = gemm.last_plan()
    stream.synchronize()
    if gemm.device_status(stream) != 0:
        raise RuntimeError("device status word set during warm-up")

    # per-kernel events for every timed step (same stream as the kernels)
    evs = [{dt: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for dt in DTYPES}
           for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = gemm.launch_count()
    with ClockSampler(local) as clocks:
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for k in range(args.steps):
                step(evs[k])
            t1.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
    launches = gemm.launch_count() - launches0
    elapsed_ms = t0.elapsed_time(t1)
    elapsed_ms = reduce_max(elapsed_ms, world, dev)
    if gemm.device_status(stream) != 0:
        raise RuntimeError("device status word set during the timed region")

    per_dtype = {}
    peaks, peak_src = load_peaks()
    for dt in DTYPES:
        ms = statistics.mean(e[dt][0].elapsed_time(e[dt][1]) for e in evs)
        ach = FLOP_PER_PRODUCT / (ms * 1e-3) / 1e12
        pk = peak_for(dt, peaks)
        pk_burst = peak_for(dt, peaks, sustained=False)
        per_dtype[dt] = {"kernel_ms": round(ms, 5), "tflops": round(ach, 2), "peak_tflops": round(pk, 1),
                         "frac": round(ach / pk, 4), "frac_of_burst_peak": round(ach / pk_burst, 4)}
    dominant = max(DTYPES, key=lambda d: per_dtype[d]["kernel_ms"])
    total_flop = FLOP_PER_PRODUCT * len(DTYPES) * args.steps * world
    value = total_flop / (elapsed_ms * 1e-3) / 1e12

    # end to end through the host-memory call: pinned operands in, C out, each step
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    host = {dt: (probs[dt].a.pin_memory(), probs[dt].b.pin_memory()) for dt in DTYPES}
    # two sets of device and pinned result buffers, taken by alternate steps
    bufs = [{dt: {} for dt in DTYPES} for _ in range(2)]
    for bset in bufs:  # warm the buffers
        for dt in DTYPES:
            gemm.matmul_from_host(host[dt][0], host[dt][1], device=dev, stream=stream, buffers=bset[dt])
    h2d = sum(host[dt][0].numel() * host[dt][0].element_size() + host[dt][1].numel() * host[dt][1].element_size()
              for dt in DTYPES)
    d2h = sum(M * N * host[dt][0].element_size() for dt in DTYPES)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    w0 = time.perf_counter()
    previous = []
    for step in range(e2e_steps):
        # the step's three products are enqueued at once (their copies queue on the
        # device's shared copy streams, behind the previous step's); then the
        # previous step's three results are waited for on the host, so every
        # step's inputs go in and its results come out within the timed region
        pending = [gemm.matmul_from_host(host[dt][0], host[dt][1], device=dev, stream=stream,
                                         buffers=bufs[step % 2][dt], wait=False) for dt in DTYPES]
        for _, done in previous:
            done.synchronize()
        previous = pending
    for _, done in previous:
        done.synchronize()
    torch.cuda.synchronize(dev)
    e2e_s = reduce_max(time.perf_counter() - w0, world, dev)
    e2e_value = FLOP_PER_PRODUCT * len(DTYPES) * e2e_steps * world / e2e_s / 1e12

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "tf32+f16+bf16 (fp32 accumulate)",
        "data": "synthetic (seeded U[-1,1) fp32 for TF32, N(0,1) rounded to f16/bf16)",
        "config": {"workload": "gemm_4096^3_tf32+f16+bf16", "M": M, "N": N, "K": K,
                   "layout": "A, B, C row-major", "products_per_step": len(DTYPES),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "no flush: each step streams 384 MiB of operands (3x the 129 MB L2), so a product's "
                         "inputs are evicted by the other two before it runs again"},
        "per_dtype": per_dtype,
        "roofline": {"bound": "tensor", "kernel": kernel_name(dominant, plans[dominant]),
                     "plan": {k: plans[dominant][k] for k in ("kernel", "tile_n", "raster", "tail_segs")},
                     "achieved": per_dtype[dominant]["tflops"], "peak": per_dtype[dominant]["peak_tflops"],
                     "unit": "TFLOP/s", "frac": per_dtype[dominant]["frac"],
                     "frac_of_burst_peak": per_dtype[dominant]["frac_of_burst_peak"], "traffic": None,
                     "peak_source": f"{peak_src} bf16 sustained (timed inside a long power-capped loop) "
                                    f"x nominal {dominant}/bf16 ratio"},
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "overlap": "a step's three products are enqueued before the previous step's results are waited "
                           "for (two buffer sets); every step's copies run inside the timed region"},
        "clocks": clocks.summary(),
        "gpu_launches": launches,
    }
    traffic = _traffic_record(dominant, plans[dominant])
    if traffic is not None:
        line["roofline"]["traffic"] = traffic
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(probs, args.cpu_seconds)
    if world > 1:
        dist.destroy_process_group()
    return line, rank


KIND_INDEX = {"f16": 0, "bf16": 1, "tf32": 2}


def kernel_name(dtype, plan):
    """The product kernel a plan launches, as ncu names it (row-major B).
    Plan kernel 1: single CTA; 2 and 4: one or two CTA pairs per cluster
    (operand arrangement 0); 3: a CTA pair on the transposed product
    (arrangement 2)."""
    k, bn = plan["kernel"], plan["tile_n"]
    if k == 1:
        return f"gemm_kernel<{KIND_INDEX[dtype]}, 0, {bn}>"
    if k == 3:
        return f"gemm_kernel_pair<{KIND_INDEX[dtype]}, 2, {bn}, 1>"
    return f"gemm_kernel_pair<{KIND_INDEX[dtype]}, 0, {bn}, {k // 2}>"


# Device code of the product kernels: the traffic record holds while these are unchanged.
KERNEL_SOURCES = ("gemm_kernel.cuh", "gemm_kernel_pair.cuh", "ptx.cuh")


def _kernel_sources_sha256():
    import hashlib
    csrc = os.path.join(ROOT, "dense_gemm_tensor_gb300", "csrc")
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _traffic_record(dtype, plan):
    """DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum) from the
    committed summary, or None when the kernel's device code changed since it was captured
    or this run's plan launched a different kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_sources_sha256") != _kernel_sources_sha256():
        return None
    rec = d.get(dtype)
    if not isinstance(rec, dict) or rec.get("kernel") != kernel_name(dtype, plan) or \
            rec.get("tail_segs") != plan["tail_segs"]:
        return None
    return rec.get("bytes")


def cpu_baseline(probs, seconds):
    """The oracle, as it stands, on a bounded sample of the workload: whole
    4096^3 products in the order TF32, FP16, BF16, repeated until `seconds`
    of wall time have passed."""
    import oracle
    done = 0
    t0 = time.perf_counter()
    while True:
        for dt in DTYPES:
            p = probs[dt]
            oracle.gemm(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, p.layout)
            done += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(done * FLOP_PER_PRODUCT / el / 1e12, 5), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{done} whole 4096^3 products (float64 numpy matmul via OpenBLAS, default thread count) "
                      f"in {el:.1f} s"}


def run_reference(args, world, rank):
    """The CPU oracle timed on the same workload: each step computes a slice
    of `rows` output rows of each of the three 4096^3 products."""
    if world > 1 and rank != 0:
        return None, rank
    import oracle
    probs = make_inputs()
    rows = args.ref_rows

    def step():
        for dt in DTYPES:
            p = probs[dt]
            oracle.gemm(rows, p.N, p.K, p.a, p.lda, p.b, p.ldb, p.layout)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    flop = 2.0 * rows * N * K * len(DTYPES) * args.steps
    value = flop / el / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = f"rows 0..{rows - 1} of each 4096^3 product (TF32, FP16, BF16) per step"
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 5), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": "gemm_4096^3_tf32+f16+bf16", "M": M, "N": N, "K": K},
        "cpu_baseline": {"value": round(value, 5), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line, rank


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-rows", type=int, default=128)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        line, rank = run_reference(args, world, rank)
    else:
        line, rank = run_ours(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
