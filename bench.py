"""Benchmark of the dense GEMM at M = N = K = 4096 in TF32, FP16 and BF16.

One step is one pass of the whole path over one batch of synthetic input:
the three 4096^3 products (TF32 with fp32 operands uniform in [-1, 1);
FP16 and BF16 with N(0, 1) operands), each one launch of the library's
kernel through its C interface. ``value`` is TFLOP/s (2MNK per product)
over the timed steps with the operands resident in device memory, timed by
events at the two ends of the region only (an event between two products
stops the second from overlapping the first one's tail under programmatic
dependent launch); the roofline's per-kernel durations come from a second
pass of the same steps with events around every product. ``e2e``
is the same metric through the library's host-memory C call
(``gemm_{tf32,f16,bf16}_host``: pinned host operands copied in, C copied out,
every step). ``--impl reference`` times the CPU oracle on
the same workload instead (a bounded slice of rows per step).

Launch: ``python bench.py [--steps K] [--warmup W]``. The library and this
benchmark use one GPU: ``--gpus`` must be 1, and a run under torchrun with
more than one rank stops with an error (its reference arm runs on rank 0
only). The SM clock and throttle reasons are sampled through NVML during the
timed region; the roofline's peak is the burst figure when the clock stayed
at its maximum and the sustained (power-capped) figure otherwise, and the
line also gives the fraction of the tensor pipe's rate at the sampled clock.
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
# Dense tensor-pipe work per SM per clock: tcgen05.mma kind::f16 takes 2 x N
# cycles for a 128 x N x 16 step of one SM (kind::tf32: 128 x N x 8), i.e.
# 8192 and 4096 FLOP per clock per SM.
FLOP_PER_CLK_SM = {"bf16": 8192, "f16": 8192, "tf32": 4096}
SM_COUNT = 152
# A clock median within this fraction of the maximum counts as an unthrottled (burst) run.
BURST_CLOCK_FRACTION = 0.97


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


def peak_for(dtype: str, peaks: dict, sustained: bool) -> float:
    """Dense tensor peak for ``dtype`` in TFLOP/s: the measured BF16 figure
    times the nominal ratio. The burst figure is for kernels that ran at the
    maximum SM clock; the sustained figure (a seconds-long loop under the
    power cap) is for kernels whose clock the power cap pulled down."""
    burst = peaks["bf16_tflops"]
    base = peaks.get("bf16_tflops_sustained", burst) if sustained else burst
    return base * NOMINAL_RATIO[dtype]


def peak_is_sustained(clocks: dict) -> bool:
    """The sustained (power-capped) peak applies unless the clock record shows
    the SM clock at its maximum through the timed region (median within
    BURST_CLOCK_FRACTION of it, and no slowdown reason); without samples the
    sustained figure, the lower one, is taken."""
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if not sm or not smax:
        return True
    slowed = any(r != "no samples" for r in clocks.get("reasons", []))
    return slowed or sm < BURST_CLOCK_FRACTION * smax


class _Nvml:
    """The few NVML calls the clock record needs, through ctypes (NVML is the
    library nvidia-smi reads its clocks and reasons from)."""

    # nvmlClocksEventReasons bits that slow the clock down
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int):
        import ctypes
        self.c = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        uuid = _device_uuid(device_index)
        ok = False
        for u in ([uuid, "GPU-" + uuid] if uuid else []):
            if lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(self.h)) == 0:
                ok = True
                break
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(_nvml_index(device_index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for the device")
        self._reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self._u = ctypes.c_uint(0)
        self._ull = ctypes.c_ulonglong(0)

    def sm_mhz(self) -> int:
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.c.byref(self._u))  # NVML_CLOCK_SM
        return self._u.value

    def sm_max_mhz(self) -> int:
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, self.c.byref(self._u))
        return self._u.value

    def reasons(self) -> int:
        self._reasons(self.h, self.c.byref(self._ull))
        return self._ull.value

    def power_w(self) -> float:
        self.lib.nvmlDeviceGetPowerUsage(self.h, self.c.byref(self._u))
        return self._u.value / 1000.0


def _device_uuid(index: int) -> str | None:
    try:
        import torch
        u = str(torch.cuda.get_device_properties(index).uuid)
        return u if u and u != "None" else None
    except Exception:  # noqa: BLE001 - older torch without the field
        return None


def _nvml_index(index: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [x.strip() for x in vis.split(",") if x.strip()]
    if index < len(parts) and parts[index].isdigit():
        return int(parts[index])
    return index


class ClockSampler:
    """SM clock, throttle reasons and power read through NVML every ~0.5 ms
    by a background thread (from before the warm-up to after the timed
    region), each sample stamped with the host clock; ``summary(t0, t1)``
    keeps the samples taken inside a host-time window. Without NVML it falls
    back to an ``nvidia-smi -lms 50`` process."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_s: float = 0.0005):
        self.dev = device_index
        self.period = period_s
        self.samples = []  # (host time, sm MHz, reason names, power W)
        self.sm_max = None
        self.source = None
        self._stop = False
        self._thread = None
        self._proc = None

    def __enter__(self):
        import threading
        try:
            nv = _Nvml(self.dev)
            self.sm_max = nv.sm_max_mhz()
            self.source = "nvml"
            target = lambda: self._poll_nvml(nv)  # noqa: E731
        except OSError:
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={_nvml_index(self.dev)}", f"--query-gpu={self.QUERY}",
                     "--format=csv,noheader,nounits", "-lms", "50"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi"
                target = self._poll_smi
            except OSError:
                return self
        self._thread = threading.Thread(target=target, daemon=True)
        self._thread.start()
        return self

    def _poll_nvml(self, nv):
        while not self._stop:
            bits = nv.reasons()
            names = tuple(n for b, n in _Nvml.REASONS.items() if bits & b)
            self.samples.append((time.perf_counter(), nv.sm_mhz(), names, nv.power_w()))
            time.sleep(self.period)

    def _poll_smi(self):
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm, smax, power = float(parts[0]), float(parts[1]), float(parts[2])
            except ValueError:
                continue
            names = tuple(n for n, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                             "sw_power_cap"), parts[3:7]) if v.lower() == "active")
            self.sm_max = smax
            self.samples.append((time.perf_counter(), sm, names, power))

    def __exit__(self, *exc):
        self._stop = True
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        rows = [r for r in self.samples if t0 <= r[0] <= t1]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": self.sm_max, "reasons": ["no samples"], "samples": 0,
                    "source": self.source, "window_ms": round((t1 - t0) * 1e3, 3)}
        reasons = sorted({n for r in rows for n in r[2]})
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": self.sm_max,
                "sm_min_mhz": min(r[1] for r in rows), "reasons": reasons, "samples": len(rows),
                "power_w_max": max(r[3] for r in rows), "source": self.source,
                "window_ms": round((t1 - t0) * 1e3, 3)}


def make_inputs():
    from dense_gemm_tensor_gb300 import inputs
    return {dt: inputs.workload(WORKLOAD[dt]) for dt in DTYPES}


def run_ours(args):
    import torch
    from dense_gemm_tensor_gb300 import build as libbuild
    from dense_gemm_tensor_gb300 import gemm

    libbuild.build()
    gemm.load()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
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

    sampler = ClockSampler(0)
    sampler.__enter__()  # sampling from before the warm-up on
    try:
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

        # the timed region: K steps, events only at its two ends (an event
        # recorded between two products stops the second one's programmatic
        # dependent launch from overlapping the first one's tail: 6% per step)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        launches0 = gemm.launch_count()
        torch.cuda.synchronize(dev)
        h0 = time.perf_counter()
        with torch.cuda.stream(stream):
            t0.record(stream)
            for k in range(args.steps):
                step()
            t1.record(stream)
        torch.cuda.synchronize(dev)
        h1 = time.perf_counter()
        launches = gemm.launch_count() - launches0
        # per-kernel durations for the roofline: K more steps with events
        # around every product (same stream as the kernels)
        evs = [{dt: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for dt in DTYPES}
               for _ in range(args.steps)]
        torch.cuda.synchronize(dev)
        h2 = time.perf_counter()
        with torch.cuda.stream(stream):
            for k in range(args.steps):
                step(evs[k])
        torch.cuda.synchronize(dev)
        h3 = time.perf_counter()
    finally:
        sampler.__exit__(None, None, None)
    clocks = sampler.summary(h0, h1)
    kernel_clocks = sampler.summary(h2, h3)
    elapsed_ms = t0.elapsed_time(t1)
    if gemm.device_status(stream) != 0:
        raise RuntimeError("device status word set during the timed region")

    # the peak: burst when the sampled SM clock stayed at its maximum, sustained otherwise
    peaks, peak_src = load_peaks()
    sm_mhz, sm_max = kernel_clocks.get("sm_mhz"), kernel_clocks.get("sm_max_mhz")
    sustained = peak_is_sustained(kernel_clocks)
    per_dtype = {}
    for dt in DTYPES:
        ms = statistics.mean(e[dt][0].elapsed_time(e[dt][1]) for e in evs)
        ach = FLOP_PER_PRODUCT / (ms * 1e-3) / 1e12
        pk = peak_for(dt, peaks, sustained)
        rec = {"kernel_ms": round(ms, 5), "tflops": round(ach, 2), "peak_tflops": round(pk, 1),
               "frac": round(ach / pk, 4),
               "frac_of_burst_peak": round(ach / peak_for(dt, peaks, False), 4),
               "frac_of_sustained_peak": round(ach / peak_for(dt, peaks, True), 4)}
        if sm_mhz:
            clock_peak = SM_COUNT * sm_mhz * 1e6 * FLOP_PER_CLK_SM[dt] / 1e12
            rec["frac_of_clock_peak"] = round(ach / clock_peak, 4)
        per_dtype[dt] = rec
    dominant = max(DTYPES, key=lambda d: per_dtype[d]["kernel_ms"])
    total_flop = FLOP_PER_PRODUCT * len(DTYPES) * args.steps
    value = total_flop / (elapsed_ms * 1e-3) / 1e12
    kind = "sustained" if sustained else "burst"
    clock_note = (f"sampled SM clock median {sm_mhz} of max {sm_max} MHz" if sm_mhz else "no clock samples")

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
    e2e_s = time.perf_counter() - w0
    e2e_value = FLOP_PER_PRODUCT * len(DTYPES) * e2e_steps / e2e_s / 1e12

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": 1,
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
                   "parallelism": "single GPU",
                   "l2": "no flush: each step streams 384 MiB of operands (3x the 129 MB L2), so a product's "
                         "inputs are evicted by the other two before it runs again"},
        "per_dtype": per_dtype,
        "roofline": {"bound": "tensor", "kernel": kernel_name(dominant, plans[dominant]),
                     "plan": {k: plans[dominant][k] for k in ("kernel", "tile_n", "raster", "tail_segs")},
                     "achieved": per_dtype[dominant]["tflops"], "peak": per_dtype[dominant]["peak_tflops"],
                     "unit": "TFLOP/s", "frac": per_dtype[dominant]["frac"], "peak_kind": kind,
                     "frac_of_burst_peak": per_dtype[dominant]["frac_of_burst_peak"],
                     "frac_of_sustained_peak": per_dtype[dominant]["frac_of_sustained_peak"],
                     "frac_of_clock_peak": per_dtype[dominant].get("frac_of_clock_peak"), "traffic": None,
                     "peak_source": f"{peak_src} bf16 {kind} x nominal {dominant}/bf16 ratio ({clock_note}); "
                                    f"frac_of_clock_peak: against {FLOP_PER_CLK_SM[dominant]} FLOP per clock per "
                                    f"SM x {SM_COUNT} SMs at the sampled median clock",
                     "timing": "mean of CUDA-event pairs around each launch of the kernel, over a second pass of "
                               "the K steps right after the timed region (events between products would slow "
                               "the timed region itself)",
                     "clocks": kernel_clocks},
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "call": "gemm_{tf32,f16,bf16}_host (C interface, host pointers)",
                "overlap": "a step's three calls are enqueued before the previous step's results are waited "
                           "for; every step's copies run inside the timed region"},
        "clocks": clocks,
        "gpu_launches": launches,
    }
    traffic = _traffic_record(dominant, plans[dominant])
    if traffic is not None:
        line["roofline"]["traffic"] = traffic
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(probs, args.cpu_seconds)
    return line


KIND_INDEX = {"f16": 0, "bf16": 1, "tf32": 2}


def kernel_name(dtype, plan):
    """The product kernel a plan launches, as ncu names it (row-major B; the
    last template argument, 0 or 1, is whether it carries the fused epilogue).
    Plan kernel 1: single CTA; 2 and 4: one or two CTA pairs per cluster
    (operand arrangement 0); 3: a CTA pair on the transposed product
    (arrangement 2). Plain launches of the single-CTA kernel and of one pair
    per cluster take the builds without the fused epilogue."""
    k, bn = plan["kernel"], plan["tile_n"]
    if k == 1:
        return f"gemm_kernel<{KIND_INDEX[dtype]}, 0, {bn}, 0>"
    if k == 3:
        return f"gemm_kernel_pair<{KIND_INDEX[dtype]}, 2, {bn}, 1, 0>"
    return f"gemm_kernel_pair<{KIND_INDEX[dtype]}, 0, {bn}, {k // 2}, {0 if k == 2 else 1}>"


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
    world, rank, _ = dist_env()
    if args.impl == "reference":
        line, rank = run_reference(args, world, rank)
    else:
        if args.gpus != 1 or world > 1:
            # one GPU only: the product does not shard in these workloads, and the
            # library's cluster kernels are built for runs that use a single GPU
            sys.stderr.write("bench.py runs on one GPU: use --gpus 1 without torchrun\n")
            sys.exit(2)
        line, rank = run_ours(args), 0
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
