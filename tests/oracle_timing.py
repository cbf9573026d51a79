"""Times the CPU oracle (float64, oracle.gemm) on every synthetic workload, on
this machine's host cores, and prints a Markdown table.

    python tests/oracle_timing.py [--out FILE]

Products of at most 4096^3 multiply-adds are timed whole; the larger ones on a
fixed 256-row slice of A (the same arithmetic per output row), with the full
time extrapolated by rows and labelled so. A product that takes under a
second is timed three times and the best kept. The 512^3 product is also timed on
one thread (in a child process whose BLAS thread count is fixed before numpy
loads). The oracle is a reported baseline, not a target; operand generation
is not timed.
"""

import argparse
import json
import os
import subprocess
import sys
import time

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
from dense_gemm_tensor_gb300 import inputs  # noqa: E402

WHOLE_LIMIT = 4096 ** 3
SLICE_ROWS = 256
THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def warm_up() -> None:
    """One untimed small product, so that starting the BLAS threads is not timed."""
    p = inputs.make_problem("warm", "bf16", 256, 256, 256)
    oracle.gemm(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, p.layout)


def time_one(name: str) -> dict:
    p = inputs.workload(name)
    whole = p.M * p.N * p.K <= WHOLE_LIMIT
    rows = p.M if whole else min(SLICE_ROWS, p.M)
    a = p.a[:rows]
    sec = None
    for _ in range(3):  # best of three for a product under a second, else one run
        t0 = time.perf_counter()
        oracle.gemm(rows, p.N, p.K, a, p.lda, p.b, p.ldb, p.layout)
        dt = time.perf_counter() - t0
        sec = dt if sec is None else min(sec, dt)
        if dt >= 1.0:
            break
    full = sec * p.M / rows
    return dict(name=name, shape=f"{p.M}×{p.N}×{p.K}", timed="whole" if whole else f"{rows} rows of A",
                seconds=sec, full_seconds=full, extrapolated=not whole,
                gflops=2.0 * p.M * p.N * p.K / full / 1e9)


def single_thread_512() -> dict:
    env = dict(os.environ, **{v: "1" for v in THREAD_VARS})
    code = ("import json, sys; sys.path.insert(0, %r); import oracle_timing as t; "
            "t.warm_up(); print(json.dumps(t.time_one('bf16_512')))" % os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True)
    r = json.loads(out.stdout.strip().splitlines()[-1])
    r["name"] += " (1 thread)"
    return r


def table(rows: list[dict], cores: int) -> str:
    out = [f"Oracle (float64 numpy matrix product) on {cores} host cores:", "",
           "| workload | M×N×K | timed | measured s | full product s | GFLOP/s |",
           "|---|---|---|---|---|---|"]
    for r in rows:
        full = f"{r['full_seconds']:.3f}" + (" (extrapolated)" if r["extrapolated"] else "")
        out.append(f"| {r['name']} | {r['shape']} | {r['timed']} | {r['seconds']:.3f} | {full} | {r['gflops']:.1f} |")
    return "\n".join(out)


def main() -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--out", default=None, help="also write the table to this file")
    args = ap.parse_args()
    warm_up()
    rows = []
    for name in inputs.WORKLOADS:
        r = time_one(name)
        print(f"{name}: {r['seconds']:.3f} s ({r['timed']})", flush=True)
        rows.append(r)
    rows.append(single_thread_512())
    text = table(rows, os.cpu_count() or 1)
    print(text)
    if args.out:
        with open(args.out, "w") as f:
            f.write(text + "\n")
    return 0


if __name__ == "__main__":
    sys.exit(main())
