"""Host-side logic of bench.py without a GPU: the one-GPU rule, the clock
record and peak choice, the reference arm's rank handling, and its JSON line."""

import json
import os
import subprocess
import sys


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_ours_refuses_more_than_one_gpu():
    """The product runs on one GPU: --gpus 2 (or a multi-rank launch) stops
    with an error before any device work."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 2 and "one GPU" in r.stderr
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "1"], capture_output=True,
                       text=True, env=env, timeout=300)
    assert r.returncode == 2 and r.stdout.strip() == ""


def test_clock_window_and_peak_choice():
    """Samples outside the timed region's host-time window are left out; the
    burst peak applies only with the median clock at its maximum and no
    slowdown reason."""
    sys.path.insert(0, ROOT)
    import bench
    s = bench.ClockSampler(0)
    s.sm_max, s.source = 2070, "nvml"
    s.samples = [(0.5, 1500, ("sw_power_cap",), 900.0), (1.0, 2070, (), 500.0), (1.1, 2070, (), 600.0),
                 (1.2, 2055, (), 700.0), (2.5, 1600, ("sw_power_cap",), 1300.0)]
    d = s.summary(1.0, 2.0)
    assert d["samples"] == 3 and d["sm_mhz"] == 2070 and d["sm_min_mhz"] == 2055
    assert d["reasons"] == [] and d["power_w_max"] == 700.0 and d["window_ms"] == 1000.0
    assert not bench.peak_is_sustained(d)
    d = s.summary(0.0, 3.0)
    assert d["reasons"] == ["sw_power_cap"] and bench.peak_is_sustained(d)
    assert bench.peak_is_sustained(s.summary(5.0, 6.0))  # no samples: the lower, sustained peak
    assert bench.peak_is_sustained({"sm_mhz": 1700, "sm_max_mhz": 2070, "reasons": []})
    peaks = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0}
    assert bench.peak_for("bf16", peaks, False) == 2000.0 and bench.peak_for("bf16", peaks, True) == 1800.0
    assert abs(bench.peak_for("tf32", peaks, False) - 2000.0 * 1.1 / 2.25) < 1e-9


def test_reference_arm_other_ranks_do_no_work():
    sys.path.insert(0, ROOT)
    import bench
    line, rank = bench.run_reference(None, 2, 1)
    assert line is None and rank == 1


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--ref-rows", "2"], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("gemm_4096")


def test_bench_rejects_short_warmup():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2", "--impl", "reference"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0


def test_kernel_names_and_traffic_record():
    """The launch plan -> kernel name mapping (as ncu names the kernels) for
    every plan kind, and the committed traffic record: it names the kernels of
    the plans it was captured with and carries the device sources' hash."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.kernel_name("bf16", {"kernel": 1, "tile_n": 256}) == "gemm_kernel<1, 0, 256, 0>"
    assert bench.kernel_name("tf32", {"kernel": 2, "tile_n": 224}) == "gemm_kernel_pair<2, 0, 224, 1, 0>"
    assert bench.kernel_name("f16", {"kernel": 3, "tile_n": 224}) == "gemm_kernel_pair<0, 2, 224, 1, 0>"
    assert bench.kernel_name("bf16", {"kernel": 4, "tile_n": 256}) == "gemm_kernel_pair<1, 0, 256, 2, 1>"
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for dt in ("tf32", "f16", "bf16"):
        assert rec[dt]["kernel"].startswith("gemm_kernel") and rec[dt]["bytes"] > 0
    assert len(rec["kernel_sources_sha256"]) == 64
