"""Host cost of one call of the C interface (no Python in the loop): a small
C++ program, built here against libdgt_gemm.so, enqueues 400 BF16 512^3
products back to back and times the calls. The library's own work per call
(argument and memory checks, the cached plan and tensor maps, the launch
itself) must stay within 2 microseconds, and within 0.6 microseconds of an
empty kernel launch on the same machine (the part that is the library's)."""

import os
import subprocess

import pytest
import torch

from dense_gemm_tensor_gb300 import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def call_cost_binary():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = build.build()
    out_dir = os.path.join(ROOT, "_build", "tests")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "call_cost")
    libdir = os.path.dirname(lib)
    cmd = [build.nvcc(), *build.ARCH, "-O2", "-std=c++17", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "call_cost.cu"), "-o", exe, "-L", libdir, "-ldgt_gemm",
           "-Xlinker", f"-rpath={libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    return exe


def test_back_to_back_call_host_time(call_cost_binary):
    r = subprocess.run([call_cost_binary], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    vals = dict(line.split() for line in r.stdout.splitlines() if line.strip())
    call, launch = float(vals["call_us"]), float(vals["launch_us"])
    print(f"C call {call:.3f} us, empty launch {launch:.3f} us")
    assert call <= 2.0, (call, launch)
    assert call - launch <= 0.6, (call, launch)
