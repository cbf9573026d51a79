"""The range-checked debug build (every shared-memory, tensor-memory,
TMA-coordinate and scratch access the kernels compute tested against its
range, failures recorded in the device status word instead of trapping):
built for sm_103a, it runs every kernel family on representative products
with no range violation and results within the oracle's tolerance."""

import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_reports_no_violation():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_run.py")], capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res.pop("status") == 0, res
    assert res.pop("split_segments") > 1
    assert res.pop("swap_split_segments") > 1
    assert all(res.values()), res
