"""The stream-K split shared by the product kernels and the finishing prep
(SplitK), checked on the host: contiguous non-empty ranges covering every
unit, and the owner of each unit, for uniform and lighter-tail splits."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_split_ranges_and_owners(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "split_check")
    src = os.path.join(HERE, "split_check.cu")
    inc = os.path.join(ROOT, "bit_weight_streaming_gb300", "csrc")
    r = subprocess.run([nvcc, "-std=c++17", "-O1", "-I", inc, src, "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0 and "split ok" in r.stdout, r.stdout + r.stderr
