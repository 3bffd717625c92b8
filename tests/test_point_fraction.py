"""The value stage computes each sample point in integers (point_fraction) instead of fp64.
It must equal, bit for bit, the IEEE double evaluation that the oracle performs: a host
build of the same header, checked against doubles on this machine (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_integer_points_equal_the_fp64_points(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "point_fraction_check")
    src = os.path.join(HERE, "host", "point_fraction_check.cu")
    subprocess.run([nvcc, "-std=c++17", "-O2", "--expt-relaxed-constexpr", src, "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout[-2000:]
    assert " 0 mismatches" in out.stdout
