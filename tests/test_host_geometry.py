"""Host-side invariants of the step kernel's geometry, checked on the CPU.

The kernels turn two run-time divisions into cheaper operations: stage row
counts and segments per row are shifted by (so they must be powers of two
for every inner dimension the weight stream accepts), and a ring slot is
found by a multiply-high with ring_magic(ns) (exact only for stage counters
below 2^32 / ns).  tests/host/geometry_check.cu includes the library's own
headers, enumerates both, and fails on any exception.  Needs nvcc; no GPU."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_stage_geometry_powers_of_two_and_ring_magic(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "geometry_check")
    src = os.path.join(HERE, "host", "geometry_check.cu")
    csrc = os.path.join(ROOT, "ar_decode_step_gb300", "csrc")
    subprocess.run([nvcc, "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a",
                    "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", csrc, src, "-o", exe],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
