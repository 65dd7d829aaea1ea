"""The kernels divide by launch-invariant divisors (tile count, v-heads, group
size, tokens) with a multiply and a shift; this checks that division on the
host against the exact integer quotient over edge and random numerators for
thousands of divisors (the same header the kernels are built from)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "linear_attention_speculative_gb300", "csrc")


def test_fast_division_is_exact(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "fastdiv_check"
    r = subprocess.run([nvcc, "-std=c++17", "-O2", "-I", CSRC, "-o", str(exe),
                        os.path.join(ROOT, "tests", "fastdiv_check.cu")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.startswith("ok "), out.stdout
    assert int(out.stdout.split()[1]) > 1_000_000
