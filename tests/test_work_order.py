"""The work decode of the persistent attention kernels (work_slot,
csrc/sm103.cuh) on the host: compiled with nvcc as host code (no GPU needed)
and checked to be a bijection from work indices onto (item, head) pairs for
many shapes, with the head as the slow index inside a block of items."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_work_slot_is_a_bijection(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "work_slot_check"
    src = os.path.join(ROOT, "tests", "host", "work_slot_check.cu")
    r = subprocess.run([nvcc, "-std=c++17", "-O1", "-o", str(exe), src], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr
