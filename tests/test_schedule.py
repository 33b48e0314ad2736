"""The kernels' work schedule (csrc/schedule.cuh), checked on the CPU: the
same functions the kernels call are compiled for the host and run over the
benchmark's and the tests' launch shapes (every work item taken exactly
once, every workspace row inside the buffer)."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_schedule_covers_every_item_once(tmp_path):
    nvcc = os.environ.get("NVCC", "nvcc")
    exe = tmp_path / "schedule_check"
    src = os.path.join(ROOT, "tests", "schedule_check.cu")
    inc = os.path.join(ROOT, "exact_io_aware_108_b300", "csrc")
    try:
        subprocess.run([nvcc, "-std=c++17", "-O1", "-I", inc, "-o", str(exe), src], check=True,
                       capture_output=True, text=True)
    except FileNotFoundError:
        pytest.skip("nvcc is not available")
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip().endswith("ok"), out.stdout + out.stderr
