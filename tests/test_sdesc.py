"""The tcgen05 shared-memory descriptor arithmetic (csrc/sdesc.cuh),
checked on the CPU: the issue loops build a descriptor's low word once per
tile and step it by adds, with a constant high word; the host program
compares that with the descriptor built from each stepped address, over the
whole shared-memory window of a CTA."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_descriptor_words_step_like_addresses(tmp_path):
    nvcc = os.environ.get("NVCC", "nvcc")
    exe = tmp_path / "sdesc_check"
    src = os.path.join(ROOT, "tests", "sdesc_check.cu")
    inc = os.path.join(ROOT, "exact_io_aware_108_b300", "csrc")
    try:
        subprocess.run([nvcc, "-std=c++17", "-O2", "-I", inc, "-o", str(exe), src], check=True,
                       capture_output=True, text=True)
    except FileNotFoundError:
        pytest.skip("nvcc is not available")
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.strip().endswith("ok"), out.stdout + out.stderr
