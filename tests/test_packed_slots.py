"""Chunk slots of packed sequences (packed_seq.cuh), checked on the host.

The KDA backward and the DPLR entry points give each sequence of a packed batch
the chunk slots b + floor(lo_b / C) + n (B + ceil(T / C) per head) and find a
CTA's sequence by bisection.  tests/host/packed_seq_check.cu includes the same
header the kernels do and checks, for random packings (and for clamped,
non-monotone offsets), that every index stays inside the workspace, that no two
chunks share a slot and that the bisection inverts the slot map.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else shutil.which("nvcc")


def test_packed_slot_arithmetic(tmp_path):
    nvcc = _nvcc()
    if not nvcc:
        pytest.skip("nvcc not found")
    exe = tmp_path / "packed_seq_check"
    src = os.path.join(ROOT, "tests", "host", "packed_seq_check.cu")
    inc = os.path.join(ROOT, "chunkwise_gated_delta_gb300", "csrc")
    r = subprocess.run([nvcc, "-O1", "-std=c++17", "-I", inc, src, "-o", str(exe)], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
