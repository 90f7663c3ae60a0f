"""Host-side check of the per-warp workspace layout (`ws_layout` in the library's internal
header): regions ordered, aligned and inside the total, and every second-level subtree of a
root inside that root's regions; and of the records of subtrees built ahead (`rec_layout`).
Compiled with nvcc as host code and run on the CPU.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_workspace_layout_invariants(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "layout_check"
    subprocess.run([nvcc, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "maximal_clique_enumeration_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "layout", "layout_check.cu"), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr
