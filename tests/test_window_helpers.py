"""The sliding-window helpers of the CUDA path (tile test, row spans, bit
ranges in csrc/bsa_common.h) against brute force on every small case,
compiled for the host with g++. No GPU; independent of the oracle."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_window_helpers_match_brute_force(tmp_path):
    gxx = shutil.which("g++")
    cuda_inc = "/usr/local/cuda/include"
    if gxx is None or not os.path.isdir(cuda_inc):
        pytest.skip("g++ or the CUDA headers are missing")
    exe = str(tmp_path / "window_check")
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "block_sparse_attention_attn_gb300", "csrc"),
                    "-I", cuda_inc, os.path.join(ROOT, "tests", "window_helpers_check.cpp"), "-o", exe],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
