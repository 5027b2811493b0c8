"""The kernels' layout index math (csrc/common.cuh: per-row key spans, tile
key ranges with the forward's range-by-range masks and full-tile shortcut,
and the backward's key-major row ranges) checked on the host against a
pairwise restatement of the BDLM mask, over random lengths (ragged last
blocks included), block sizes, key windows, query row ranges and block
groups. The check program is compiled with nvcc and runs on the CPU."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "block_diffusion_lm_bdlm_gb300", "csrc")


def test_layout_math_matches_the_mask(tmp_path):
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "layout_check")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-I", CSRC, os.path.join(HERE, "layout_check.cu"), "-o", exe],
                   check=True, capture_output=True, timeout=300)
    r = subprocess.run([exe, "300"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 failures" in r.stdout
