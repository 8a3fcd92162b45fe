"""The 2-CTA weight-row kernels walk their tile sequence with an incremental
iterator (pair_tiles.cuh, TileIter) instead of decoding each tile from
scratch; this checks, on the host, that both give the same tile at every
position a CTA pair visits.  Needs nvcc (host code only, no GPU)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "mixture_experts_ffn_permute_gb300", "csrc")


def test_tile_iterator_matches_decode(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "tile_order_check")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-I", CSRC, "-o", exe,
                    os.path.join(ROOT, "tests", "tile_order_check.cu")], check=True,
                   capture_output=True)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0 and res.stdout.strip() == "ok", res.stdout + res.stderr
