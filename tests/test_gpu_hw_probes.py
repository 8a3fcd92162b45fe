"""Hardware probes behind the kernel design (tests/hw_probes/*.cu).

Each probe is built for sm_103a and run on the GPU; the test checks that every
configuration ran without a CUDA error or a timed-out wait and prints the
measured table (``pytest -s``), which the profiles quote:

* ``mma_rate.cu``: tcgen05.mma kind::f16 rate per tile shape (1-CTA M=128 and
  cta_group::2 M=256, N = 16..256), and the cost of a tcgen05.commit per K step
  and of independent accumulators -- why the 2-CTA weight-row tiles fit N to
  the expert, what a K step of a small-N tile costs, and why the decode kernel
  releases a stage of two K steps with one commit.
* ``tma_stream.cu``: per-SM streaming rate of K-major bulk-tensor weight loads,
  128-byte rows (64-column boxes) against 256-byte rows (two 64-column planes)
  -- why the 2-CTA GEMMs load stages of two K steps.
"""
import os
import re
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "mixture_experts_ffn_permute_gb300", "csrc")


def _build_and_run(name, tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / name)
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", CSRC, "-o", exe, os.path.join(HERE, "hw_probes", name + ".cu"), "-lcuda"],
                   check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=300).stdout
    print(out)
    return out


@pytest.mark.gpu
def test_mma_rate_probe(tmp_path):
    out = _build_and_run("mma_rate", tmp_path)
    lines = [l for l in out.splitlines() if "TFLOP/s" in l]
    assert len(lines) == 24
    for l in lines:
        assert "err=0 status=0" in l, l
    base = [l for l in lines if "commits=0 chains=1" in l]
    rate = {(l.split()[0], int(re.search(r"N=\s*(\d+)", l).group(1))):
            float(re.search(r"([\d.]+) TFLOP/s", l).group(1)) for l in base}
    # a pair at N = 256 does twice the work of one CTA per K step at the same rate
    assert rate[("pair", 256)] > 0.8 * rate[("1-CTA", 256)]


@pytest.mark.gpu
def test_tma_stream_probe(tmp_path):
    out = _build_and_run("tma_stream", tmp_path)
    lines = [l for l in out.splitlines() if "GB/s" in l]
    assert len(lines) == 40
    for l in lines:
        assert "err=0 status=0" in l, l
