"""The append kernels divide by the block scale with a reciprocal product and
one fused-multiply-add correction instead of an IEEE divide.  This test
builds tests/cuda/quant_exhaustive.cu and checks, on the GPU, that the e4m3
code of every bf16 value over every reachable scale (amax/448 of a bf16 amax)
equals the code of CUDA's correctly rounded quotient."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_division_matches_ieee_on_every_input(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "quant_exhaustive")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", os.path.join(ROOT, "paged_fp8_kv_append_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "cuda", "quant_exhaustive.cu"), "-o", exe],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches=0" in r.stdout
