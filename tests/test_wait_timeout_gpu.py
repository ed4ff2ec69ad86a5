"""Failure detection without a GPU fault: every wait inside the library's
kernels is a bounded mbarrier wait that gives up with KV_ERR_TIMEOUT.  This
test makes one run out -- a barrier that nothing arrives on -- in a small
kernel of its own (tests/cuda/wait_timeout.cu) built on the library's wait
helper, and checks the status, the location word, that the other waiting
warps give up with it, and that the context stays usable for the next
launch.  The library's own kernels are never made to stall."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_lost_arrival_becomes_timeout_status(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "wait_timeout")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", os.path.join(ROOT, "paged_fp8_kv_append_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "cuda", "wait_timeout.cu"), "-o", exe],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "PASS" in r.stdout
