"""The LayerNorm producer's mbarrier waits are bounded: tests/csrc/mbarrier_timeout_check.cu
shows, on the GPU and without any fault, that a wait whose bulk copy arrives succeeds
and that a wait nothing completes gives up after about one second and reports it."""
import os
import subprocess

import pytest

from conftest import ROOT
from quantize_amax_scaling_gb300 import build

CSRC = os.path.join(ROOT, "tests", "csrc", "mbarrier_timeout_check.cu")


@pytest.mark.gpu
def test_empty_mbarrier_wait_gives_up_and_reports(tmp_path):
    exe = str(tmp_path / "mbarrier_timeout_check")
    subprocess.run([build.nvcc_path(), *build.ARCH, "-O3", "-std=c++17", "-I", build.CSRC, "-o", exe, CSRC],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("OK"), r.stdout
