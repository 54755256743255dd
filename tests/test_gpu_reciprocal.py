"""The producers' two-lane reciprocal (hardware approximation plus one
correction step, with the IEEE reciprocal for d >= 2^126) is bit-identical to
CUDA's IEEE reciprocal for every binary32 d >= 1: tests/csrc/reciprocal_check.cu,
compiled here and run on the GPU."""
import os
import subprocess

import pytest

from conftest import ROOT
from quantize_amax_scaling_gb300 import build

CSRC = os.path.join(ROOT, "tests", "csrc", "reciprocal_check.cu")


@pytest.mark.gpu
def test_reciprocal_matches_ieee_for_every_d_at_least_one(tmp_path):
    exe = str(tmp_path / "reciprocal_check")
    subprocess.run([build.nvcc_path(), *build.ARCH, "-O3", "-std=c++17", "-I", build.CSRC, "-o", exe, CSRC],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("mismatches: 0"), r.stdout
