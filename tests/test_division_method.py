"""The quantize kernel divides by the scale with a Markstein correction step
instead of an IEEE divide; this checks the method exhaustively on the host.

The GPU parity tests then compare the kernel's bytes with the oracle's (which
divides with plain IEEE binary32 division) over all 65536 bf16 inputs.
"""
import os
import subprocess
import tempfile

from conftest import ROOT


def test_markstein_step_equals_ieee_division():
    src = os.path.join(ROOT, "tests", "csrc", "division_method_check.c")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "check")
        subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-o", exe, src, "-lm"],
                       check=True)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=600)
        assert out.returncode == 0, out.stdout + out.stderr
        assert "mismatches 0 (significand sweep) 0 (band edges)" in out.stdout
