"""The boundary is a plain C ABI: a C program built with gcc against
include/fp8q.h and linked to libfp8q.so uses it with no Python in between."""
import os
import subprocess
import tempfile

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "tests", "csrc", "abi_from_c.c")
PKG = os.path.join(ROOT, "quantize_amax_scaling_gb300")


def _build(d, with_cuda):
    from quantize_amax_scaling_gb300 import build
    build.build()
    exe = os.path.join(d, "abi_from_c")
    cmd = ["gcc", "-std=c11", "-O1", "-I", os.path.join(ROOT, "include"), "-o", exe, SRC,
           "-L", PKG, "-lfp8q", "-Wl,-rpath," + PKG]
    if with_cuda:
        cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
        cmd[1:1] = ["-DWITH_CUDA", "-I", os.path.join(cuda, "include")]
        cmd += ["-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64")]
    subprocess.run(cmd, check=True)
    return exe


def test_c_program_argument_checks():
    with tempfile.TemporaryDirectory() as d:
        out = subprocess.run([_build(d, False), "args"], capture_output=True, text=True, timeout=120)
        assert out.returncode == 0 and "OK" in out.stdout, out.stdout + out.stderr


@pytest.mark.gpu
def test_c_program_on_the_gpu():
    with tempfile.TemporaryDirectory() as d:
        out = subprocess.run([_build(d, True), "gpu"], capture_output=True, text=True, timeout=300)
        assert out.returncode == 0 and "OK" in out.stdout, out.stdout + out.stderr
