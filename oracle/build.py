"""Compile the CPU oracle (test infrastructure) into ``oracle/libfp8q_oracle.so``.

Plain C11 with ``-ffp-contract=off`` and no fast-math, so every float
operation is one IEEE binary32 operation rounded to nearest even on both
x86-64 and AArch64 hosts.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fp8q_oracle.c")
LIB = os.path.join(HERE, "libfp8q_oracle.so")

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its sources."""
    srcs = [SRC, os.path.join(HERE, "fp8q_oracle.h")]
    if not force and os.path.exists(LIB):
        if os.path.getmtime(LIB) >= max(os.path.getmtime(s) for s in srcs):
            return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
