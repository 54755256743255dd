"""Compile libfp8q.so (the CUDA kernels and their C ABI) for sm_103a, in tree.

Four translation units compiled in parallel with one -gencode each, then
linked; no cmake.  The library and its objects are written next to this file
and git-ignored.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
UNITS = ["quantize.cu", "producers.cu", "scale_update.cu", "abi.cu"]
SRCS = [os.path.join(CSRC, u) for u in UNITS]
DEPS = SRCS + [os.path.join(CSRC, h) for h in ("fp8q_common.cuh", "packed_f32.cuh", "quant_tile.cuh",
                                                "slot_math.cuh", "mbarrier.cuh")] + [os.path.join(ROOT, "include", "fp8q.h")]
LIB = os.path.join(PKG, "libfp8q.so")
OBJ_DIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-lineinfo", "-O3", "-std=c++17",
    "-Xcompiler", "-fPIC",
    "-Xptxas", "-warn-spills",
]


def nvcc_path() -> str:
    cand = [os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"]
    for c in cand:
        p = os.path.join(c, "bin", "nvcc") if c else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return p


def build(force: bool = False, verbose: bool = False) -> str:
    """Build libfp8q.so if missing or older than its sources; return its path."""
    if not force and os.path.exists(LIB):
        if os.path.getmtime(LIB) >= max(os.path.getmtime(p) for p in DEPS):
            return LIB
    os.makedirs(OBJ_DIR, exist_ok=True)
    nvcc = nvcc_path()
    tag = f".{os.getpid()}"

    def compile_one(src):
        obj = os.path.join(OBJ_DIR, os.path.basename(src) + tag + ".o")
        cmd = [nvcc, *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-c", "-o", obj, src]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        subprocess.run(cmd, check=True)
        return obj

    with ThreadPoolExecutor(len(SRCS)) as ex:
        objs = list(ex.map(compile_one, SRCS))
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
    for o in objs:
        os.remove(o)
    return LIB


def build_variant(lib_path: str, defines) -> str:
    """Compile the same sources with extra preprocessor definitions into lib_path.

    Only tests use this: it builds libraries whose test hooks (for example
    FP8Q_TEST_LN_GIVE_UP_AT) exercise paths that correct operation never takes.
    """
    nvcc = nvcc_path()
    out_dir = os.path.dirname(os.path.abspath(lib_path))
    os.makedirs(out_dir, exist_ok=True)
    flags = [f"-D{d}" for d in defines]

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        subprocess.run([nvcc, *NVCC_FLAGS, *flags, "-I", os.path.join(ROOT, "include"), "-c", "-o", obj, src],
                       check=True)
        return obj

    with ThreadPoolExecutor(len(SRCS)) as ex:
        objs = list(ex.map(compile_one, SRCS))
    subprocess.run([nvcc, *ARCH, "-shared", "-o", lib_path, *objs], check=True)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
