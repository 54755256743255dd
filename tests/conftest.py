import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this environment")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle


@pytest.fixture(scope="session")
def seq_gelu(tmp_path_factory):
    """bf16 bits of the GELU producer's fixed binary32 sequence (tests/csrc/gelu_sequence.c):
    a determinism check of the kernels' bits, not the oracle."""
    import ctypes
    import subprocess

    import numpy as np

    d = tmp_path_factory.mktemp("gelu_sequence")
    so = str(d / "libgelu_sequence.so")
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-o", so,
                    os.path.join(ROOT, "tests", "csrc", "gelu_sequence.c"), "-lm"], check=True)
    L = ctypes.CDLL(so)
    L.seq_gelu_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    L.seq_gelu_bf16.restype = None

    def run(h_bits):
        h = np.ascontiguousarray(h_bits, np.uint16).reshape(-1)
        y = np.empty(h.shape, np.uint16)
        L.seq_gelu_bf16(h.ctypes.data, h.size, y.ctypes.data)
        return y

    return run


@pytest.fixture(scope="session")
def hooks_lib(tmp_path_factory):
    """libfp8q built once more with its test hooks (never the product build):
    FP8Q_TEST_LN_GIVE_UP_AT=1 makes each LayerNorm warp's wait for its second row
    report failure; FP8Q_TEST_GELU_TABLE_MIN_ELEMS=1 sends every vector-path GELU
    tensor through the table kernel, however small; FP8Q_TEST_HOOKS exports
    fp8q_test_set_gelu_max_cluster and fp8q_test_set_ln_max_cluster, which make larger
    thread-block clusters of the GELU table and the LayerNorm kernels count as not
    fitting.  Loaded with ctypes; only the entry points the hook tests call are
    declared."""
    import ctypes

    from quantize_amax_scaling_gb300 import build

    path = str(tmp_path_factory.mktemp("hooks") / "libfp8q_test_hooks.so")
    build.build_variant(path, ["FP8Q_TEST_LN_GIVE_UP_AT=1", "FP8Q_TEST_GELU_TABLE_MIN_ELEMS=1", "FP8Q_TEST_HOOKS"])
    L = ctypes.CDLL(path)
    vp = ctypes.c_void_p
    L.fp8q_layernorm_quantize_amax.argtypes = [vp, vp, vp, ctypes.c_int64, ctypes.c_int32, vp, vp, ctypes.c_float,
                                               ctypes.c_int, vp, vp, vp]
    L.fp8q_layernorm_quantize_amax.restype = ctypes.c_int
    L.fp8q_gelu_quantize_amax.argtypes = [vp, vp, vp, ctypes.c_int64, ctypes.c_int, vp, vp, vp]
    L.fp8q_gelu_quantize_amax.restype = ctypes.c_int
    L.fp8q_test_set_gelu_max_cluster.argtypes = [ctypes.c_int]
    L.fp8q_test_set_gelu_max_cluster.restype = None
    L.fp8q_test_set_ln_max_cluster.argtypes = [ctypes.c_int]
    L.fp8q_test_set_ln_max_cluster.restype = None
    return L
