"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/fp8q.h declares, and rejects bad arguments before it
touches CUDA (so these calls launch nothing)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HDR = os.path.join(ROOT, "include", "fp8q.h")


@pytest.fixture(scope="module")
def L():
    from quantize_amax_scaling_gb300 import build, fp8q
    build.build()
    return fp8q.lib()


def declared_functions():
    text = open(HDR).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|fp8q_status)\s+(fp8q_\w+)\s*\(", text, re.M)))


def test_header_declares_the_four_operations():
    names = declared_functions()
    for f in ("fp8q_quantize_amax", "fp8q_multi_quantize_amax", "fp8q_dequantize",
              "fp8q_amax_scale_update", "fp8q_qdq_amax", "fp8q_amax_scale_update_ring",
              "fp8q_gelu_quantize_amax", "fp8q_layernorm_quantize_amax",
              "fp8q_amax_scale_update_ring_quantize", "fp8q_status_string", "fp8q_last_cuda_error"):
        assert f in names


def test_library_exports_every_declared_symbol(L):
    from quantize_amax_scaling_gb300 import fp8q
    names = declared_functions()
    assert sorted(fp8q.EXPORTS) == names
    for f in names:
        assert hasattr(L, f), f


def test_status_strings(L):
    from quantize_amax_scaling_gb300 import fp8q
    for code, name in fp8q.STATUS.items():
        assert fp8q.status_string(code) == name
    assert L.fp8q_last_cuda_error() == b""


INVALID, TOO_MANY, OK = 1, 4, 0
P = ctypes.c_void_p(0x10000)       # never dereferenced: every call below fails validation first
ODD = ctypes.c_void_p(0x10001)


def test_quantize_argument_errors(L):
    q = L.fp8q_quantize_amax
    assert q(None, None, 0, 0, None, None, None) == OK            # empty: nothing to do
    assert q(P, P, -1, 0, P, P, None) == INVALID
    assert q(P, P, 5, 2, P, P, None) == INVALID                   # unknown format
    assert q(P, P, 0, 7, P, P, None) == INVALID                   # unknown format even when empty
    for args in ((None, P, P, P), (P, None, P, P), (P, P, None, P), (P, P, P, None)):
        x, qq, s, a = args
        assert q(x, qq, 5, 0, s, a, None) == INVALID
    assert q(ODD, P, 5, 0, P, P, None) == INVALID                 # bf16 pointer must be even
    assert q(P, P, 5, 0, ctypes.c_void_p(0x10002), P, None) == INVALID  # float pointer alignment


def test_multi_argument_errors(L):
    from quantize_amax_scaling_gb300.fp8q import Tensor
    m = L.fp8q_multi_quantize_amax
    assert m(None, 0, 0, None) == OK
    assert m(None, -1, 0, None) == INVALID
    assert m(None, 3, 0, None) == INVALID
    arr = (Tensor * 600)()
    assert m(ctypes.cast(arr, ctypes.c_void_p), 513, 0, None) == TOO_MANY
    assert m(ctypes.cast(arr, ctypes.c_void_p), 600, 1, None) == TOO_MANY
    # all-empty list: OK, nothing launched
    assert m(ctypes.cast(arr, ctypes.c_void_p), 512, 0, None) == OK
    arr[3].n = 10            # one live tensor with NULL pointers
    assert m(ctypes.cast(arr, ctypes.c_void_p), 5, 0, None) == INVALID
    arr[3].n = -2
    assert m(ctypes.cast(arr, ctypes.c_void_p), 5, 0, None) == INVALID
    assert m(ctypes.cast(arr, ctypes.c_void_p), 5, 9, None) == INVALID


def test_gelu_quantize_argument_errors(L):
    f = L.fp8q_gelu_quantize_amax
    assert f(None, None, None, 0, 0, None, None, None) == OK
    assert f(P, None, P, -1, 0, P, P, None) == INVALID
    assert f(P, None, P, 4, 2, P, P, None) == INVALID
    for h, q, sc, am in ((None, P, P, P), (P, None, P, P), (P, P, None, P), (P, P, P, None)):
        assert f(h, None, q, 4, 0, sc, am, None) == INVALID
    assert f(ODD, None, P, 4, 0, P, P, None) == INVALID
    assert f(P, ODD, P, 4, 0, P, P, None) == INVALID


def test_layernorm_quantize_argument_errors(L):
    f = L.fp8q_layernorm_quantize_amax
    UNSUPPORTED = 2
    #          x  y     q  rows hidden gamma beta eps  fmt sc am  stream
    good = [P, None, P, 4, 64, P, P, 1e-6, 0, P, P, None]
    def call(i, v):
        a = list(good)
        a[i] = v
        return f(*a)
    assert call(3, 0) == OK                          # no rows: nothing launched
    assert call(3, -1) == INVALID
    for h in (0, 8, 24, -16):                        # hidden >= 16 and a multiple of 16
        assert call(4, h) == INVALID
    assert call(4, 32768 + 16) == UNSUPPORTED        # longest row one CTA holds is 32768
    assert call(8, 2) == INVALID
    for i in (0, 2, 5, 6, 9, 10):
        assert call(i, None) == INVALID
    assert call(9, ctypes.c_void_p(0x10002)) == INVALID
    assert call(10, ctypes.c_void_p(0x10002)) == INVALID
    for i in (0, 1, 2, 5, 6):                  # x (bulk copies), y, q, gamma, beta: 16-byte aligned
        assert call(i, ctypes.c_void_p(0x10008)) == UNSUPPORTED


def test_qdq_argument_errors(L):
    f = L.fp8q_qdq_amax
    assert f(None, None, 0, 0, None, None, None) == OK
    assert f(P, P, -1, 0, P, P, None) == INVALID
    assert f(P, P, 4, 3, P, P, None) == INVALID
    for args in ((None, P, P, P), (P, None, P, P), (P, P, None, P), (P, P, P, None)):
        x, y, sc, am = args
        assert f(x, y, 4, 0, sc, am, None) == INVALID
    assert f(ODD, P, 4, 0, P, P, None) == INVALID
    assert f(P, ODD, 4, 0, P, P, None) == INVALID


def test_ring_update_argument_errors(L):
    u = L.fp8q_amax_scale_update_ring
    good = [P, P, 16, 4, P, P, P, None, 0, 0, 0, None]
    def call(i, v):
        a = list(good)
        a[i] = v
        return u(*a)
    assert call(2, 0) == INVALID
    assert call(3, 0) == INVALID
    assert call(8, 5) == INVALID
    assert call(9, 7) == INVALID
    assert call(10, 99) == INVALID
    for i in (0, 1, 4, 5, 6):
        assert call(i, None) == INVALID
        assert call(i, ctypes.c_void_p(0x10002)) == INVALID


def test_ring_update_quantize_argument_errors(L):
    f = L.fp8q_amax_scale_update_ring_quantize
    P2 = ctypes.c_void_p(0x20000)
    #       hist head_in head_out H  S  new sc si  sf  fmt algo margin x  q  n  slot amax stream
    good = [P, P, P2, 16, 4, P, P, P, None, 0, 0, 0, P, P, 64, 1, P, None]
    def call(i, v):
        a = list(good)
        a[i] = v
        return f(*a)
    assert call(3, 0) == INVALID                 # history_len
    assert call(4, 0) == INVALID                 # num_slots
    assert call(9, 5) == INVALID                 # fmt
    assert call(10, 3) == INVALID                # algo
    assert call(11, 65) == INVALID               # margin
    for slot in (-1, 4):
        assert call(15, slot) == INVALID
    assert call(2, P) == INVALID                 # head_out must differ from head_in
    for i in (0, 1, 2, 5, 6, 7):
        assert call(i, None) == INVALID
        assert call(i, ctypes.c_void_p(0x10002)) == INVALID
    assert call(14, -1) == INVALID               # n
    for i in (12, 13, 16):                       # x, q, amax with n > 0
        assert call(i, None) == INVALID
    assert call(12, ODD) == INVALID              # bf16 x must be even


def test_dequantize_argument_errors(L):
    d = L.fp8q_dequantize
    assert d(None, None, 0, 0, None, None) == OK
    assert d(P, P, -3, 0, P, None) == INVALID
    assert d(P, P, 3, 5, P, None) == INVALID
    assert d(None, P, 3, 0, P, None) == INVALID
    assert d(P, None, 3, 0, P, None) == INVALID
    assert d(P, P, 3, 0, None, None) == INVALID
    assert d(P, ODD, 3, 0, P, None) == INVALID


def test_scale_update_argument_errors(L):
    u = L.fp8q_amax_scale_update
    good = (P, 16, 4, P, P, P, None, 0, 0, 0, None)
    def call(i, v):
        a = list(good)
        a[i] = v
        return u(*a)
    assert call(1, 0) == INVALID          # history_len < 1
    assert call(2, 0) == INVALID          # num_slots < 1
    assert call(7, 2) == INVALID          # fmt
    assert call(8, 2) == INVALID          # algo
    assert call(9, 65) == INVALID         # margin
    assert call(9, -65) == INVALID
    for i in (0, 3, 4, 5):
        assert call(i, None) == INVALID
        assert call(i, ctypes.c_void_p(0x10002)) == INVALID


def test_binding_refuses_host_tensors():
    import torch
    from quantize_amax_scaling_gb300 import fp8q
    x = torch.zeros(8, dtype=torch.bfloat16)
    q = torch.zeros(8, dtype=torch.uint8)
    s = torch.ones(1)
    with pytest.raises(ValueError):
        fp8q.fp8q_quantize_amax(x, q, fp8q.E4M3FN, s, s.clone())
    with pytest.raises(ValueError):
        fp8q.fp8q_dequantize(q, x, fp8q.E4M3FN, s)
    with pytest.raises(ValueError):
        fp8q.fp8q_amax_scale_update(torch.zeros(4, 2), s.expand(2), s.expand(2), s.expand(2))


def test_binding_refuses_tensors_on_another_device(monkeypatch):
    """The library launches on the current device: a tensor on another GPU is refused."""
    import types
    import torch
    from quantize_amax_scaling_gb300 import fp8q

    def fake(dtype, index):
        return types.SimpleNamespace(is_cuda=True, dtype=dtype, is_contiguous=lambda: True,
                                     device=torch.device("cuda", index), numel=lambda: 8)

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    fp8q._dev(fake(torch.bfloat16, 0), "bf16", "x")  # on the current device: accepted
    with pytest.raises(ValueError, match="current CUDA device"):
        fp8q._dev(fake(torch.bfloat16, 1), "bf16", "x")
    with pytest.raises(ValueError, match="current CUDA device"):
        fp8q.fp8q_quantize_amax(fake(torch.bfloat16, 0), fake(torch.uint8, 0), fp8q.E4M3FN,
                                fake(torch.float32, 1), fake(torch.float32, 0))


def test_tensor_list_refuses_host_tensors_and_other_devices(monkeypatch):
    """The multi-tensor list's one-pass checks refuse what the per-tensor checks refuse."""
    import types
    import torch
    from quantize_amax_scaling_gb300 import fp8q
    x = torch.zeros(8, dtype=torch.bfloat16)
    q = torch.zeros(8, dtype=torch.uint8)
    s = torch.ones(1)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fp8q.TensorList([x], [q], [s], [s.clone()])

    def fake(dtype, index, n=8):
        return types.SimpleNamespace(is_cuda=True, dtype=dtype, is_contiguous=lambda: True,
                                     device=torch.device("cuda", index), get_device=lambda: index,
                                     numel=lambda: n, data_ptr=lambda: 0x10000)

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    ok = fp8q.TensorList([fake(torch.bfloat16, 0)], [fake(torch.float8_e4m3fn, 0)], [fake(torch.float32, 0)],
                         [fake(torch.float32, 0)])
    assert ok.count == 1 and ok.array[0].n == 8
    with pytest.raises(ValueError, match="current CUDA device"):
        fp8q.TensorList([fake(torch.bfloat16, 0)], [fake(torch.uint8, 0)], [fake(torch.float32, 1)],
                        [fake(torch.float32, 0)])
    with pytest.raises(ValueError, match="dtype"):
        fp8q.TensorList([fake(torch.float16, 0)], [fake(torch.uint8, 0)], [fake(torch.float32, 0)],
                        [fake(torch.float32, 0)])
    with pytest.raises(ValueError, match="as many elements"):
        fp8q.TensorList([fake(torch.bfloat16, 0)], [fake(torch.uint8, 0, 9)], [fake(torch.float32, 0)],
                        [fake(torch.float32, 0)])


def test_product_code_never_touches_the_oracle():
    """The package (kernels, binding, build) neither imports, includes nor links the oracle."""
    pkg = os.path.join(ROOT, "quantize_amax_scaling_gb300")
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle|#\s*include\s*[<\"].*oracle)|fp8q_oracle|orc_",
                     re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not pat.search(text), f
