"""CPU oracle for FP8 delayed-scaling quantization -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It wraps ``fp8q_oracle.c`` (plain single-threaded C)
with numpy marshalling; it shares nothing with the CUDA library.

bf16 tensors are numpy ``uint16`` arrays of bit patterns; FP8 tensors are
``uint8`` code arrays.
"""
import ctypes
import os

import numpy as np

from . import build as _build

E4M3FN = 0
E5M2 = 1
ALGO_MAX = 0
ALGO_MOST_RECENT = 1

_lib = None


class _Tensor(ctypes.Structure):
    _fields_ = [("x_bf16", ctypes.c_void_p), ("q", ctypes.c_void_p), ("n", ctypes.c_int64),
                ("scale", ctypes.c_float), ("amax", ctypes.c_void_p)]


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        # FP8Q_ORACLE_LIB lets the mutation tests load a deliberately broken copy.
        path = os.environ.get("FP8Q_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f32.restype = f32
        L.orc_f32_to_bf16.argtypes = [f32]
        L.orc_f32_to_bf16.restype = ctypes.c_uint16
        L.orc_fp8_max_code.argtypes = [ctypes.c_int]
        L.orc_fp8_max_code.restype = ctypes.c_int
        L.orc_fp8_decode.argtypes = [ctypes.c_uint8, ctypes.c_int]
        L.orc_fp8_decode.restype = ctypes.c_double
        L.orc_fp8_max.argtypes = [ctypes.c_int]
        L.orc_fp8_max.restype = ctypes.c_double
        L.orc_fp8_encode.argtypes = [f32, ctypes.c_int]
        L.orc_fp8_encode.restype = ctypes.c_uint8
        L.orc_quantize_amax.argtypes = [vp, i64, ctypes.c_int, f32, vp, vp]
        L.orc_quantize_amax.restype = None
        L.orc_multi_quantize_amax.argtypes = [vp, i32, ctypes.c_int]
        L.orc_multi_quantize_amax.restype = None
        L.orc_amax.argtypes = [vp, i64]
        L.orc_amax.restype = f32
        L.orc_dequantize.argtypes = [vp, i64, ctypes.c_int, f32, vp]
        L.orc_dequantize.restype = None
        L.orc_qdq_amax.argtypes = [vp, i64, ctypes.c_int, f32, vp, vp]
        L.orc_qdq_amax.restype = None
        L.orc_exp_f32.argtypes = [f32]
        L.orc_exp_f32.restype = f32
        L.orc_gelu_f32.argtypes = [f32]
        L.orc_gelu_f32.restype = f32
        L.orc_gelu_quantize_amax.argtypes = [vp, i64, ctypes.c_int, f32, vp, vp, vp]
        L.orc_gelu_quantize_amax.restype = None
        L.orc_layernorm_stats.argtypes = [vp, i32, f32, vp, vp]
        L.orc_layernorm_stats.restype = None
        L.orc_layernorm_quantize_amax.argtypes = [vp, i64, i32, vp, vp, f32, ctypes.c_int, f32, vp, vp, vp]
        L.orc_layernorm_quantize_amax.restype = None
        L.orc_gelu_amax.argtypes = [vp, i64]
        L.orc_gelu_amax.restype = f32
        L.orc_amax_scale_update.argtypes = [vp, i32, i32, vp, vp, vp, vp, ctypes.c_int,
                                            ctypes.c_int, i32]
        L.orc_amax_scale_update.restype = None
        L.orc_amax_scale_update_ring.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, ctypes.c_int,
                                                 ctypes.c_int, i32]
        L.orc_amax_scale_update_ring.restype = None
        _lib = L
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c_u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def bf16_to_f32(h):
    """bf16 bit patterns -> float32 values (exact)."""
    return float(lib().orc_bf16_to_f32(int(h)))


def f32_to_bf16(f):
    """float32 value -> nearest bf16 bit pattern (ties to even)."""
    return int(lib().orc_f32_to_bf16(float(np.float32(f))))


def fp8_decode(code, fmt):
    return lib().orc_fp8_decode(int(code), fmt)


def fp8_max(fmt):
    return lib().orc_fp8_max(fmt)


def fp8_max_code(fmt):
    return lib().orc_fp8_max_code(fmt)


def fp8_encode(y, fmt):
    return int(lib().orc_fp8_encode(float(np.float32(y)), fmt))


def quantize_amax(x_bf16, fmt, scale, amax=0.0):
    """Return (q uint8 array, amax float32) for one bf16 tensor."""
    x = _c_u16(x_bf16).reshape(-1)
    q = np.empty(x.shape, np.uint8)
    a = np.array([amax], np.float32)
    lib().orc_quantize_amax(_ptr(x), x.size, fmt, float(np.float32(scale)), _ptr(q), _ptr(a))
    return q, np.float32(a[0])


def multi_quantize_amax(xs, fmt, scales, amaxes=None):
    """Ragged list: returns ([q arrays], [amax values])."""
    xs = [_c_u16(x).reshape(-1) for x in xs]
    qs = [np.empty(x.shape, np.uint8) for x in xs]
    am = np.array(amaxes if amaxes is not None else [0.0] * len(xs), np.float32)
    arr = (_Tensor * max(1, len(xs)))()
    for i, x in enumerate(xs):
        arr[i].x_bf16 = x.ctypes.data
        arr[i].q = qs[i].ctypes.data
        arr[i].n = x.size
        arr[i].scale = float(np.float32(scales[i]))
        arr[i].amax = am.ctypes.data + 4 * i
    lib().orc_multi_quantize_amax(ctypes.cast(arr, ctypes.c_void_p), len(xs), fmt)
    return qs, [np.float32(v) for v in am]


def amax(x_bf16):
    x = _c_u16(x_bf16).reshape(-1)
    return np.float32(lib().orc_amax(_ptr(x), x.size))


def dequantize(q, fmt, scale):
    """Return the bf16 bit patterns of DQ(q)."""
    q = np.ascontiguousarray(q, dtype=np.uint8).reshape(-1)
    y = np.empty(q.shape, np.uint16)
    lib().orc_dequantize(_ptr(q), q.size, fmt, float(np.float32(scale)), _ptr(y))
    return y


def qdq_amax(x_bf16, fmt, scale, amax=0.0):
    """Return (bf16 bits of DQ(Q(x)), amax float32) for one bf16 tensor."""
    x = _c_u16(x_bf16).reshape(-1)
    y = np.empty(x.shape, np.uint16)
    a = np.array([amax], np.float32)
    lib().orc_qdq_amax(_ptr(x), x.size, fmt, float(np.float32(scale)), _ptr(y), _ptr(a))
    return y, np.float32(a[0])


def amax_scale_update(hist, amax_new, scale, scale_inv, fmt=E4M3FN, algo=ALGO_MAX, margin=0,
                      slot_format=None):
    """In-place update of float32 arrays hist[H][S], scale[S], scale_inv[S]."""
    assert hist.dtype == np.float32 and hist.flags.c_contiguous and hist.ndim == 2
    H, S = hist.shape
    amax_new = np.ascontiguousarray(amax_new, np.float32)
    for a in (scale, scale_inv):
        assert a.dtype == np.float32 and a.flags.c_contiguous and a.size == S
    sf = None if slot_format is None else np.ascontiguousarray(slot_format, np.uint8)
    lib().orc_amax_scale_update(_ptr(hist), H, S, _ptr(amax_new), _ptr(scale), _ptr(scale_inv),
                                _ptr(sf), fmt, algo, margin)


def amax_scale_update_ring(hist, head, amax_new, scale, scale_inv, fmt=E4M3FN, algo=ALGO_MAX,
                           margin=0, slot_format=None):
    """In-place ring-buffer update of hist[H][S], head[S] (int32), scale[S], scale_inv[S]."""
    assert hist.dtype == np.float32 and hist.flags.c_contiguous and hist.ndim == 2
    H, S = hist.shape
    assert head.dtype == np.int32 and head.flags.c_contiguous and head.size == S
    amax_new = np.ascontiguousarray(amax_new, np.float32)
    sf = None if slot_format is None else np.ascontiguousarray(slot_format, np.uint8)
    lib().orc_amax_scale_update_ring(_ptr(hist), _ptr(head), H, S, _ptr(amax_new), _ptr(scale),
                                     _ptr(scale_inv), _ptr(sf), fmt, algo, margin)


def amax_scale_update_ring_quantize(hist, head, amax_new, scale, scale_inv, x_bf16, slot, fmt=E4M3FN,
                                    algo=ALGO_MAX, margin=0, slot_format=None, amax=0.0):
    """The update fused with the next quantize, by its definition: the ring
    update of every slot (in place on hist, head, scale, scale_inv), then the
    quantize of x with slot `slot`'s scale after the update.  Returns (q, amax)."""
    amax_scale_update_ring(hist, head, amax_new, scale, scale_inv, fmt, algo, margin, slot_format)
    return quantize_amax(x_bf16, fmt, scale[slot], amax)


def exp_f32(v):
    return np.float32(lib().orc_exp_f32(float(np.float32(v))))


def gelu_f32(x):
    return np.float32(lib().orc_gelu_f32(float(np.float32(x))))


def gelu_quantize_amax(h_bf16, fmt, scale, amax=0.0):
    """Return (q codes, bf16 bits of y = GELU(h), amax float32)."""
    h = _c_u16(h_bf16).reshape(-1)
    q = np.empty(h.shape, np.uint8)
    y = np.empty(h.shape, np.uint16)
    a = np.array([amax], np.float32)
    lib().orc_gelu_quantize_amax(_ptr(h), h.size, fmt, float(np.float32(scale)), _ptr(q), _ptr(y), _ptr(a))
    return q, y, np.float32(a[0])


def gelu_amax(h_bf16):
    """max|bf16(GELU(h))| over the whole tensor."""
    h = _c_u16(h_bf16).reshape(-1)
    return np.float32(lib().orc_gelu_amax(_ptr(h), h.size))


def layernorm_stats(row_bf16, eps=1e-6):
    """(mean, rstd) of one bf16 row, in the fixed summation order."""
    r = _c_u16(row_bf16).reshape(-1)
    m = np.zeros(1, np.float32)
    rs = np.zeros(1, np.float32)
    lib().orc_layernorm_stats(_ptr(r), r.size, float(np.float32(eps)), _ptr(m), _ptr(rs))
    return m[0], rs[0]


def layernorm_quantize_amax(x_bf16, H, gamma, beta, fmt, scale, eps=1e-6, amax=0.0):
    """Return (q codes, bf16 bits of y = LayerNorm(x), amax) for rows of H elements."""
    x = _c_u16(x_bf16).reshape(-1)
    assert x.size % H == 0
    g = np.ascontiguousarray(gamma, np.float32)
    b = np.ascontiguousarray(beta, np.float32)
    q = np.empty(x.shape, np.uint8)
    y = np.empty(x.shape, np.uint16)
    a = np.array([amax], np.float32)
    lib().orc_layernorm_quantize_amax(_ptr(x), x.size // H, H, _ptr(g), _ptr(b), float(np.float32(eps)), fmt,
                                      float(np.float32(scale)), _ptr(q), _ptr(y), _ptr(a))
    return q, y, np.float32(a[0])
