"""CPU oracle for FP8 delayed-scaling quantization -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It wraps ``fp8q_oracle.c`` (plain single-threaded C)
with numpy marshalling; it shares nothing with the CUDA library.

bf16 tensors are numpy ``uint16`` arrays of bit patterns; FP8 tensors are
``uint8`` code arrays.
"""
import ctypes
import math
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
        L.orc_f64_to_bf16.argtypes = [ctypes.c_double]
        L.orc_f64_to_bf16.restype = ctypes.c_uint16
        L.orc_f64_to_bf16_array.argtypes = [vp, i64, vp]
        L.orc_f64_to_bf16_array.restype = None
        L.orc_gelu_ref.argtypes = [ctypes.c_double]
        L.orc_gelu_ref.restype = ctypes.c_double
        L.orc_gelu_ref_array.argtypes = [vp, i64, vp]
        L.orc_gelu_ref_array.restype = None
        L.orc_layernorm_ref.argtypes = [vp, i64, i32, vp, vp, ctypes.c_double, vp, vp, vp]
        L.orc_layernorm_ref.restype = None
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


def f64_to_bf16(g):
    """float64 value -> nearest bf16 bit pattern (ties to even), one rounding."""
    return int(lib().orc_f64_to_bf16(float(g)))


def gelu_ref(x):
    """GELU (tanh form) of one value in float64."""
    return float(lib().orc_gelu_ref(float(x)))


def gelu_ref_array(h_bf16):
    """GELU (tanh form) in float64 of every bf16 input."""
    h = _c_u16(h_bf16).reshape(-1)
    g = np.empty(h.shape, np.float64)
    lib().orc_gelu_ref_array(_ptr(h), h.size, _ptr(g))
    return g


def layernorm_ref(x_bf16, H, gamma, beta, eps=1e-6):
    """LayerNorm (Flax defaults) in float64 of rows of H bf16 values.

    Returns (y float64 [rows*H], mean float64 [rows], rstd float64 [rows])."""
    x = _c_u16(x_bf16).reshape(-1)
    assert x.size % H == 0
    rows = x.size // H
    g = np.ascontiguousarray(gamma, np.float32)
    b = np.ascontiguousarray(beta, np.float32)
    y = np.empty(x.size, np.float64)
    mean = np.empty(rows, np.float64)
    rstd = np.empty(rows, np.float64)
    lib().orc_layernorm_ref(_ptr(x), rows, H, _ptr(g), _ptr(b), float(eps), _ptr(y), _ptr(mean), _ptr(rstd))
    return y, mean, rstd


# --------------------------------------------------------------------------- producer tolerances
#
# The fused producers compute in binary32 and round to bf16; the definitions
# above are float64.  A kernel's y is accepted when it is the bf16 rounding of
# some value within E of the float64 value r: RN(r - E) <= y <= RN(r + E)
# (RN is monotone).  Wherever r lies farther than E from every bf16 rounding
# boundary, that leaves exactly one value, RN(r).  E is derived from the
# binary32 arithmetic below; u = 2^-24 is binary32's unit roundoff.

U32 = 2.0 ** -24
GELU_TINY = 2.0 ** -122


def gelu_tolerance(h_f64, r):
    """E for y = bf16(GELU(h)) evaluated in binary32.

    The binary32 evaluation x / (1 + e^v), v = -2 sqrt(2/pi) x (1 + 0.044715 x^2):
    v carries at most 6u relative error (the constants' roundings and three
    operations), so e^v carries 6u|v| from its argument plus at most 7u of
    its own (range reduction, a degree-6 polynomial whose truncation stays
    under 3u, Horner roundings); 1 + e^v, the reciprocal and the final
    product add u each.  So |error| <= (6|v| + 10) u |GELU| while
    1 / (1 + e^v) is a normal binary32.  Where |GELU| < 2^-122 that
    reciprocal is subnormal or zero (|x| <= 10.6 there), and y may be any
    value within 2^-122 of r.  At x = +inf the result is +inf exactly (E = 0).
    """
    h = np.asarray(h_f64, np.float64)
    r = np.asarray(r, np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        v = np.minimum(np.abs(2.0 * math.sqrt(2.0 / math.pi) * h * (1.0 + 0.044715 * h * h)), 89.0)
    v = np.where(np.isfinite(v), v, 89.0)
    with np.errstate(invalid="ignore"):
        e = np.where(np.isinf(r), 0.0, (6.0 * v + 10.0) * U32 * np.abs(r))   # GELU(+inf) = +inf exactly
    return np.where(np.abs(r) < GELU_TINY, np.maximum(e, GELU_TINY), e)


def layernorm_chain_bound(H):
    """D: the longest chain of binary32 additions in either row sum that the
    tolerance below allows (H / 128 + 32)."""
    return H // 128 + 32


def layernorm_tolerance(x_f64, gamma, beta, eps, mean, rstd, r):
    """E for y = bf16(LayerNorm(x) * gamma + beta) evaluated in binary32.

    x_f64 [rows, H]; mean, rstd [rows] and r [rows, H] from layernorm_ref.
    The binary32 evaluation sums S = sum x and Q = sum x^2 (each x^2 exact)
    in any order whose longest chain has at most D additions, so
    |dS| <= g sum|x| and |dQ| <= g Q with g = D u / (1 - D u).  Then
    mean = S / H, mean^2, Q / H and their difference add one rounding each
    (dmean, dvar below, to first order in u, with the squares kept); the
    variance error bounds rstd = 1 / sqrt(var + eps) through the exact
    interval 1 / sqrt(var +- dvar + eps), and the square root and
    reciprocal add at most 4u.  Each element then takes x - mean,
    rstd * gamma and the product and sum with beta: at most 3u on
    t = (x - mean) rstd gamma and u on |y| and |beta| each.  A factor 1.01
    covers the neglected second-order terms.
    Rows outside binary32's range for these sums (a non-finite x, Q over
    2^126, var + eps under 2^-100) have no bound: E = inf there.
    """
    x = np.asarray(x_f64, np.float64)
    rows, H = x.shape
    D = layernorm_chain_bound(H)
    g = D * U32 / (1.0 - D * U32)
    ax = np.abs(x)
    A = ax.mean(axis=1)
    M2 = (x * x).mean(axis=1)
    mean = np.asarray(mean, np.float64)
    var = np.maximum(M2 - mean * mean, 0.0)
    dmean = g * A + U32 * (np.abs(mean) + g * A)
    dm2 = g * M2 + U32 * M2 * (1.0 + g)
    dsq = 2.0 * np.abs(mean) * dmean + dmean ** 2 + U32 * (np.abs(mean) + dmean) ** 2
    dvar = dm2 + dsq + U32 * (var + dm2 + dsq)
    lo = np.maximum(var - dvar, 0.0) + eps
    hi = var + dvar + eps
    e_rho = np.maximum(np.sqrt((var + eps) / lo) - 1.0, 1.0 - np.sqrt((var + eps) / hi)) + 4.0 * U32
    gam = np.abs(np.asarray(gamma, np.float64))[None, :]
    bet = np.abs(np.asarray(beta, np.float64))[None, :]
    rs = np.asarray(rstd, np.float64)[:, None]
    t = np.abs(x - mean[:, None]) * rs * gam
    E = 1.01 * (dmean[:, None] * rs * gam + t * (e_rho[:, None] + 3.0 * U32)
                + U32 * (np.abs(np.asarray(r, np.float64).reshape(rows, H)) + bet))
    bad = ~np.isfinite(x).all(axis=1) | (M2 * H > 2.0 ** 126) | (var + eps < 2.0 ** -100)
    E[bad] = np.inf
    return E


def f64_to_bf16_array(v):
    """Nearest bf16 (ties to even) of each float64 value, one rounding."""
    v = np.ascontiguousarray(v, np.float64).reshape(-1)
    out = np.empty(v.shape, np.uint16)
    lib().orc_f64_to_bf16_array(_ptr(v), v.size, _ptr(out))
    return out


def _bf16_order_key(bits):
    """Integer key in which bf16 values order like the numbers (-0 equal to +0)."""
    b = np.asarray(bits, np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_within(y_bits, r, E):
    """Boolean mask: y is the bf16 rounding of some value in [r - E, r + E].

    y_bits are bf16 patterns, r and E float64 of the same size.  A NaN r
    accepts exactly the NaN patterns; E = inf accepts anything.
    """
    y = np.asarray(y_bits, np.uint16).reshape(-1)
    r = np.asarray(r, np.float64).reshape(-1)
    E = np.asarray(E, np.float64).reshape(-1)
    ynan = ((y & 0x7F80) == 0x7F80) & ((y & 0x7F) != 0)
    rnan = np.isnan(r)
    ok = np.zeros(y.shape, bool)
    inf = np.isinf(E)
    ok[inf] = True
    ok[rnan & ~inf] = ynan[rnan & ~inf]
    m = ~inf & ~rnan
    lo = f64_to_bf16_array(r[m] - E[m])
    hi = f64_to_bf16_array(r[m] + E[m])
    k = _bf16_order_key(y[m])
    ok[m] = ~ynan[m] & (k >= _bf16_order_key(lo)) & (k <= _bf16_order_key(hi))
    return ok
