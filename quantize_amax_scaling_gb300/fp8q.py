"""Thin Python binding of libfp8q's C ABI (include/fp8q.h).

Argument marshalling only: every step of the FP8 path runs in the CUDA
kernels of libfp8q.so.  Tensors are torch CUDA tensors (torch supplies device
memory and streams); the functions keep the C names and raise Fp8qError on a
non-OK status.  If the library has not been built, loading fails loudly --
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

E4M3FN = 0
E5M2 = 1
ALGO_MAX = 0
ALGO_MOST_RECENT = 1
MAX_TENSORS = 512

STATUS = {0: "FP8Q_OK", 1: "FP8Q_ERR_INVALID_ARG", 2: "FP8Q_ERR_UNSUPPORTED", 3: "FP8Q_ERR_CUDA",
          4: "FP8Q_ERR_TOO_MANY_TENSORS"}

# Every symbol the header declares.
EXPORTS = ("fp8q_quantize_amax", "fp8q_multi_quantize_amax", "fp8q_dequantize",
           "fp8q_amax_scale_update", "fp8q_qdq_amax", "fp8q_amax_scale_update_ring",
           "fp8q_gelu_quantize_amax", "fp8q_layernorm_quantize_amax",
           "fp8q_amax_scale_update_ring_quantize", "fp8q_status_string",
           "fp8q_last_cuda_error")

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfp8q.so")


class Fp8qError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


class Tensor(ctypes.Structure):
    """fp8q_tensor: one entry of a ragged list."""
    _fields_ = [("x_bf16", ctypes.c_void_p), ("q", ctypes.c_void_p), ("n", ctypes.c_int64),
                ("scale", ctypes.c_void_p), ("amax", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libfp8q.so (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
        L.fp8q_quantize_amax.argtypes = [vp, vp, i64, c_int, vp, vp, vp]
        L.fp8q_multi_quantize_amax.argtypes = [vp, i32, c_int, vp]
        L.fp8q_dequantize.argtypes = [vp, vp, i64, c_int, vp, vp]
        L.fp8q_amax_scale_update.argtypes = [vp, i32, i32, vp, vp, vp, vp, c_int, c_int, i32, vp]
        L.fp8q_qdq_amax.argtypes = [vp, vp, i64, c_int, vp, vp, vp]
        L.fp8q_amax_scale_update_ring.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, c_int, c_int, i32,
                                                  vp]
        L.fp8q_gelu_quantize_amax.argtypes = [vp, vp, vp, i64, c_int, vp, vp, vp]
        L.fp8q_layernorm_quantize_amax.argtypes = [vp, vp, vp, i64, i32, vp, vp, ctypes.c_float, c_int,
                                                   vp, vp, vp]
        L.fp8q_amax_scale_update_ring_quantize.argtypes = [vp, vp, vp, i32, i32, vp, vp, vp, vp, c_int, c_int,
                                                           i32, vp, vp, i64, i32, vp, vp]
        for f in ("fp8q_quantize_amax", "fp8q_multi_quantize_amax", "fp8q_dequantize",
                  "fp8q_amax_scale_update", "fp8q_qdq_amax", "fp8q_amax_scale_update_ring",
                  "fp8q_gelu_quantize_amax", "fp8q_layernorm_quantize_amax",
                  "fp8q_amax_scale_update_ring_quantize"):
            getattr(L, f).restype = c_int
        L.fp8q_status_string.argtypes = [c_int]
        L.fp8q_status_string.restype = ctypes.c_char_p
        L.fp8q_last_cuda_error.argtypes = []
        L.fp8q_last_cuda_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != 0:
        detail = lib().fp8q_last_cuda_error().decode() if status == 3 else ""
        raise Fp8qError(status, where, detail)


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


_FP8_DTYPES = None


def _dev(t, kind, name):
    """Reject anything but a contiguous CUDA tensor of the right element type
    on the current CUDA device.

    Pointers reach the kernels unchanged, so a host tensor must never get
    through, and the library launches on the current device, so a tensor on
    another GPU must not either.  ``kind`` is "bf16", "u8" (uint8 or a float8
    dtype), "f32" or "i32".
    """
    global _FP8_DTYPES
    if _FP8_DTYPES is None:
        import torch
        _FP8_DTYPES = (torch.uint8, torch.float8_e4m3fn, torch.float8_e5m2)
    if t is None:
        return
    import torch
    ok = {"bf16": (torch.bfloat16,), "u8": _FP8_DTYPES, "f32": (torch.float32,),
          "i32": (torch.int32,)}[kind]
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in ok:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {ok}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    cur = torch.cuda.current_device()
    if t.device.index != cur:
        raise ValueError(f"{name} is on {t.device} but the current CUDA device is cuda:{cur}; "
                         "the kernels launch on the current device (wrap the call in torch.cuda.device)")


def _numel(t):
    return 0 if t is None else t.numel()


def fp8q_quantize_amax(x, q, fmt, scale, amax, stream=None):
    """q = FP8(x / scale) (saturating RNE) and amax = max(amax, max|x|) in one launch."""
    n = _numel(x)
    if q is not None and _numel(q) != n:
        raise ValueError("q must have as many elements as x")
    for t, k, nm in ((x, "bf16", "x"), (q, "u8", "q"), (scale, "f32", "scale"), (amax, "f32", "amax")):
        _dev(t, k, nm)
    _check(lib().fp8q_quantize_amax(_ptr(x), _ptr(q), n, fmt, _ptr(scale), _ptr(amax),
                                    _stream(stream)), "fp8q_quantize_amax")


def fp8q_qdq_amax(x, y, fmt, scale, amax, stream=None):
    """y = DQ(Q(x)) in bf16 and amax = max(amax, max|x|) in one launch (y may be x)."""
    n = _numel(x)
    if y is not None and _numel(y) != n:
        raise ValueError("y must have as many elements as x")
    for t, k, nm in ((x, "bf16", "x"), (y, "bf16", "y"), (scale, "f32", "scale"), (amax, "f32", "amax")):
        _dev(t, k, nm)
    _check(lib().fp8q_qdq_amax(_ptr(x), _ptr(y), n, fmt, _ptr(scale), _ptr(amax), _stream(stream)),
           "fp8q_qdq_amax")


def fp8q_gelu_quantize_amax(h, y, q, fmt, scale, amax, stream=None):
    """y = bf16(GELU(h)) (y may be None), q = FP8(y / scale), amax = max(amax, max|y|), one launch."""
    n = _numel(h)
    for t, nm in ((y, "y"), (q, "q")):
        if t is not None and _numel(t) != n:
            raise ValueError(f"{nm} must have as many elements as h")
    for t, k, nm in ((h, "bf16", "h"), (y, "bf16", "y"), (q, "u8", "q"), (scale, "f32", "scale"),
                     (amax, "f32", "amax")):
        _dev(t, k, nm)
    _check(lib().fp8q_gelu_quantize_amax(_ptr(h), _ptr(y), _ptr(q), n, fmt, _ptr(scale), _ptr(amax),
                                         _stream(stream)), "fp8q_gelu_quantize_amax")


def fp8q_layernorm_quantize_amax(x, y, q, gamma, beta, fmt, scale, amax, eps=1e-6, stream=None):
    """y = bf16(LayerNorm(x) * gamma + beta) (y may be None), q = FP8(y / scale),
    amax = max(amax, max|y|), one launch.

    ``x`` is bf16 [rows, hidden]; ``gamma`` and ``beta`` are float32 [hidden].
    """
    if x.dim() != 2:
        raise ValueError("x must be [rows, hidden]")
    rows, hidden = x.shape
    for t, nm in ((y, "y"), (q, "q")):
        if t is not None and _numel(t) != rows * hidden:
            raise ValueError(f"{nm} must have as many elements as x")
    for t, nm in ((gamma, "gamma"), (beta, "beta")):
        if _numel(t) != hidden:
            raise ValueError(f"{nm} must have hidden={hidden} elements")
    for t, k, nm in ((x, "bf16", "x"), (y, "bf16", "y"), (q, "u8", "q"), (gamma, "f32", "gamma"),
                     (beta, "f32", "beta"), (scale, "f32", "scale"), (amax, "f32", "amax")):
        _dev(t, k, nm)
    _check(lib().fp8q_layernorm_quantize_amax(_ptr(x), _ptr(y), _ptr(q), rows, hidden, _ptr(gamma),
                                              _ptr(beta), float(eps), fmt, _ptr(scale), _ptr(amax),
                                              _stream(stream)), "fp8q_layernorm_quantize_amax")


class TensorList:
    """A ragged list checked and marshalled once into the ``fp8q_tensor`` array that
    ``fp8q_multi_quantize_amax`` takes.

    ``scales`` and ``amaxes`` are sequences of one-element float32 tensors (or views
    into one vector) aligned with ``xs``.  Passing a TensorList instead of the four
    sequences skips the per-tensor checks on every call, which for hundreds of small
    tensors take longer than the launch itself.  The list keeps the tensors alive; it
    reads their storage when called, so tensors resized or replaced since it was built
    need a new list.
    """

    def __init__(self, xs, qs, scales, amaxes):
        count = len(xs)
        if not (len(qs) == len(scales) == len(amaxes) == count):
            raise ValueError("xs, qs, scales and amaxes must have the same length")
        import torch
        _dev(None, "bf16", "")
        cur = None
        kinds = ((torch.bfloat16,), _FP8_DTYPES, (torch.float32,), (torch.float32,))
        arr = (Tensor * max(1, count))()
        for i in range(count):
            ts = (xs[i], qs[i], scales[i], amaxes[i])
            for t, ok, k, nm in zip(ts, kinds, ("bf16", "u8", "f32", "f32"), ("x", "q", "scale", "amax")):
                if t is None:
                    raise ValueError(f"{nm}[{i}] is None")
                # the common case in one expression; anything else gets _dev's message
                if t.dtype not in ok or not t.is_cuda or not t.is_contiguous():
                    _dev(t, k, f"{nm}[{i}]")
                if cur is None:
                    cur = torch.cuda.current_device()
                if t.get_device() != cur:
                    _dev(t, k, f"{nm}[{i}]")
            n = ts[0].numel()
            if ts[1].numel() != n:
                raise ValueError(f"tensor {i}: q must have as many elements as x")
            arr[i].x_bf16 = ts[0].data_ptr()
            arr[i].q = ts[1].data_ptr()
            arr[i].n = n
            arr[i].scale = ts[2].data_ptr()
            arr[i].amax = ts[3].data_ptr()
        self.count = count
        self.array = arr
        self.address = ctypes.cast(arr, ctypes.c_void_p)
        self._keep = (list(xs), list(qs), list(scales), list(amaxes))


def fp8q_multi_quantize_amax(xs, qs=None, fmt=E4M3FN, scales=None, amaxes=None, stream=None):
    """fp8q_quantize_amax over a ragged list of tensors, one launch.

    Either the four aligned sequences (xs, qs, scales, amaxes: see TensorList),
    checked on every call, or a TensorList built once as ``xs`` (leave qs, scales
    and amaxes out).
    """
    if isinstance(xs, TensorList):
        if qs is not None or scales is not None or amaxes is not None:
            raise ValueError("pass either a TensorList or xs, qs, scales and amaxes")
        tl = xs
    else:
        tl = TensorList(xs, qs, scales, amaxes)
    _check(lib().fp8q_multi_quantize_amax(tl.address, tl.count, fmt, _stream(stream)),
           "fp8q_multi_quantize_amax")


def fp8q_dequantize(q, y, fmt, scale, stream=None):
    """y = bf16_rne(float(q) * scale)."""
    n = _numel(q)
    if y is not None and _numel(y) != n:
        raise ValueError("y must have as many elements as q")
    for t, k, nm in ((q, "u8", "q"), (y, "bf16", "y"), (scale, "f32", "scale")):
        _dev(t, k, nm)
    _check(lib().fp8q_dequantize(_ptr(q), _ptr(y), n, fmt, _ptr(scale), _stream(stream)),
           "fp8q_dequantize")


def fp8q_amax_scale_update(history, amax_new, scale, scale_inv, fmt=E4M3FN, algo=ALGO_MAX,
                           margin=0, slot_format=None, stream=None):
    """In-place amax-history roll, amax selection and scale/scale_inv update.

    ``history`` is a float32 [history_len, num_slots] tensor, row 0 newest.
    """
    if history.dim() != 2:
        raise ValueError("history must be [history_len, num_slots]")
    H, S = history.shape
    for t, k, nm in ((history, "f32", "history"), (amax_new, "f32", "amax_new"),
                     (scale, "f32", "scale"), (scale_inv, "f32", "scale_inv"),
                     (slot_format, "u8", "slot_format")):
        _dev(t, k, nm)
    for t, nm in ((amax_new, "amax_new"), (scale, "scale"), (scale_inv, "scale_inv"),
                  (slot_format, "slot_format")):
        if t is not None and t.numel() != S:
            raise ValueError(f"{nm} must have num_slots={S} elements")
    _check(lib().fp8q_amax_scale_update(_ptr(history), H, S, _ptr(amax_new), _ptr(scale),
                                        _ptr(scale_inv), _ptr(slot_format), fmt, algo, margin,
                                        _stream(stream)), "fp8q_amax_scale_update")


def fp8q_amax_scale_update_ring(history, head, amax_new, scale, scale_inv, fmt=E4M3FN,
                                algo=ALGO_MAX, margin=0, slot_format=None, stream=None):
    """Ring-buffer amax history update: overwrite each slot's oldest row, advance head.

    ``history`` is float32 [history_len, num_slots]; ``head`` is int32 [num_slots],
    the row of each slot's newest entry.
    """
    if history.dim() != 2:
        raise ValueError("history must be [history_len, num_slots]")
    H, S = history.shape
    for t, k, nm in ((history, "f32", "history"), (head, "i32", "head"), (amax_new, "f32", "amax_new"),
                     (scale, "f32", "scale"), (scale_inv, "f32", "scale_inv"),
                     (slot_format, "u8", "slot_format")):
        if t is None and nm == "head":
            raise ValueError("head must be a contiguous int32 CUDA tensor")
        _dev(t, k, nm)
    for t, nm in ((head, "head"), (amax_new, "amax_new"), (scale, "scale"), (scale_inv, "scale_inv"),
                  (slot_format, "slot_format")):
        if t is not None and t.numel() != S:
            raise ValueError(f"{nm} must have num_slots={S} elements")
    _check(lib().fp8q_amax_scale_update_ring(_ptr(history), _ptr(head), H, S, _ptr(amax_new),
                                             _ptr(scale), _ptr(scale_inv), _ptr(slot_format), fmt,
                                             algo, margin, _stream(stream)),
           "fp8q_amax_scale_update_ring")


def fp8q_amax_scale_update_ring_quantize(history, head_in, head_out, amax_new, scale, scale_inv, x, q, slot,
                                         amax, fmt=E4M3FN, algo=ALGO_MAX, margin=0, slot_format=None,
                                         stream=None):
    """The ring-buffer update of every slot, then q = FP8(x / scale[slot]) with the
    new scale and amax = max(amax, max|x|), in one launch.  head_in is read,
    head_out written (two int32 [num_slots] arrays, swapped between steps)."""
    if history.dim() != 2:
        raise ValueError("history must be [history_len, num_slots]")
    H, S = history.shape
    n = _numel(x)
    if q is not None and _numel(q) != n:
        raise ValueError("q must have as many elements as x")
    for t, k, nm in ((history, "f32", "history"), (amax_new, "f32", "amax_new"), (scale, "f32", "scale"),
                     (scale_inv, "f32", "scale_inv"), (slot_format, "u8", "slot_format"), (x, "bf16", "x"),
                     (q, "u8", "q"), (amax, "f32", "amax")):
        _dev(t, k, nm)
    for t, nm in ((head_in, "head_in"), (head_out, "head_out")):
        if t is None:
            raise ValueError(f"{nm} must be a contiguous int32 CUDA tensor")
        _dev(t, "i32", nm)
    for t, nm in ((head_in, "head_in"), (head_out, "head_out"), (amax_new, "amax_new"), (scale, "scale"),
                  (scale_inv, "scale_inv"), (slot_format, "slot_format")):
        if t is not None and t.numel() != S:
            raise ValueError(f"{nm} must have num_slots={S} elements")
    _check(lib().fp8q_amax_scale_update_ring_quantize(
        _ptr(history), _ptr(head_in), _ptr(head_out), H, S, _ptr(amax_new), _ptr(scale), _ptr(scale_inv),
        _ptr(slot_format), fmt, algo, margin, _ptr(x), _ptr(q), n, slot, _ptr(amax), _stream(stream)),
        "fp8q_amax_scale_update_ring_quantize")


def status_string(status: int) -> str:
    return lib().fp8q_status_string(status).decode()
