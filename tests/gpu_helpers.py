"""Helpers shared by the GPU parity tests: exact comparisons, canary-guarded
buffers, and the oracle run over every host core for full-size compares.

The path is elementwise and amax is a max, so splitting a tensor into
contiguous chunks, running the oracle on each (ctypes releases the GIL during
the C call) and combining the amaxes gives exactly the single call's results.
"""
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle

E4M3FN, E5M2 = 0, 1
GUARD = 64
CANARY = 0xA5

SCALES_ALL = [1.0, 0.5, 2.0 ** -6, 2.0 ** 20, 1.0 / 3.0, 0.012345678, 7.5, 448.0 / 3.9, 3.0e-5,
              1.7e4, 2.0 ** -60, 2.0 ** 60, float.fromhex("0x1.fffffep-61"), float.fromhex("0x1.000002p60"), 2.0 ** -70, 2.0 ** 70,
              1.0e-38, 5.0e-45, -2.5, 0.0, -0.0, math.inf, math.nan, 3.4e38, float.fromhex("0x1.fffffep-1"),
              float.fromhex("0x1.000002p0"), 1.0 / 448.0, 57344.0]

HOST_THREADS = max(1, os.cpu_count() or 1)
CHUNK = 1 << 22


def f32(v, dev):
    return torch.tensor([v], dtype=torch.float32, device=dev)


def is_nan_code(c, fmt):
    c = np.asarray(c) & 0x7F
    return c == 0x7F if fmt == E4M3FN else c > 0x7C


def assert_codes_equal(got, want, fmt, what=""):
    got = np.asarray(got, np.uint8).reshape(-1)
    want = np.asarray(want, np.uint8).reshape(-1)
    assert got.shape == want.shape
    nan_w = is_nan_code(want, fmt)
    assert np.array_equal(is_nan_code(got, fmt), nan_w), f"{what}: NaN codes differ"
    bad = np.nonzero((got != want) & ~nan_w)[0]
    assert bad.size == 0, f"{what}: {bad.size} codes differ, first at {bad[:5]}: got {got[bad[:5]]} want {want[bad[:5]]}"


def assert_f32_equal(got, want, what=""):
    g = np.asarray(got, np.float32).reshape(-1)
    w = np.asarray(want, np.float32).reshape(-1)
    gn, wn = np.isnan(g), np.isnan(w)
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
    bad = np.nonzero((g.view(np.uint32) != w.view(np.uint32)) & ~wn)[0]
    assert bad.size == 0, f"{what}: {bad.size} differ, first {bad[:5]}: got {g[bad[:5]]} want {w[bad[:5]]}"


def bf16_nan(bits):
    b = np.asarray(bits, np.uint16)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)


def assert_bf16_equal(got_bits, want_bits, what=""):
    g = np.asarray(got_bits, np.uint16).reshape(-1)
    w = np.asarray(want_bits, np.uint16).reshape(-1)
    gn, wn = bf16_nan(g), bf16_nan(w)
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
    bad = np.nonzero((g != w) & ~wn)[0]
    assert bad.size == 0, f"{what}: {bad.size} differ, first {bad[:5]}: got {g[bad[:5]]} want {w[bad[:5]]}"


def guarded(n, dtype, dev, offset=0, fill=CANARY):
    """A contiguous view of n elements inside a buffer with canary guards on both sides."""
    buf = torch.full((n + 2 * GUARD + offset,), fill, dtype=torch.uint8 if dtype == torch.uint8 else torch.int16,
                     device=dev)
    if dtype != torch.uint8:
        buf = buf.view(dtype)
    return buf, buf[GUARD + offset: GUARD + offset + n]


def check_guards(buf, n, offset, fill=CANARY):
    raw = buf.view(torch.uint8) if buf.dtype != torch.uint8 else buf
    es = buf.element_size()
    lo = raw[: (GUARD + offset) * es].cpu().numpy()
    hi = raw[(GUARD + offset + n) * es:].cpu().numpy()
    if buf.dtype == torch.uint8:
        assert np.all(lo == fill) and np.all(hi == fill), "write outside the output"
    else:
        lo16 = lo.view(np.uint16)
        hi16 = hi.view(np.uint16)
        assert np.all(lo16 == fill) and np.all(hi16 == fill), "write outside the output"


def oracle_scale_from(amax_prev, fmt):
    """Delayed scale for the next step, computed by the oracle's own update."""
    hist = np.zeros((1, 1), np.float32)
    s = np.ones(1, np.float32)
    si = np.ones(1, np.float32)
    oracle.amax_scale_update(hist, np.array([amax_prev], np.float32), s, si, fmt)
    return np.float32(s[0])


def _chunks(n):
    return [(i, min(n, i + CHUNK)) for i in range(0, n, CHUNK)]


def combine_amax(values, seed=0.0):
    """max over chunk amaxes (and the seed), NaN winning, as one pass would give."""
    vals = [np.float32(seed)] + [np.float32(v) for v in values]
    if any(np.isnan(v) for v in vals):
        return np.float32(np.nan)
    return np.float32(max(vals))


def par_quantize_amax(xb, fmt, scale, amax=0.0):
    """oracle.quantize_amax over every host core; returns (q, amax)."""
    xb = np.ascontiguousarray(xb, np.uint16).reshape(-1)
    q = np.empty(xb.size, np.uint8)

    def work(c):
        a, b = c
        qq, am = oracle.quantize_amax(xb[a:b], fmt, scale)
        q[a:b] = qq
        return am

    with ThreadPoolExecutor(HOST_THREADS) as ex:
        ams = list(ex.map(work, _chunks(xb.size)))
    return q, (combine_amax(ams, amax) if xb.size else np.float32(amax))


def par_dequantize(q, fmt, scale):
    q = np.ascontiguousarray(q, np.uint8).reshape(-1)
    y = np.empty(q.size, np.uint16)

    def work(c):
        a, b = c
        y[a:b] = oracle.dequantize(q[a:b], fmt, scale)

    with ThreadPoolExecutor(HOST_THREADS) as ex:
        list(ex.map(work, _chunks(q.size)))
    return y


def par_qdq_amax(xb, fmt, scale, amax=0.0):
    xb = np.ascontiguousarray(xb, np.uint16).reshape(-1)
    y = np.empty(xb.size, np.uint16)

    def work(c):
        a, b = c
        yy, am = oracle.qdq_amax(xb[a:b], fmt, scale)
        y[a:b] = yy
        return am

    with ThreadPoolExecutor(HOST_THREADS) as ex:
        ams = list(ex.map(work, _chunks(xb.size)))
    return y, (combine_amax(ams, amax) if xb.size else np.float32(amax))


def check_quantize_full(x, q, am, fmt, scale, what, amax0=0.0):
    """Every code of a device tensor's quantization, and its amax, against the oracle."""
    xb = bf16_bits_of(x)
    rq, ra = par_quantize_amax(xb, fmt, scale, amax0)
    assert_codes_equal(q.reshape(-1).cpu().numpy(), rq, fmt, what)
    assert_f32_equal([float(am)], [ra], what + " amax")
    return rq


def bf16_bits_of(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)
