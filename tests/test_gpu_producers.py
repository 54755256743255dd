"""GPU parity of the producers fused with quantize + amax (GELU and LayerNorm).

The bar, for every element of every case:
  - y, the producer's bf16 output, is the bf16 rounding of a value within the
    stated tolerance E of the oracle's float64 definition (oracle.gelu_ref /
    oracle.layernorm_ref; E from oracle.gelu_tolerance /
    oracle.layernorm_tolerance, derived from binary32 arithmetic);
  - the FP8 codes and the amax are bit-exact against oracle.quantize_amax of
    that y, and a call without y gives the same codes and amax.
GELU also has a determinism check: both GELU kernels give the bits of the
fixed binary32 sequence they are built on (tests/csrc/gelu_sequence.c).
"""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (SCALES_ALL, assert_bf16_equal, assert_codes_equal, assert_f32_equal, check_guards, f32,
                         guarded, par_quantize_amax)
from quantize_amax_scaling_gb300 import fp8q
from quantize_amax_scaling_gb300 import workloads as W

pytestmark = pytest.mark.gpu

E4M3FN, E5M2 = fp8q.E4M3FN, fp8q.E5M2
OFFSETS = [(0, 0), (1, 1), (3, 3), (7, 7), (0, 1), (1, 0), (5, 2), (2, 13), (4, 4), (6, 14),
           (8, 8), (15, 15), (9, 1), (12, 12), (8, 0)]


@pytest.fixture(scope="module")
def dev():
    fp8q.lib()
    return torch.device("cuda:0")


def _bf16_key(bits):
    b = np.asarray(bits, np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


# --------------------------------------------------------------------------- GELU

_GELU_ACCEPT = None


def gelu_accept():
    """Per bf16 input pattern: (lowest, highest) acceptable y as order keys, and
    whether y must be a NaN (a NaN input)."""
    global _GELU_ACCEPT
    if _GELU_ACCEPT is None:
        h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
        x = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        r = oracle.gelu_ref_array(h)
        nan = np.isnan(r)
        with np.errstate(invalid="ignore"):
            E = np.where(nan, 0.0, oracle.gelu_tolerance(np.where(nan, 0.0, x), np.where(nan, 0.0, r)))
            lo = _bf16_key(oracle.f64_to_bf16_array(np.where(nan, 0.0, r - E)))
            hi = _bf16_key(oracle.f64_to_bf16_array(np.where(nan, 0.0, r + E)))
        _GELU_ACCEPT = (lo, hi, nan)
    return _GELU_ACCEPT


def assert_gelu_y(hb, yb, what):
    """y within the GELU tolerance of the float64 definition, element by element."""
    lo, hi, nan = gelu_accept()
    hb = np.asarray(hb, np.uint16).reshape(-1).astype(np.int64)
    yb = np.asarray(yb, np.uint16).reshape(-1)
    ynan = ((yb & 0x7F80) == 0x7F80) & ((yb & 0x7F) != 0)
    k = _bf16_key(yb)
    want_nan = nan[hb]
    ok = np.where(want_nan, ynan, ~ynan & (k >= lo[hb]) & (k <= hi[hb]))
    bad = np.nonzero(~ok)[0]
    assert bad.size == 0, (f"{what}: {bad.size} y outside the GELU tolerance, first at {bad[:5]}: "
                           f"h {hb[bad[:5]]} y {yb[bad[:5]]}")


def run_gelu(h, fmt, scale, dev, want_y=True, amax0=0.0):
    n = h.numel()
    y = torch.empty(n, dtype=torch.bfloat16, device=dev) if want_y else None
    q = torch.empty(n, dtype=torch.uint8, device=dev)
    am = f32(amax0, dev)
    fp8q.fp8q_gelu_quantize_amax(h.reshape(-1), y, q, fmt, f32(scale, dev), am)
    torch.cuda.synchronize()
    return y, q, am


def check_gelu(h, fmt, scale, dev, what, amax0=0.0):
    """Run with and without y; y within tolerance, codes and amax exact vs Q(y)."""
    y, q, am = run_gelu(h, fmt, scale, dev, True, amax0)
    _, q2, am2 = run_gelu(h, fmt, scale, dev, False, amax0)
    hb, yb = W.bf16_bits(h), W.bf16_bits(y)
    assert_gelu_y(hb, yb, what)
    rq, ra = par_quantize_amax(yb, fmt, np.float32(scale), amax0)
    assert_codes_equal(q.cpu().numpy(), rq, fmt, what + " codes")
    assert_codes_equal(q2.cpu().numpy(), rq, fmt, what + " codes (no y)")
    assert_f32_equal([float(am), float(am2)], [ra, ra], what + " amax")
    return yb


@pytest.mark.parametrize("fmt", [E4M3FN, E5M2])
def test_gelu_every_bf16_pattern_many_scales(dev, fmt, seq_gelu):
    h = W.all_bf16_patterns(dev)
    hb = W.bf16_bits(h)
    want_bits = seq_gelu(hb)
    for s in SCALES_ALL:
        yb = check_gelu(h, fmt, s, dev, f"scale {s!r}")
        assert_bf16_equal(yb, want_bits, "determinism: the fixed binary32 sequence")
    # without NaN inputs the amax is a number
    f = (hb.astype(np.uint32) << 16).view(np.float32)
    fin = hb[~np.isnan(f)]
    hx = torch.from_numpy(fin.view(np.int16).copy()).view(torch.bfloat16).to(dev)
    check_gelu(hx, fmt, 0.37, dev, "no NaN", amax0=0.5)


@pytest.mark.parametrize("n", [1, 15, 16, 17, 33, 4095, 8193, 70001])
def test_gelu_sizes_offsets_canaries(dev, n):
    g = torch.Generator(device=dev)
    g.manual_seed(11 * n)
    for k, (ho, qo) in enumerate(OFFSETS):
        fmt = E4M3FN if k % 2 else E5M2
        scale = [0.0123, 1.0, 2.0 ** 70, 3.3e-3][k % 4]
        hbuf = (torch.randn(n + 16, generator=g, device=dev) * 3.0).to(torch.bfloat16)
        h = hbuf[ho: ho + n]
        qbuf, q = guarded(n, torch.uint8, dev, qo)
        yo = (ho + 7 * k) % 16                   # often not aligned like h: scalar path
        ybuf, y = guarded(n, torch.bfloat16, dev, yo, fill=0x5A5A)
        am = f32(0.0, dev)
        fp8q.fp8q_gelu_quantize_amax(h, y, q, fmt, f32(scale, dev), am)
        torch.cuda.synchronize()
        yb = W.bf16_bits(y)
        what = f"n={n} off={ho},{qo},{yo}"
        assert_gelu_y(W.bf16_bits(h), yb, what)
        rq, ra = oracle.quantize_amax(yb, fmt, np.float32(scale))
        assert_codes_equal(q.cpu().numpy(), rq, fmt, what)
        assert_f32_equal([float(am)], [ra], f"amax {what}")
        check_guards(qbuf, n, qo)
        check_guards(ybuf, n, yo, fill=0x5A5A)


def test_gelu_full_size(dev):
    """Pre-activation 8192x16384 (N(0,1)), the FFN intermediate of the MLP workload:
    every element, with y and without."""
    g = torch.Generator(device=dev)
    g.manual_seed(W.SEED_FFN)
    h = torch.randn((8192, 16384), generator=g, device=dev).to(torch.bfloat16).reshape(-1)
    check_gelu(h, E4M3FN, np.float32(0.0091), dev, "gelu 8192x16384")


def test_gelu_table_path_every_bf16_pattern(dev, seq_gelu):
    """Large tensors take the table path (every bf16 result computed once per thread-block
    cluster into shared memory): 2^23 elements and more for the codes alone, 2^25 with y.
    All 65536 patterns, repeated to those sizes; every element compared."""
    pat = W.all_bf16_patterns(dev)
    pb = W.bf16_bits(pat)
    want_y = seq_gelu(pb)
    assert_gelu_y(pb, want_y, "the fixed sequence")
    wy = torch.from_numpy(want_y.view(np.int16).copy()).view(torch.bfloat16).to(dev)
    for fmt, s, with_y in [(E4M3FN, 1.0, True), (E5M2, 0.37, False), (E4M3FN, 2.0 ** 70, True),
                           (E5M2, 3.0e-5, False), (E4M3FN, 0.0, True), (E4M3FN, math.nan, False),
                           (E4M3FN, 2.0 ** 70, False), (E5M2, 0.0, False)]:
        reps = 1024 if with_y else 256                    # 2^26 or 2^24 elements
        h = pat.repeat(reps)
        y, q, am = run_gelu(h, fmt, s, dev, want_y=with_y)
        rq, ra = oracle.quantize_amax(want_y, fmt, np.float32(s))
        assert_f32_equal([float(am)], [ra], f"table amax, scale {s!r}")
        wq = torch.from_numpy(rq).to(dev)
        # every element against its pattern's expected value, compared on the device
        assert torch.equal(q.view(reps, 65536), wq.expand(reps, 65536)) or \
            _codes_equal_nan_aware(q.view(reps, 65536), wq, fmt), f"table q, scale {s!r}"
        if y is not None:
            assert torch.equal(_canon_nan(y).view(reps, 65536),
                               _canon_nan(wy).expand(reps, 65536)), f"table y, scale {s!r}"
        del h, y, q


def _canon_nan(t):
    """bf16 bits as int16, every NaN replaced by the canonical 0x7FC0 (any NaN is correct)."""
    b = t.view(torch.int16)
    nan = ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    return torch.where(nan, torch.full_like(b, 0x7FC0), b)


def _codes_equal_nan_aware(q2d, want, fmt):
    """Codes equal, where a NaN code may be any NaN code (device-side compare)."""
    w = want.expand_as(q2d)
    if fmt == E4M3FN:
        wn, gn = (w & 0x7F) == 0x7F, (q2d & 0x7F) == 0x7F
    else:
        wn, gn = (w & 0x7F) > 0x7C, (q2d & 0x7F) > 0x7C
    return bool(torch.equal(wn, gn) and torch.equal(torch.where(wn, 0, q2d), torch.where(wn, 0, w)))


def test_gelu_table_path_unaligned_head_and_tail(dev):
    n, off = (1 << 26) + 13, 3
    g = torch.Generator(device=dev)
    g.manual_seed(17)
    hbuf = (torch.randn(n + 16, generator=g, device=dev) * 4.0).to(torch.bfloat16)
    h = hbuf[off: off + n]
    qbuf, q = guarded(n, torch.uint8, dev, off)
    ybuf, y = guarded(n, torch.bfloat16, dev, off, fill=0x5A5A)
    am = f32(0.0, dev)
    fp8q.fp8q_gelu_quantize_amax(h, y, q, E4M3FN, f32(0.021, dev), am)
    torch.cuda.synchronize()
    yb = W.bf16_bits(y)
    assert_gelu_y(W.bf16_bits(h), yb, "table path unaligned")
    rq, ra = par_quantize_amax(yb, E4M3FN, np.float32(0.021))
    assert_codes_equal(q.cpu().numpy(), rq, E4M3FN, "table path unaligned q")
    assert_f32_equal([float(am)], [ra], "table path amax")
    check_guards(qbuf, n, off)
    check_guards(ybuf, n, off, fill=0x5A5A)


def _patterns(lo, hi):
    """bf16 patterns lo..hi (inclusive) as a host array."""
    return np.arange(lo, hi + 1, dtype=np.uint32).astype(np.uint16)


def _to_dev(bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


@pytest.mark.parametrize("case", ["negative", "small positive", "half N(0,1) half negative", "one NaN",
                                  "one +inf", "seeded amax"])
def test_gelu_code_table_amax(dev, seq_gelu, case):
    """Codes alone on the table path (2^23 elements and more): the amax comes from each
    thread's largest input, and a thread whose largest input is below about 0.3 (or
    negative) reads its elements again.  Tensors where every thread, no thread or some
    threads do; every code and the amax against the oracle's quantize of y."""
    n = (1 << 23) + 5                                # the smallest size on the table path, and a tail
    rng = np.random.default_rng(zlib.crc32(case.encode()))
    normal = np.asarray(torch.from_numpy(rng.standard_normal(n).astype(np.float32)).to(torch.bfloat16)
                        .view(torch.int16).numpy()).view(np.uint16)
    neg = _patterns(0x8000, 0xFF80)                          # -0 ... -inf
    amax0 = 0.0
    if case == "negative":
        hb = neg[rng.integers(0, neg.size, n)]
    elif case == "small positive":
        hb = _patterns(0x0000, 0x3E7F)[rng.integers(0, 0x3E80, n)]   # +0 ... just under 0.25
    elif case == "half N(0,1) half negative":
        hb = normal.copy()
        hb[n // 2:] = neg[rng.integers(0, neg.size, n - n // 2)]
    elif case == "one NaN":
        hb = normal.copy()
        hb[n // 3] = 0x7FC1
    elif case == "one +inf":
        hb = normal.copy()
        hb[n - 2] = 0x7F80                                   # in the scalar tail
    else:
        hb = neg[rng.integers(0, neg.size, n)]
        amax0 = 0.5                                          # above every |y|: the seed stays
    h = _to_dev(hb, dev)
    for fmt, scale in ((E4M3FN, np.float32(0.0123)), (E5M2, np.float32(2.0 ** 70))):
        _, q, am = run_gelu(h, fmt, scale, dev, want_y=False, amax0=amax0)
        want_y = seq_gelu(hb)
        rq, ra = par_quantize_amax(want_y, fmt, scale, amax0)
        assert_codes_equal(q.cpu().numpy(), rq, fmt, f"{case} codes")
        assert_f32_equal([float(am)], [ra], f"{case} amax")


def test_gelu_table_path_more_than_2_pow_31_elements(dev, seq_gelu):
    """The table path's vector and tail arithmetic stays 64-bit: 2^31 + 19 elements, with y,
    made of every finite bf16 pattern repeated; every element is compared (on the device)
    with its pattern's expected value, and the amax is known exactly."""
    pat = W.all_bf16_patterns(dev)
    pb = W.bf16_bits(pat)
    pf = (pb.astype(np.uint32) << 16).view(np.float32)
    keep = ~np.isnan(pf)
    fin_b = pb[keep]
    fin = torch.from_numpy(fin_b.view(np.int16).copy()).view(torch.bfloat16).to(dev)
    m = fin.numel()
    n = (1 << 31) + 19
    h = fin.repeat(n // m + 1)[:n].contiguous()
    y = torch.empty(n, dtype=torch.bfloat16, device=dev)
    q = torch.empty(n, dtype=torch.uint8, device=dev)
    am = f32(0.0, dev)
    scale = np.float32(0.0123)
    fp8q.fp8q_gelu_quantize_amax(h, y, q, E4M3FN, f32(scale, dev), am)
    torch.cuda.synchronize()
    want_y = seq_gelu(fin_b)
    assert_gelu_y(fin_b, want_y, "the fixed sequence")
    rq, ra = oracle.quantize_amax(want_y, E4M3FN, scale)
    assert_f32_equal([float(am)], [ra], "amax over 2^31 + 19 elements")
    wy = torch.from_numpy(want_y.view(np.int16).copy()).to(dev)
    wq = torch.from_numpy(rq).to(dev)
    full = n // m
    assert torch.equal(y.view(torch.int16)[:full * m].view(full, m), wy.expand(full, m)), "y, whole periods"
    assert torch.equal(y.view(torch.int16)[full * m:], wy[: n - full * m]), "y, last partial period"
    assert torch.equal(q[:full * m].view(full, m), wq.expand(full, m)), "q, whole periods"
    assert torch.equal(q[full * m:], wq[: n - full * m]), "q, last partial period"
    # the codes alone (the code table kernel) on the same input
    q.fill_(0)
    am2 = f32(0.0, dev)
    fp8q.fp8q_gelu_quantize_amax(h, None, q, E4M3FN, f32(scale, dev), am2)
    torch.cuda.synchronize()
    assert_f32_equal([float(am2)], [ra], "amax over 2^31 + 19 elements, codes alone")
    assert torch.equal(q[:full * m].view(full, m), wq.expand(full, m)), "q alone, whole periods"
    assert torch.equal(q[full * m:], wq[: n - full * m]), "q alone, last partial period"
    del h, y, q
    torch.cuda.empty_cache()


# --------------------------------------------------------------------------- LayerNorm

def run_layernorm(x, gamma, beta, fmt, scale, dev, want_y=True, eps=1e-6, amax0=0.0):
    rows, H = x.shape
    y = torch.empty((rows, H), dtype=torch.bfloat16, device=dev) if want_y else None
    q = torch.empty((rows, H), dtype=torch.uint8, device=dev)
    am = f32(amax0, dev)
    fp8q.fp8q_layernorm_quantize_amax(x, y, q, gamma, beta, fmt, f32(scale, dev), am, eps=eps)
    torch.cuda.synchronize()
    return y, q, am


def assert_layernorm_y(xb, H, g, b, eps, yb, what, row_chunk=2048):
    """y within the LayerNorm tolerance of the float64 definition, element by element."""
    xb = np.asarray(xb, np.uint16).reshape(-1, H)
    yb = np.asarray(yb, np.uint16).reshape(-1, H)
    for r0 in range(0, xb.shape[0], row_chunk):
        xs = xb[r0:r0 + row_chunk]
        r, mean, rstd = oracle.layernorm_ref(xs, H, g, b, eps)
        x64 = (xs.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        with np.errstate(invalid="ignore", over="ignore"):
            E = oracle.layernorm_tolerance(x64, g, b, eps, mean, rstd, r)
        ok = oracle.bf16_within(yb[r0:r0 + row_chunk], r, E)
        bad = np.nonzero(~ok)[0]
        assert bad.size == 0, (f"{what}: {bad.size} y outside the LayerNorm tolerance, first at flat "
                               f"{bad[:5] + r0 * H}")


def check_layernorm(x, gamma, beta, fmt, scale, dev, eps=1e-6, amax0=0.0, what=""):
    """Run with and without y; y within tolerance, codes and amax exact vs Q(y)."""
    y, q, am = run_layernorm(x, gamma, beta, fmt, scale, dev, True, eps, amax0)
    _, q2, am2 = run_layernorm(x, gamma, beta, fmt, scale, dev, False, eps, amax0)
    H = x.shape[1]
    yb = W.bf16_bits(y)
    assert_layernorm_y(W.bf16_bits(x), H, gamma.cpu().numpy(), beta.cpu().numpy(), eps, yb, what)
    rq, ra = par_quantize_amax(yb, fmt, np.float32(scale), amax0)
    assert_codes_equal(q.cpu().numpy(), rq, fmt, f"ln q {what}")
    assert_codes_equal(q2.cpu().numpy(), rq, fmt, f"ln q without y {what}")
    assert_f32_equal([float(am), float(am2)], [ra, ra], f"ln amax {what}")
    return yb


LN_SHAPES = [(1, 16), (3, 272), (2, 4096), (2, 16384), (7, 4112), (300, 48), (5, 4080), (4, 8208),
             (33, 1024), (2, 12288), (9, 2064), (17, 6160),
             (3, 16400), (5, 18432), (2, 24576), (4, 32768)]   # rows longer than 16384: one row a batch


@pytest.mark.parametrize("rows,H", LN_SHAPES)
def test_layernorm_shapes(dev, rows, H):
    """Row lengths from 16 to 32768 (one to eight warps a row in the statistics, ragged last vectors)."""
    x = W.residual_stream(seed=rows * 7919 + H, device=dev, shape=(rows, H))
    gamma, beta = W.layernorm_params(H, seed=H, device=dev)
    for k, (fmt, scale) in enumerate([(E4M3FN, 0.0123), (E5M2, 1.0), (E4M3FN, 2.0 ** 70), (E5M2, 3.3e-3)]):
        check_layernorm(x, gamma, beta, fmt, scale, dev, amax0=0.25 * k, what=f"{rows}x{H} scale {scale}")


@pytest.mark.parametrize("k", range(12))
def test_layernorm_random_shapes(dev, k):
    """Seeded random row counts and lengths (H a multiple of 16 up to 32768), a scale per
    case (slow-path ones too) and both formats, on the LayerNorm input workload's rows."""
    rng = np.random.default_rng(500 + k)
    H = 16 * int(rng.integers(1, 2049))
    rows = int(rng.integers(1, max(2, min(600, (1 << 21) // H))))
    x = W.residual_stream(seed=900 + k, device=dev, shape=(rows, H))
    gamma, beta = W.layernorm_params(H, seed=k, device=dev)
    fmt = E4M3FN if k % 2 else E5M2
    scale = [0.0123, 1.0, 2.0 ** 70, 3.3e-3, 0.0, 0.07][k % 6]
    check_layernorm(x, gamma, beta, fmt, scale, dev, amax0=0.1 * (k % 3), what=f"{rows}x{H} scale {scale}")


@pytest.mark.parametrize("rows,H", [(20000, 48), (5000, 4096), (3000, 8192), (1000, 16384), (7001, 272),
                                    (600, 32768)])
def test_layernorm_many_rows(dev, rows, H):
    """More rows than the persistent grid has warps (or warp groups), so each one loops."""
    x = W.residual_stream(seed=rows + H, device=dev, shape=(rows, H))
    gamma, beta = W.layernorm_params(H, seed=H + 1, device=dev)
    check_layernorm(x, gamma, beta, E4M3FN, 0.021, dev, what=f"{rows}x{H}")
    check_layernorm(x, gamma, beta, E5M2, 0.5, dev, what=f"{rows}x{H} e5m2")


def test_layernorm_every_scale_and_flax_defaults(dev):
    x = W.residual_stream(seed=5, device=dev, shape=(64, 4096))
    ones = torch.ones(4096, dtype=torch.float32, device=dev)
    zeros = torch.zeros(4096, dtype=torch.float32, device=dev)
    for fmt in (E4M3FN, E5M2):
        for s in SCALES_ALL:
            check_layernorm(x, ones, zeros, fmt, s, dev, what=f"scale {s!r}")


@pytest.mark.parametrize("H", [512, 8192, 20480])   # one CTA a batch; clusters of 2 and 5
def test_layernorm_degenerate_rows(dev, H):
    """Constant rows (var = 0: y = beta exactly), rows with inf or NaN (y NaN), and rows
    outside binary32's range for the statistics (Q overflows; eps = 0 on constant or
    subnormal rows), where no tolerance applies but the codes and amax must still be
    exactly those of y."""
    rows = []
    rows.append(np.full(H, 0x3F80, np.uint16))                        # all 1.0
    rows.append(np.zeros(H, np.uint16))                               # all +0
    r = np.full(H, 0x4000, np.uint16); r[17] = 0x7F80; rows.append(r)   # +inf
    r = np.full(H, 0x4000, np.uint16); r[300] = 0x7FC1; rows.append(r)  # NaN
    r = np.full(H, 0x4000, np.uint16); r[5] = 0xFF80; r[H - 6] = 0x7F80; rows.append(r)  # +inf and -inf
    rows.append(np.where(np.arange(H) % 2 == 0, 0x7F00, 0xFF00).astype(np.uint16))  # +-1.7e38: Q overflows
    rows.append(np.where(np.arange(H) % 3 == 0, 0x0001, 0x8002).astype(np.uint16))  # bf16 subnormals
    rows.append((np.arange(H) % 7 + 0x3F80).astype(np.uint16))        # values near 1 (cancellation)
    xb = np.stack(rows)
    x = torch.from_numpy(xb.view(np.int16).copy()).view(torch.bfloat16).to(dev)
    gamma, beta = W.layernorm_params(H, seed=77, device=dev)
    g, b = gamma.cpu().numpy(), beta.cpu().numpy()
    beta_bf16 = torch.from_numpy(b).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for eps in (1e-6, 0.0, 1e-2):
        for fmt in (E4M3FN, E5M2):
            yb = check_layernorm(x, gamma, beta, fmt, 0.05, dev, eps=eps, what=f"eps {eps}").reshape(-1, H)
            if eps > 0:
                assert_bf16_equal(yb[0], beta_bf16, "constant row gives beta")
                assert_bf16_equal(yb[1], beta_bf16, "zero row gives beta")
            for i in (2, 3, 4):
                assert np.all(((yb[i] & 0x7F80) == 0x7F80) & ((yb[i] & 0x7F) != 0)), f"row {i} not NaN"


def test_layernorm_does_not_write_outside(dev):
    rows, H = 9, 4112
    x = W.residual_stream(seed=3, device=dev, shape=(rows, H))
    gamma, beta = W.layernorm_params(H, device=dev)
    n = rows * H
    qbuf, q = guarded(n, torch.uint8, dev, 0)
    ybuf, y = guarded(n, torch.bfloat16, dev, 0, fill=0x5A5A)
    am = f32(0.0, dev)
    fp8q.fp8q_layernorm_quantize_amax(x, y.view(rows, H), q.view(rows, H), gamma, beta, E4M3FN,
                                      f32(0.02, dev), am)
    torch.cuda.synchronize()
    yb = W.bf16_bits(y)
    assert_layernorm_y(W.bf16_bits(x), H, gamma.cpu().numpy(), beta.cpu().numpy(), 1e-6, yb, "guarded")
    rq, ra = oracle.quantize_amax(yb, E4M3FN, np.float32(0.02))
    assert_codes_equal(q.cpu().numpy(), rq, E4M3FN, "guarded q")
    assert_f32_equal([float(am)], [ra], "guarded amax")
    check_guards(qbuf, n, 0)
    check_guards(ybuf, n, 0, fill=0x5A5A)


def test_layernorm_full_size(dev):
    """The MLP's LayerNorm input, 8192x4096: every element, with y and without."""
    x = W.residual_stream(device=dev)
    gamma, beta = W.layernorm_params(x.shape[1], device=dev)
    check_layernorm(x, gamma, beta, E4M3FN, np.float32(0.031), dev, what="8192x4096")


def test_layernorm_more_than_2_pow_31_elements(dev):
    """Row offsets stay 64-bit: 131073 rows of 16384 (2^31 + 16384 elements).  The rows
    around the 2^31 boundary, the first and the last are compared with the oracle (y within
    the tolerance, codes exact against the quantize of y); the amax equals max|y| over the
    whole output, and the codes-alone call gives the same codes and amax."""
    rows, H = 131073, 16384
    g = torch.Generator(device=dev)
    g.manual_seed(23)
    x = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
    for r0 in range(0, rows, 8192):                  # N(mu_r, sigma_r^2) rows, in slices
        r1 = min(rows, r0 + 8192)
        mu = torch.randn((r1 - r0, 1), generator=g, device=dev)
        sd = torch.rand((r1 - r0, 1), generator=g, device=dev) * 2 + 0.1
        x[r0:r1] = (torch.randn((r1 - r0, H), generator=g, device=dev) * sd + mu).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(H, generator=g, device=dev)).float()
    beta = (0.1 * torch.randn(H, generator=g, device=dev)).float()
    scale = np.float32(0.027)
    y, q, am = run_layernorm(x, gamma, beta, E4M3FN, scale, dev, True)
    _, q2, am2 = run_layernorm(x, gamma, beta, E4M3FN, scale, dev, False)
    assert torch.equal(q, q2), "codes with and without y"
    yi = y.view(torch.int16)
    amax_y = (yi.view(-1) & 0x7FFF).max().item()          # |y| bits (no NaN here)
    assert_f32_equal([float(am), float(am2)], [np.uint32(amax_y << 16).view(np.float32)] * 2, "amax = max|y|")
    picks = [0, 1, 2, 131070, 131071, 131072]          # row 131072 starts at element 2^31
    xb = W.bf16_bits(x[picks])
    yb = W.bf16_bits(y[picks])
    assert_layernorm_y(xb, H, gamma.cpu().numpy(), beta.cpu().numpy(), 1e-6, yb, "rows around 2^31")
    rq, _ = oracle.quantize_amax(yb.reshape(-1), E4M3FN, scale)
    assert_codes_equal(q[picks].cpu().numpy().reshape(-1), rq, E4M3FN, "codes of rows around 2^31")
    del x, y, q, q2
    torch.cuda.empty_cache()


def test_layernorm_close_to_torch_layer_norm(dev):
    """Sanity check against torch's float32 layer_norm (another binary32 evaluation)."""
    x = W.residual_stream(seed=9, device=dev, shape=(256, 4096))
    gamma, beta = W.layernorm_params(4096, device=dev)
    y, _, _ = run_layernorm(x, gamma, beta, E4M3FN, 1.0, dev)
    ref = torch.nn.functional.layer_norm(x.float(), (4096,), gamma, beta, eps=1e-6)
    torch.testing.assert_close(y.float(), ref, rtol=2 ** -7, atol=1e-5)


def test_layernorm_output_is_deterministic(dev):
    """Two calls on the same input give the same bits (fixed reduction order per row)."""
    x = W.residual_stream(seed=21, device=dev, shape=(1000, 4096))
    gamma, beta = W.layernorm_params(4096, device=dev)
    y1, q1, a1 = run_layernorm(x, gamma, beta, E4M3FN, 0.03, dev)
    y2, q2, a2 = run_layernorm(x, gamma, beta, E4M3FN, 0.03, dev)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)) and torch.equal(q1, q2)
    assert float(a1) == float(a2)
