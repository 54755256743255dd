"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties one oracle function to an independent fact: hand-derived
landmarks (tests/golden), library casts (torch's and ml_dtypes' float8/bf16
conversions, used only in the range where they agree with the spec),
closed forms, brute force and invariants.

Sources: "User Guide on Native XLA-FP8" (NVIDIA JAX-Toolbox), sections
"JAX" (Q, DQ, delayed scaling) and "Gradient accumulation of FP8 params";
"Fusion of Fp8 quantization and amax reduction kernels" (openxla/xla issue);
"Implement fused kernel for FP8 scale update" (TransformerEngine PR).
"""
import math
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN

E4M3FN, E5M2 = 0, 1
FMT_NAME = {"e4m3fn": E4M3FN, "e5m2": E5M2}
TORCH_FP8 = {E4M3FN: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
FP8_MAX = {E4M3FN: 448.0, E5M2: 57344.0}
MAX_CODE = {E4M3FN: 0x7E, E5M2: 0x7B}


def _val(expr: str) -> float:
    expr = expr.strip()
    if expr == "nan":
        return math.nan
    if expr in ("inf", "-inf"):
        return math.inf if expr == "inf" else -math.inf
    if expr == "-0":
        return -0.0
    total = 0.0
    for term in expr.split("+"):
        if "*2^" in term:
            p, e = term.split("*2^")
            total += float(p) * 2.0 ** int(e)
        else:
            total += float(term)
    return total


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def _is_nan_code(c, fmt):
    c &= 0x7F
    return c == 0x7F if fmt == E4M3FN else c > 0x7C


def _torch_decode(fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(TORCH_FP8[fmt]).to(torch.float32).numpy()


def _torch_cast_codes(y, fmt):
    """Library cast float32 -> fp8 codes (non-saturating; valid for |y| <= max only)."""
    return torch.from_numpy(np.ascontiguousarray(y, np.float32)).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()


ALL_BF16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)
ALL_BF16_F32 = (ALL_BF16.astype(np.uint32) << 16).view(np.float32)

SCALES = [1.0, 0.5, 2.0 ** -6, 2.0 ** 20, 1.0 / 3.0, 0.012345678, 7.5, 448.0 / 3.9,
          3.0e-5, 1.7e4, 2.0 ** -70, 2.0 ** 70, 1.0e-38, 5.0e-45]


# --------------------------------------------------------------------------- decode

def test_decode_landmarks(orc):
    for fmt_s, code_s, val_s in _golden("fp8_landmarks.txt"):
        fmt, code, want = FMT_NAME[fmt_s], int(code_s, 16), _val(val_s)
        got = orc.fp8_decode(code, fmt)
        if math.isnan(want):
            assert math.isnan(got), (fmt_s, code_s)
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (fmt_s, code_s, got)


@pytest.mark.parametrize("fmt", [E4M3FN, E5M2])
def test_decode_all_codes_match_torch(orc, fmt):
    lib_vals = _torch_decode(fmt)
    for c in range(256):
        got = orc.fp8_decode(c, fmt)
        want = float(lib_vals[c])
        if math.isnan(want):
            assert math.isnan(got), c
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (c, got, want)
    assert orc.fp8_max(fmt) == FP8_MAX[fmt]
    assert orc.fp8_max_code(fmt) == MAX_CODE[fmt]


@pytest.mark.parametrize("fmt", [E4M3FN, E5M2])
def test_decode_all_codes_match_ml_dtypes(orc, fmt):
    ml = pytest.importorskip("ml_dtypes")
    t = ml.float8_e4m3fn if fmt == E4M3FN else ml.float8_e5m2
    vals = np.arange(256, dtype=np.uint32).astype(np.uint8).view(t).astype(np.float64)
    for c in range(256):
        got = orc.fp8_decode(c, fmt)
        assert (math.isnan(got) and math.isnan(vals[c])) or got == vals[c], c


def test_format_resolution_and_range(orc):
    # E4M3 has twice the resolution of E5M2 (one more mantissa bit) and about half
    # the dynamic range in binades ("User Guide on Native XLA-FP8", opening section).
    def binades(fmt):
        return math.log2(orc.fp8_max(fmt) / orc.fp8_decode(1, fmt))
    assert orc.fp8_decode(0x39, E4M3FN) - 1.0 == 0.125      # ulp at 1: 2^-3
    assert orc.fp8_decode(0x3D, E5M2) - 1.0 == 0.25          # ulp at 1: 2^-2
    assert 0.45 < binades(E4M3FN) / binades(E5M2) < 0.65


# --------------------------------------------------------------------------- encode

def test_encode_landmarks(orc):
    for fmt_s, y_s, code_s in _golden("fp8_rounding_cases.txt"):
        fmt, y, want = FMT_NAME[fmt_s], _val(y_s), int(code_s, 16)
        assert float(np.float32(y)) == y or math.isnan(y) or abs(y) > 3e38, "fixture must be exact in fp32"
        got = orc.fp8_encode(y, fmt)
        if math.isnan(y):
            assert _is_nan_code(got, fmt), (fmt_s, y_s, hex(got))
        else:
            assert got == want, (fmt_s, y_s, hex(got), hex(want))


@pytest.mark.parametrize("fmt", [E4M3FN, E5M2])
def test_quantize_exhaustive_bf16_vs_library_cast(orc, fmt):
    """All 65536 bf16 inputs x many scales: in range the oracle equals the library cast
    of the IEEE fp32 quotient; above range it saturates; NaN gives a NaN code."""
    x = ALL_BF16_F32
    for s in SCALES:
        s32 = np.float32(s)
        with np.errstate(all="ignore"):
            y = (x / s32).astype(np.float32)          # IEEE binary32 division, RN
        q, _ = orc.quantize_amax(ALL_BF16, fmt, s32)
        nan = np.isnan(y)
        inr = ~nan & (np.abs(y) <= FP8_MAX[fmt])
        lib_codes = _torch_cast_codes(np.where(inr, y, 0).astype(np.float32), fmt)
        assert np.array_equal(q[inr], lib_codes[inr]), f"scale {s}"
        over = ~nan & ~inr
        sat = np.where(np.signbit(y[over]), 0x80 | MAX_CODE[fmt], MAX_CODE[fmt]).astype(np.uint8)
        assert np.array_equal(q[over], sat), f"scale {s}"
        assert all(_is_nan_code(int(c), fmt) for c in q[nan])


@pytest.mark.parametrize("fmt", [E4M3FN, E5M2])
def test_quantize_in_range_vs_ml_dtypes(orc, fmt):
    ml = pytest.importorskip("ml_dtypes")
    t = ml.float8_e4m3fn if fmt == E4M3FN else ml.float8_e5m2
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    y = bits.view(np.float32)
    y = y[np.isfinite(y) & (np.abs(y) <= FP8_MAX[fmt])]
    want = y.astype(t).view(np.uint8)
    got = np.array([orc.fp8_encode(v, fmt) for v in y[:20000]], np.uint8)
    assert np.array_equal(got, want[:20000])


@pytest.mark.parametrize("fmt", [E4M3FN, E5M2])
def test_exactly_representable_values_round_trip(orc, fmt):
    """Every finite code's value, quantized with scale 1, returns the same code."""
    for c in range(256):
        v = orc.fp8_decode(c, fmt)
        if math.isnan(v) or math.isinf(v):
            continue
        h = torch.tensor([v], dtype=torch.float32).to(torch.bfloat16)
        assert float(h) == v or (v == 0 and float(h) == 0)
        hb = h.view(torch.int16).numpy().view(np.uint16)
        q, _ = orc.quantize_amax(hb, fmt, 1.0)
        assert int(q[0]) == c, (c, v, hex(int(q[0])))


# --------------------------------------------------------------------------- amax

def _brute_amax(vals):
    m = 0.0
    for v in vals:
        if math.isnan(v):
            return math.nan
        m = max(m, abs(v))
    return m


def test_amax_brute_force(orc):
    rng = np.random.default_rng(11)
    for trial in range(20):
        n = int(rng.integers(1, 3000))
        bits = rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16)
        f = (bits.astype(np.uint32) << 16).view(np.float32)
        if trial % 3 == 0:  # mostly without NaN so the finite max is exercised
            bits = np.where(np.isnan(f), np.uint16(0x8000), bits).astype(np.uint16)
            f = (bits.astype(np.uint32) << 16).view(np.float32)
        want = _brute_amax([float(v) for v in f])
        got = float(orc.amax(bits))
        _, got2 = orc.quantize_amax(bits, E4M3FN, 1.0)
        for g in (got, float(got2)):
            assert (math.isnan(want) and math.isnan(g)) or g == want
        perm = rng.permutation(n)
        g3 = float(orc.amax(bits[perm]))
        assert (math.isnan(want) and math.isnan(g3)) or g3 == want


def test_amax_signs_infs_and_accumulation(orc):
    vals = torch.tensor([-3.0, 2.0, -0.0, 1e-40, -5.5], dtype=torch.float32).to(torch.bfloat16)
    bits = vals.view(torch.int16).numpy().view(np.uint16)
    _, a = orc.quantize_amax(bits, E4M3FN, 1.0)
    assert float(a) == 5.5
    _, a = orc.quantize_amax(bits, E4M3FN, 1.0, amax=7.25)   # max-accumulate, not overwrite
    assert float(a) == 7.25
    _, a = orc.quantize_amax(bits[:0], E4M3FN, 1.0, amax=3.5)  # empty: unchanged
    assert float(a) == 3.5
    neg_inf = torch.tensor([1.0, -math.inf], dtype=torch.float32).to(torch.bfloat16)
    _, a = orc.quantize_amax(neg_inf.view(torch.int16).numpy().view(np.uint16), E5M2, 1.0)
    assert math.isinf(float(a)) and float(a) > 0                # inf propagates, sign dropped
    zeros = torch.tensor([-0.0, -0.0], dtype=torch.float32).to(torch.bfloat16)
    _, a = orc.quantize_amax(zeros.view(torch.int16).numpy().view(np.uint16), E4M3FN, 1.0)
    assert float(a) == 0.0 and not math.copysign(1, float(a)) < 0


# --------------------------------------------------------------------------- dequantize / bf16

def test_bf16_rounding_landmarks(orc):
    for fb, hb in _golden("bf16_rounding_cases.txt"):
        f = np.array([int(fb, 16)], np.uint32).view(np.float32)[0]
        got = orc.f32_to_bf16(f)
        if hb == "nan":
            assert (got & 0x7F80) == 0x7F80 and (got & 0x7F) != 0, hex(got)
        else:
            assert got == int(hb, 16), (fb, hex(got), hb)


def test_bf16_rounding_vs_torch(orc):
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, 50000, dtype=np.uint64).astype(np.uint32)
    bits[:2000] &= 0x007FFFFF                       # subnormals
    bits[2000:4000] = (bits[2000:4000] & 0x0000FFFF) | 0x7F7F0000   # near overflow
    bits[4000:6000] = (bits[4000:6000] & 0xFFFF0000) | 0x8000      # exact ties
    f = bits.view(np.float32)
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for i in range(len(f)):
        if np.isnan(f[i]):
            continue
        assert orc.f32_to_bf16(f[i]) == want[i], hex(bits[i])


@pytest.mark.parametrize("fmt", [E4M3FN, E5M2])
def test_dequantize_all_codes_vs_library(orc, fmt):
    codes = np.arange(256, dtype=np.uint32).astype(np.uint8)
    dec = torch.from_numpy(codes.copy()).view(TORCH_FP8[fmt]).to(torch.float32)
    for s in SCALES + [-2.5, 0.0]:
        want = (dec * torch.tensor(np.float32(s))).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        got = orc.dequantize(codes, fmt, s)
        for c in range(256):
            wf = (int(want[c]) << 16)
            if (wf & 0x7F800000) == 0x7F800000 and (wf & 0x007FFFFF):
                assert (got[c] & 0x7F80) == 0x7F80 and (got[c] & 0x7F), (c, s)
            else:
                assert got[c] == want[c], (fmt, c, s, hex(got[c]), hex(want[c]))


@pytest.mark.parametrize("fmt", [E4M3FN, E5M2])
def test_dq_of_q_is_identity_on_representable_values(orc, fmt):
    """DQ(Q(x)) == x when scale = 2^k and x / scale is an FP8 value."""
    for k in (-8, -1, 0, 3, 12):
        vals, codes = [], []
        for c in range(256):
            v = orc.fp8_decode(c, fmt)
            if math.isnan(v) or math.isinf(v):
                continue
            vals.append(math.ldexp(v, k))
            codes.append(c)
        x = torch.tensor(vals, dtype=torch.float32)
        xb = x.to(torch.bfloat16)
        assert torch.equal(xb.float(), x)
        bits = xb.view(torch.int16).numpy().view(np.uint16)
        q, _ = orc.quantize_amax(bits, fmt, 2.0 ** k)
        assert list(q) == codes
        y = orc.dequantize(q, fmt, 2.0 ** k)
        assert np.array_equal(y, bits)


# --------------------------------------------------------------------------- multi-tensor

def test_multi_tensor_equals_per_tensor(orc):
    rng = np.random.default_rng(5)
    xs = [rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16) for n in (0, 1, 17, 4096, 333)]
    scales = [1.0, 0.25, 3.3, 1e-3, 77.0]
    qs, am = orc.multi_quantize_amax(xs, E5M2, scales)
    for x, s, q, a in zip(xs, scales, qs, am):
        q1, a1 = orc.quantize_amax(x, E5M2, s)
        assert np.array_equal(q, q1)
        assert (math.isnan(a) and math.isnan(a1)) or a == a1


# --------------------------------------------------------------------------- scale update

def _run_update(orc, H, S, seq, algo=0, margin=0, fmt=E4M3FN, slot_format=None, scale0=1.0):
    hist = np.zeros((H, S), np.float32)
    scale = np.full(S, scale0, np.float32)
    scale_inv = np.full(S, 1.0 / scale0, np.float32)
    for amax_new in seq:
        orc.amax_scale_update(hist, np.asarray(amax_new, np.float32), scale, scale_inv, fmt, algo,
                              margin, slot_format)
    return hist, scale, scale_inv


def test_history_roll_window_newest_first(orc):
    rng = np.random.default_rng(1)
    for H in (1, 2, 3, 4):
        for S in (1, 2, 3):
            seq = [rng.uniform(0.1, 10, S).astype(np.float32) for _ in range(6)]
            for k in range(1, 7):
                hist, _, _ = _run_update(orc, H, S, seq[:k])
                for h in range(H):
                    want = seq[k - 1 - h] if h < k else np.zeros(S, np.float32)
                    assert np.array_equal(hist[h], want), (H, S, k, h)


def test_scale_closed_form_powers_of_two(orc):
    # amax = FP8_MAX * 2^j gives scale exactly 2^j and scale_inv 2^-j
    for fmt in (E4M3FN, E5M2):
        for j in (-20, -3, 0, 5, 30):
            a = FP8_MAX[fmt] * 2.0 ** j
            _, sc, si = _run_update(orc, 4, 1, [[a]], fmt=fmt)
            assert sc[0] == 2.0 ** j and si[0] == 2.0 ** -j


def test_scale_matches_page_example(orc):
    """Delayed scaling example: A_scale = max|A| / E4M3_MAX ("User Guide on Native
    XLA-FP8", section "JAX"), starting from a zero history and unit scale."""
    from quantize_amax_scaling_gb300 import workloads as W
    A, B = W.tiny_pair()
    amax_A = torch.max(torch.abs(A.float()))
    amax_B = torch.max(torch.abs(B.float()))
    hist = np.zeros((16, 2), np.float32)
    scale = np.ones(2, np.float32)
    scale_inv = np.ones(2, np.float32)
    qa, ra = orc.quantize_amax(W.bf16_bits(A), E4M3FN, 1.0)
    qb, rb = orc.quantize_amax(W.bf16_bits(B), E4M3FN, 1.0)
    assert float(ra) == float(amax_A) and float(rb) == float(amax_B)
    orc.amax_scale_update(hist, np.array([ra, rb], np.float32), scale, scale_inv)
    e4m3_max = torch.tensor(torch.finfo(torch.float8_e4m3fn).max, dtype=torch.float32)
    assert scale[0] == float(amax_A / e4m3_max) and scale[1] == float(amax_B / e4m3_max)
    assert scale_inv[0] == float(1.0 / (amax_A / e4m3_max))
    # scale 1.0 is a plain cast: U[0,1) values are all in range
    assert np.array_equal(qa, _torch_cast_codes(A.float().numpy().reshape(-1), E4M3FN))


def test_scale_error_bound(orc):
    rng = np.random.default_rng(9)
    a = np.exp(rng.normal(0, 4, 64)).astype(np.float32)
    _, sc, si = _run_update(orc, 3, 64, [a])
    rel = np.abs(sc.astype(np.float64) * 448.0 / a.astype(np.float64) - 1.0)
    assert rel.max() <= 2.0 ** -24
    assert np.abs(sc.astype(np.float64) * si.astype(np.float64) - 1.0).max() <= 2.0 ** -23


def test_select_max_equals_single_entry_run_of_window_max(orc):
    rng = np.random.default_rng(4)
    H, S = 4, 3
    seq = [np.exp(rng.normal(0, 2, S)).astype(np.float32) for _ in range(7)]
    _, sc_max, _ = _run_update(orc, H, S, seq, algo=0)
    window_max = np.max(np.stack(seq[-H:]), axis=0)
    _, sc_ref, _ = _run_update(orc, 1, S, [window_max], algo=0)
    assert np.array_equal(sc_max, sc_ref)
    _, sc_mr, _ = _run_update(orc, H, S, seq, algo=1)
    _, sc_last, _ = _run_update(orc, 1, S, [seq[-1]], algo=0)
    assert np.array_equal(sc_mr, sc_last)
    assert not np.array_equal(sc_mr, sc_max)


def test_margin_is_exact_power_of_two(orc):
    rng = np.random.default_rng(6)
    a = np.exp(rng.normal(0, 3, 5)).astype(np.float32)
    _, s0, _ = _run_update(orc, 2, 5, [a], margin=0)
    for m in (-3, 1, 2, 7):
        _, sm, _ = _run_update(orc, 2, 5, [a], margin=m)
        assert np.array_equal(sm, (s0.astype(np.float64) * 2.0 ** m).astype(np.float32))


def test_pass_through_of_zero_and_non_finite(orc):
    for bad in (0.0, math.inf, math.nan, -1.0):
        hist, sc, si = _run_update(orc, 3, 2, [[bad, 448.0]], algo=1, scale0=4.0)
        assert sc[0] == 4.0 and si[0] == 0.25                 # untouched
        assert sc[1] == 1.0 and si[1] == 1.0                   # updated
        assert (math.isnan(bad) and math.isnan(hist[0, 0])) or hist[0, 0] == bad  # still recorded
    # a NaN anywhere in the window makes max-selection non-finite: pass-through
    _, sc, _ = _run_update(orc, 3, 1, [[math.nan], [2.0]], algo=0, scale0=4.0)
    assert sc[0] == 4.0
    # ... and once it leaves the window the slot updates again
    _, sc, _ = _run_update(orc, 2, 1, [[math.nan], [2.0], [448.0]], algo=0, scale0=4.0)
    assert sc[0] == 1.0
    # a scale that would underflow below the normal range passes through
    _, sc, _ = _run_update(orc, 1, 1, [[1e-37]], margin=-20, scale0=4.0)
    assert sc[0] == 4.0


def test_per_slot_formats(orc):
    sf = np.array([0, 1, 7], np.uint8)
    _, sc, _ = _run_update(orc, 2, 3, [[448.0, 57344.0, 448.0]], slot_format=sf)
    assert sc[0] == 1.0 and sc[1] == 1.0
    assert sc[2] == 1.0   # unknown format code: slot left unchanged (started at 1.0)
    _, sc, _ = _run_update(orc, 2, 3, [[57344.0, 57344.0, 448.0]], slot_format=sf, scale0=2.0)
    assert sc[0] == 128.0 and sc[1] == 1.0 and sc[2] == 2.0


# --------------------------------------------------------------------------- fused Q -> DQ

QDQ_SCALES = [1.0, 0.25, 2.0 ** 10, 1.0 / 3.0, 0.0123, 7.5, 3.0e-5]


@pytest.mark.parametrize("fmt", [E4M3FN, E5M2])
def test_qdq_matches_library_round_trip_in_range(orc, fmt):
    """In range, DQ(Q(x)) equals the library's cast to FP8 and back, times the scale, as bf16."""
    x = ALL_BF16_F32
    for s in QDQ_SCALES:
        s32 = np.float32(s)
        with np.errstate(all="ignore"):
            yq = (x / s32).astype(np.float32)
        inr = np.isfinite(yq) & (np.abs(yq) <= FP8_MAX[fmt])
        fp = torch.from_numpy(np.where(inr, yq, 0).astype(np.float32)).to(TORCH_FP8[fmt]).to(torch.float32)
        want = (fp * torch.tensor(s32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        got, _ = orc.qdq_amax(ALL_BF16, fmt, s32)
        assert np.array_equal(got[inr], want[inr]), f"scale {s}"


@pytest.mark.parametrize("fmt", [E4M3FN, E5M2])
def test_qdq_error_bound_saturation_and_idempotence(orc, fmt):
    x = ALL_BF16_F32
    fin = np.isfinite(x)
    for s in (1.0, 2.0 ** -4, 2.0 ** 6):   # powers of two: the fp32 product is exact
        y, a = orc.qdq_amax(ALL_BF16, fmt, s)
        yf = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        # saturation: |DQ(Q(x))| never exceeds FP8_MAX * scale (rounded to bf16)
        assert np.all(np.abs(yf[fin]) <= FP8_MAX[fmt] * s * (1 + 2.0 ** -8))
        # in range the error is at most half an FP8 step (relative 2^-4 or 2^-3) plus the
        # subnormal floor, and the bf16 rounding of an exact FP8 value adds nothing
        xs = x[fin].astype(np.float64)
        inr = np.abs(xs) <= FP8_MAX[fmt] * s
        rel = 2.0 ** -4 if fmt == E4M3FN else 2.0 ** -3
        floor = (2.0 ** -10 if fmt == E4M3FN else 2.0 ** -17) * s
        err = np.abs(yf[fin][inr] - xs[inr])
        assert np.all(err <= rel * np.abs(xs[inr]) + floor)
        # idempotence: QDQ(QDQ(x)) == QDQ(x)
        y2, _ = orc.qdq_amax(y, fmt, s)
        nan = np.isnan(yf)
        assert np.array_equal(y2[~nan], y[~nan])
        # amax is the plain max|x| (NaN among the inputs makes it NaN)
        assert math.isnan(float(a))


def test_qdq_amax_and_representable_identity(orc):
    for fmt in (E4M3FN, E5M2):
        vals = [orc.fp8_decode(c, fmt) for c in range(256)]
        vals = [v * 8.0 for v in vals if math.isfinite(v)]
        xb = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        y, a = orc.qdq_amax(xb, fmt, 8.0)
        assert np.array_equal(y, xb)
        assert float(a) == max(abs(v) for v in vals)


# --------------------------------------------------------------------------- ring-buffer history

def _ring_logical(hist, head):
    """Unrotate a ring history into the rolled layout (row 0 newest)."""
    H, S = hist.shape
    out = np.empty_like(hist)
    for s in range(S):
        for r in range(H):
            out[r, s] = hist[(head[s] - r) % H, s]
    return out


def test_ring_equals_roll_for_any_sequence(orc):
    """Same window contents and the same scales as the rolled history after every call."""
    rng = np.random.default_rng(21)
    for H in (1, 2, 3, 5, 8):
        for S in (1, 3, 6):
            for algo in (0, 1):
                hist_r = np.zeros((H, S), np.float32)
                hist_g = np.zeros((H, S), np.float32)
                start = rng.integers(0, H, S).astype(np.int32)       # arbitrary starting positions
                head = start.copy()
                sc_r, si_r = np.ones(S, np.float32), np.ones(S, np.float32)
                sc_g, si_g = sc_r.copy(), si_r.copy()
                sf = (np.arange(S) % 2).astype(np.uint8)
                for k in range(2 * H + 3):
                    new = np.exp(rng.normal(0, 3, S)).astype(np.float32)
                    new[rng.random(S) < 0.15] = 0.0
                    if k == H:
                        new[0] = np.nan
                    margin = int(rng.integers(-2, 3))
                    orc.amax_scale_update(hist_r, new, sc_r, si_r, E4M3FN, algo, margin, sf)
                    orc.amax_scale_update_ring(hist_g, head, new, sc_g, si_g, E4M3FN, algo, margin, sf)
                    assert np.array_equal(head, ((start + k + 1) % H).astype(np.int32))
                    lg = _ring_logical(hist_g, head)
                    assert np.array_equal(np.isnan(lg), np.isnan(hist_r))
                    assert np.array_equal(np.nan_to_num(lg), np.nan_to_num(hist_r)), (H, S, k)
                    assert np.array_equal(sc_g, sc_r) and np.array_equal(si_g, si_r), (H, S, algo, k)


def test_ring_writes_exactly_one_row_per_slot(orc):
    H, S = 6, 4
    hist = np.arange(H * S, dtype=np.float32).reshape(H, S) + 1
    head = np.array([0, 5, 2, 3], np.int32)
    before = hist.copy()
    orc.amax_scale_update_ring(hist, head, np.full(S, 99.0, np.float32), np.ones(S, np.float32),
                               np.ones(S, np.float32))
    changed = hist != before
    assert changed.sum() == S
    for s, h in enumerate([1, 0, 3, 4]):
        assert changed[h, s] and hist[h, s] == 99.0


def test_ring_invalid_head_leaves_slot_alone(orc):
    H, S = 4, 3
    hist = np.full((H, S), 2.0, np.float32)
    head = np.array([-1, 4, 1], np.int32)
    sc = np.full(S, 5.0, np.float32)
    si = np.full(S, 0.2, np.float32)
    orc.amax_scale_update_ring(hist, head, np.full(S, 448.0, np.float32), sc, si)
    assert list(head) == [-1, 4, 2]
    assert np.all(hist[:, :2] == 2.0) and sc[0] == 5.0 and sc[1] == 5.0
    assert hist[2, 2] == 448.0 and sc[2] == 1.0


def test_fp32_max_grad_example_accumulates_with_max(orc):
    """The worked example of "User Guide on Native XLA-FP8", section "Gradient
    accumulation of FP8 params": x = 2, amax history [0, 0, 0], scaling factor 1,
    three in_qdq iterations.  Each round trip returns 2 exactly (2 is an e4m3fn
    value); the amax seen over the three iterations, accumulated with max as the
    section asks, is 2 (an add would give 6); one update then puts it at the
    front of the length-3 history and sets the scale to RN(2 / 448)."""
    x = np.array([0x4000], np.uint16)  # 2.0 in bf16
    amax = np.float32(0.0)
    for _ in range(3):
        y, amax = orc.qdq_amax(x, E4M3FN, np.float32(1.0), amax)
        assert list(y) == [0x4000]
    assert amax == np.float32(2.0)
    hist = np.zeros((3, 1), np.float32)
    sc = np.ones(1, np.float32)
    si = np.ones(1, np.float32)
    orc.amax_scale_update(hist, np.array([amax], np.float32), sc, si)
    assert list(hist[:, 0]) == [2.0, 0.0, 0.0]
    assert sc[0] == np.float32(2.0) / np.float32(448.0) and si[0] == np.float32(1.0) / sc[0]


def test_ring_update_then_quantize_hand_example(orc):
    """The update fused with the next quantize: hand-derived values.  H = 4, S = 2,
    an empty history with both heads at row 3, new amaxes 2 and 3584: the new
    entries go to row 0, the windows' maxima are 2 and 3584, so scale[1] = 3584 / 448
    = 8 and scale[0] = 2 / 448.  x = (8, -16, 448, 1e9, -0) quantized with scale 8:
    1 -> 0x38, -2 -> 0xC0, 56 -> 0x66 (1.75 * 2^5), 1.25e8 saturates -> 0x7E, -0 -> 0x80."""
    hist = np.zeros((4, 2), np.float32)
    head = np.array([3, 3], np.int32)
    sc = np.ones(2, np.float32)
    si = np.ones(2, np.float32)
    x = np.array([0x4100, 0xC180, 0x43E0, 0x4E6E, 0x8000], np.uint16)  # 8, -16, 448, ~1e9, -0 in bf16
    q, a = orc.amax_scale_update_ring_quantize(hist, head, np.array([2.0, 3584.0], np.float32), sc, si, x, 1)
    assert list(head) == [0, 0]
    assert hist[0, 0] == 2.0 and hist[0, 1] == 3584.0 and np.all(hist[1:] == 0.0)
    assert sc[1] == 8.0 and si[1] == 0.125 and sc[0] == np.float32(2.0) / np.float32(448.0)
    assert list(q) == [0x38, 0xC0, 0x66, 0x7E, 0x80]
    assert a == np.float32((np.uint32(0x4E6E) << 16).view(np.float32))


# --------------------------------------------------------------------------- producers (float64 definitions)

def test_f64_to_bf16_hand_cases(orc):
    """One rounding from float64 to bf16, hand-derived (tests/golden/bf16_from_f64_cases.txt)."""
    for expr, want in _golden("bf16_from_f64_cases.txt"):
        got = orc.f64_to_bf16(_val(expr))
        assert got == int(want, 16), f"{expr}: got {got:04X} want {want}"
    assert orc.f64_to_bf16(math.nan) & 0x7FFF > 0x7F80


def test_f64_to_bf16_on_binary32_values_equals_the_binary32_rounding(orc):
    """On values exactly representable in binary32, one rounding from float64 is the
    binary32 -> bf16 rounding (itself pinned by hand cases and torch)."""
    rng = np.random.default_rng(51)
    bits = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    got = orc.f64_to_bf16_array(f.astype(np.float64))
    want = np.array([orc.f32_to_bf16(v) for v in f[:4000]], np.uint16)
    assert np.array_equal(got[:4000], want)
    want_t = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want_t)


FINITE_BF16 = ALL_BF16_F32[np.isfinite(ALL_BF16_F32)]


def test_gelu_ref_equals_the_tanh_form_in_high_precision(orc):
    """The literal formula 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) evaluated with
    120 significant digits (mpmath; at x = -12, 1 + tanh(u) is about 1e-62), on every
    third finite bf16 input with |x| <= 12 (below -10.5 the result is far under bf16's
    smallest value)."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 120
    xs = FINITE_BF16[np.abs(FINITE_BF16) <= 12.0].astype(np.float64)
    xs = xs[::3]
    k = mp.sqrt(2 / mp.pi)
    worst = 0.0
    for x in xs:
        xm = mp.mpf(float(x))
        want = 0.5 * xm * (1 + mp.tanh(k * (xm + mp.mpf("0.044715") * xm ** 3)))
        got = orc.gelu_ref(float(x))
        if want == 0:
            assert got == 0.0
            continue
        rel = abs((mp.mpf(got) - want) / want)
        worst = max(worst, float(rel))
    assert worst < 1e-13, worst


def test_gelu_ref_odd_part_is_x(orc):
    """GELU(x) - GELU(-x) = x: the tanh form is x times a sigmoid of an odd argument."""
    xs = FINITE_BF16[(FINITE_BF16 > 0) & (FINITE_BF16 < 1e4)].astype(np.float64)
    d = np.array([orc.gelu_ref(x) - orc.gelu_ref(-x) for x in xs[::2]])
    assert np.all(np.abs(d - xs[::2]) <= 4e-16 * xs[::2])


def test_gelu_ref_matches_torch_float64(orc):
    """torch's tanh GELU in float64 where its 1 + tanh(u) is free of cancellation
    (x > -2: there 1 + tanh(u) > 0.04, so float64 keeps 14 digits of it)."""
    x = FINITE_BF16[(FINITE_BF16 > -2) & (FINITE_BF16 < 5)].astype(np.float64)
    got = orc.gelu_ref_array((x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16))
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    nz = ref != 0
    assert np.all(np.abs(got[nz] - ref[nz]) <= 1e-13 * np.abs(ref[nz]))
    assert np.all(got[~nz] == 0.0)


def test_gelu_ref_special_values(orc):
    assert orc.gelu_ref(0.0) == 0.0
    assert orc.gelu_ref(math.inf) == math.inf
    g = orc.gelu_ref(-math.inf)
    assert g == 0.0 and math.copysign(1, g) < 0          # the limit
    assert orc.gelu_ref(-1e30) == 0.0
    assert orc.gelu_ref(1e30) == 1e30
    assert math.isnan(orc.gelu_ref(math.nan))
    assert orc.gelu_ref(3.0) == pytest.approx(3.0 * 0.5 * (1 + math.tanh(math.sqrt(2 / math.pi) * (3 + 0.044715 * 27))),
                                              rel=1e-15)


def _ln_rows(rng, rows, H, spread=1.0):
    x = (rng.normal(0, spread, (rows, H)) + rng.normal(0, 2 * spread, (rows, 1))).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16)


def _u16(x):
    return x.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("H", [16, 272, 4096, 16384])
def test_layernorm_ref_matches_torch_float64(orc, H):
    """torch's layer_norm (two-pass statistics) in float64 on rows with a large mean."""
    rng = np.random.default_rng(H)
    x = _ln_rows(rng, 6, H)
    g = rng.uniform(0.5, 1.5, H).astype(np.float32)
    b = rng.normal(0, 0.2, H).astype(np.float32)
    y, mean, rstd = orc.layernorm_ref(_u16(x), H, g, b, 1e-6)
    ref = torch.nn.functional.layer_norm(x.double(), (H,), torch.from_numpy(g).double(),
                                         torch.from_numpy(b).double(), eps=1e-6).numpy().reshape(-1)
    assert np.all(np.abs(y - ref) <= 1e-11 * (np.abs(ref) + 1.0))
    x64 = x.double().numpy()
    assert np.allclose(mean, x64.mean(axis=1), rtol=1e-14, atol=1e-14)
    assert np.allclose(rstd, 1.0 / np.sqrt(x64.var(axis=1) + 1e-6), rtol=1e-12)


def test_layernorm_ref_closed_forms(orc):
    """Constant rows give beta exactly; a row +a, -a, +a, ... has mean 0 and variance a^2."""
    H = 64
    b = np.linspace(-1, 1, H).astype(np.float32)
    g = np.full(H, 3.0, np.float32)
    x = torch.full((3, H), 2.5).to(torch.bfloat16)
    y, mean, rstd = orc.layernorm_ref(_u16(x), H, g, b, 1e-6)
    assert np.array_equal(y, np.tile(b.astype(np.float64), 3))
    assert np.all(mean == 2.5) and np.allclose(rstd, 1000.0, rtol=1e-15)
    a = 1.5
    x = torch.tensor(np.where(np.arange(H) % 2 == 0, a, -a), dtype=torch.float32).reshape(1, H).to(torch.bfloat16)
    for eps in (1e-6, 0.25):
        y, mean, rstd = orc.layernorm_ref(_u16(x), H, g, b, eps)
        sgn = np.where(np.arange(H) % 2 == 0, 1.0, -1.0)
        want = sgn * a / math.sqrt(a * a + eps) * 3.0 + b.astype(np.float64)
        assert mean[0] == 0.0
        assert np.allclose(y, want, rtol=1e-15, atol=1e-15)


def test_layernorm_ref_propagates_nan_and_inf(orc):
    H = 32
    x = np.full((3, H), 0x3F80, np.uint16)
    x[0, 3] = 0x7FC0
    x[1, 4] = 0x7F80
    x[2, 5] = 0xFF80
    y, _, _ = orc.layernorm_ref(x, H, np.ones(H, np.float32), np.zeros(H, np.float32), 1e-6)
    assert np.all(np.isnan(y))


def _f32_tree_sum(a):
    """Row sums of a float32 [rows, H] array (H a multiple of 8) in binary32: runs of
    8 added left to right, then a pairwise tree (longest chain 8 + log2(H / 8))."""
    a = a.astype(np.float32)
    rows, H = a.shape
    leaves = a.reshape(rows, H // 8, 8)
    s = np.zeros((rows, H // 8), np.float32)
    for k in range(8):
        s = (s + leaves[:, :, k]).astype(np.float32)
    while s.shape[1] > 1:
        if s.shape[1] % 2:
            s = np.concatenate([s, np.zeros((rows, 1), np.float32)], axis=1)
        s = (s[:, 0::2] + s[:, 1::2]).astype(np.float32)
    return s[:, 0]


def _ln_f32(x, g, b, eps):
    """LayerNorm in binary32 with Flax's formula and tree-ordered sums."""
    xf = x.float().numpy().astype(np.float32)
    H = xf.shape[1]
    S = _f32_tree_sum(xf)
    Q = _f32_tree_sum((xf * xf).astype(np.float32))
    mean = (S / np.float32(H)).astype(np.float32)
    var = np.maximum((Q / np.float32(H)).astype(np.float32) - (mean * mean).astype(np.float32), np.float32(0))
    rstd = (np.float32(1) / np.sqrt((var + np.float32(eps)).astype(np.float32))).astype(np.float32)
    d = (xf - mean[:, None]).astype(np.float32)
    m = (rstd[:, None] * g[None, :]).astype(np.float32)
    yf = ((d * m).astype(np.float32) + b[None, :]).astype(np.float32)
    return torch.from_numpy(yf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).reshape(-1)


@pytest.mark.parametrize("H", [64, 1024, 4096])
def test_layernorm_tolerance_holds_a_binary32_evaluation(orc, H):
    """A plain binary32 LayerNorm, sums well within the allowed chain length, lands
    inside the stated tolerance, also on rows whose mean dwarfs their spread."""
    rng = np.random.default_rng(61 + H)
    rows = 8
    mu = np.array([0.0, 2.0, -2.0, 30.0, 0.5, -40.0, 1.0, 3.0])[:, None]
    sd = np.array([1.0, 0.5, 0.5, 0.3, 4.0, 1.0, 1e-3, 2.0])[:, None]
    x = torch.from_numpy((rng.normal(0, 1, (rows, H)) * sd + mu).astype(np.float32)).to(torch.bfloat16)
    g = (1 + 0.1 * rng.normal(0, 1, H)).astype(np.float32)
    b = (0.1 * rng.normal(0, 1, H)).astype(np.float32)
    y32 = _ln_f32(x, g, b, 1e-6)
    r, mean, rstd = orc.layernorm_ref(_u16(x), H, g, b, 1e-6)
    E = orc.layernorm_tolerance(x.double().numpy(), g, b, 1e-6, mean, rstd, r)
    assert np.all(orc.bf16_within(y32, r, E.reshape(-1)))
    # On rows whose spread is not dwarfed by their mean the tolerance leaves one value
    # for almost every element (rows 3, 5 and 6 lose most of var = E[x^2] - mean^2 to
    # cancellation in binary32, and the tolerance widens accordingly).
    lo = orc.f64_to_bf16_array(r - E.reshape(-1)).reshape(rows, H)
    hi = orc.f64_to_bf16_array(r + E.reshape(-1)).reshape(rows, H)
    benign = [0, 1, 2, 4, 7]
    assert np.mean(lo[benign] == hi[benign]) > 0.9


def _f32_chain_sum(a, L):
    """Row sums in binary32: chains of L elements added left to right, then a pairwise
    tree over the chains (longest chain L + ceil(log2(H / L)))."""
    a = a.astype(np.float32)
    rows, H = a.shape
    nc = H // L
    s = np.zeros((rows, nc), np.float32)
    leaves = a.reshape(rows, nc, L)
    for k in range(L):
        s = (s + leaves[:, :, k]).astype(np.float32)
    while s.shape[1] > 1:
        if s.shape[1] % 2:
            s = np.concatenate([s, np.zeros((rows, 1), np.float32)], axis=1)
        s = (s[:, 0::2] + s[:, 1::2]).astype(np.float32)
    return s[:, 0]


@pytest.mark.parametrize("H", [1024, 4096, 16384])
def test_layernorm_tolerance_holds_the_longest_allowed_chains(orc, H):
    """The tolerance covers any binary32 evaluation whose sums have chains of additions up
    to D = H/128 + 32 long: here chains as long as that allows, left to right, and the
    normalisation fused (one rounding for (x - mean) * (rstd * gamma) + beta), on rows with
    outliers, large means and small spreads."""
    D = H // 128 + 32
    L = 1
    while 2 * L + int(np.ceil(np.log2(H / (2 * L)))) <= D and 2 * L <= H:
        L *= 2
    assert L + int(np.ceil(np.log2(H / L))) <= D
    rng = np.random.default_rng(97 + H)
    rows = 12
    mu = np.array([0.0, 2.0, -2.0, 30.0, 0.5, -40.0, 1.0, 3.0, 0.0, 100.0, -0.01, 7.0])[:, None]
    sd = np.array([1.0, 0.5, 0.5, 0.3, 4.0, 1.0, 1e-3, 2.0, 50.0, 1.0, 0.1, 1e-2])[:, None]
    xv = rng.normal(0, 1, (rows, H)) * sd + mu
    out = rng.random((rows, H)) < 1e-3
    xv[out] *= 100.0
    x = torch.from_numpy(xv.astype(np.float32)).to(torch.bfloat16)
    g = (1 + 0.1 * rng.normal(0, 1, H)).astype(np.float32)
    b = (0.1 * rng.normal(0, 1, H)).astype(np.float32)
    xf = x.float().numpy().astype(np.float32)
    S = _f32_chain_sum(xf, L)
    Q = _f32_chain_sum((xf * xf).astype(np.float32), L)
    mean = (S / np.float32(H)).astype(np.float32)
    var = np.maximum((Q / np.float32(H)).astype(np.float32) - (mean * mean).astype(np.float32), np.float32(0))
    rstd = (np.float32(1) / np.sqrt((var + np.float32(1e-6)).astype(np.float32))).astype(np.float32)
    d = (xf - mean[:, None]).astype(np.float32)
    m = (rstd[:, None] * g[None, :]).astype(np.float32)
    yf = (d.astype(np.float64) * m.astype(np.float64) + b[None, :].astype(np.float64)).astype(np.float32)
    y32 = torch.from_numpy(yf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).reshape(-1)
    r, mean64, rstd64 = orc.layernorm_ref(_u16(x), H, g, b, 1e-6)
    E = orc.layernorm_tolerance(x.double().numpy(), g, b, 1e-6, mean64, rstd64, r)
    ok = orc.bf16_within(y32, r, E.reshape(-1))
    assert ok.all(), f"{(~ok).sum()} elements outside, rows {np.unique(np.nonzero(~ok)[0] // H)}"


def test_gelu_tolerance_at_infinity_is_exact(orc):
    r = orc.gelu_ref_array(np.array([0x7F80, 0xFF80], np.uint16))
    E = orc.gelu_tolerance(np.array([math.inf, -math.inf]), r)
    assert E[0] == 0.0 and E[1] == orc.GELU_TINY
    assert list(orc.bf16_within(np.array([0x7F80, 0x8000], np.uint16), r, E)) == [True, True]
    assert not orc.bf16_within(np.array([0x7F7F], np.uint16), r[:1], E[:1])[0]


def test_gelu_tolerance_is_not_vacuous(orc):
    """The GELU tolerance leaves one acceptable value for almost every bf16 input whose
    GELU is at least 2^-122 (below that, the binary32 reciprocal is subnormal or zero,
    and any value within 2^-122 is accepted)."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    fin = np.isfinite(x)
    r = orc.gelu_ref_array(h)[fin]
    E = orc.gelu_tolerance(x[fin], r)
    lo = orc.f64_to_bf16_array(r - E)
    hi = orc.f64_to_bf16_array(r + E)
    big = np.abs(r) >= orc.GELU_TINY
    assert big.sum() > 30000
    assert np.mean((lo == hi)[big]) > 0.97


def test_bf16_within_accepts_only_the_interval(orc):
    r = np.array([1.0 + 2.0 ** -8, 1.0 + 2.0 ** -9, -3.0, math.nan, 0.0])
    E = np.array([2.0 ** -30, 2.0 ** -30, 0.0, 0.0, 2.0 ** -140])
    y_ok = np.array([0x3F81, 0x3F80, 0xC040, 0x7FC1, 0x8000], np.uint16)
    assert np.all(orc.bf16_within(y_ok, r, E))
    y_other = np.array([0x3F80, 0x3F81, 0xC041, 0x3F80, 0x0001], np.uint16)
    ok = orc.bf16_within(y_other, r, E)
    # 1 + 2^-8 +- 2^-30 straddles the tie: both neighbours are acceptable
    assert list(ok) == [True, False, False, False, False]


def test_gelu_tolerance_rejects_a_wrong_gelu(orc):
    """The GELU bar is discriminating: a binary32 GELU whose cubic coefficient is off by
    0.01% (0.04471) lands outside the tolerance on some bf16 inputs, and so does one that
    goes through a tanh accurate to only 2^-11 (as a hardware approximation is)."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = (h.astype(np.uint32) << 16).view(np.float32)
    fin = np.isfinite(x) & (np.abs(x) < 8)
    hf, xf = h[fin], x[fin].astype(np.float64)
    r = orc.gelu_ref_array(hf)
    E = orc.gelu_tolerance(xf, r)

    def bf16(v):
        return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    x32 = x[fin].astype(np.float32)
    k = np.float32(math.sqrt(2.0 / math.pi))
    wrong_c = x32 * np.float32(0.5) * (np.float32(1) + np.tanh(k * (x32 + np.float32(0.04471) * x32 ** 3)))
    assert (~orc.bf16_within(bf16(wrong_c), r, E)).sum() > 20
    t = np.tanh(xf * math.sqrt(2 / math.pi) * (1 + 0.044715 * xf * xf))
    coarse = 0.5 * xf * (1 + t * (1 + 2.0 ** -11))
    assert (~orc.bf16_within(bf16(coarse), r, E)).sum() > 20


def test_layernorm_tolerance_rejects_a_wrong_layernorm(orc):
    """The LayerNorm bar is discriminating: rows normalised with eps = 1e-5 instead of
    1e-6, or with the unbiased variance (divided by H - 1), land outside it."""
    rng = np.random.default_rng(71)
    H, rows = 1024, 16
    x = torch.from_numpy((rng.normal(0, 1, (rows, H)) * rng.uniform(0.05, 3, (rows, 1))
                          + rng.normal(0, 1, (rows, 1))).astype(np.float32)).to(torch.bfloat16)
    g = (1 + 0.1 * rng.normal(0, 1, H)).astype(np.float32)
    b = (0.1 * rng.normal(0, 1, H)).astype(np.float32)
    r, mean, rstd = orc.layernorm_ref(_u16(x), H, g, b, 1e-6)
    E = orc.layernorm_tolerance(x.double().numpy(), g, b, 1e-6, mean, rstd, r)
    x64 = x.double().numpy()
    for wrong in (torch.nn.functional.layer_norm(x.double(), (H,), torch.from_numpy(g).double(),
                                                 torch.from_numpy(b).double(), eps=1e-5).numpy(),
                  (x64 - x64.mean(1, keepdims=True)) / np.sqrt(x64.var(1, ddof=1, keepdims=True) + 1e-6) * g + b):
        yb = torch.from_numpy(wrong.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert (~orc.bf16_within(yb.reshape(-1), r, E.reshape(-1))).sum() > 20
