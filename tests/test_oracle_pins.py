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


# --------------------------------------------------------------------------- GELU producer fused with Q

def _ulp32(x):
    x = np.abs(np.asarray(x, np.float32))
    return (np.nextafter(x, np.float32(np.inf)) - x).astype(np.float64)


def test_exp_within_a_few_ulp_of_the_true_value(orc):
    """The GELU's exp: within 3 ulp of e^v on [-20, 88.7]; clamped outside (below -20,
    1 + e^v is exactly 1 in binary32 whatever e^v is; above 88.73 it overflows)."""
    rng = np.random.default_rng(31)
    vs = np.concatenate([np.linspace(-20, 88.7, 4001), rng.uniform(-20, 88.7, 4000),
                         rng.uniform(-1, 1, 2000)]).astype(np.float32)
    got = np.array([orc.exp_f32(v) for v in vs], np.float64)
    ref = np.exp(vs.astype(np.float64))
    assert np.all(np.abs(got - ref) <= 3 * _ulp32(ref))
    assert orc.exp_f32(0.0) == 1.0
    assert np.isinf(orc.exp_f32(88.8)) and np.isinf(orc.exp_f32(np.inf))
    e20 = orc.exp_f32(-20.0)
    for v in (-20.5, -100.0, -np.inf, np.nan):
        assert orc.exp_f32(v) == e20
    assert np.float32(1.0) + e20 == np.float32(1.0)


def _gelu_tanh_f64(x):
    """The tanh GELU in float64, written as x / (1 + exp(-2u)): the same function as
    0.5 x (1 + tanh(u)), without that form's cancellation for negative x."""
    x = np.asarray(x, np.float64)
    u = math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)
    return x / (1.0 + np.exp(-2.0 * u))


def test_gelu_close_to_the_float64_tanh_form(orc):
    rng = np.random.default_rng(32)
    xs = np.concatenate([np.linspace(-9, 9, 6001), rng.normal(0, 3, 6000),
                         rng.uniform(-0.01, 0.01, 500)]).astype(np.float32)
    got = np.array([orc.gelu_f32(x) for x in xs], np.float64)
    ref = _gelu_tanh_f64(xs)
    tiny = np.abs(ref) < 2.0 ** -120
    rel = np.abs(got - ref)[~tiny] / np.abs(ref[~tiny])
    assert rel.max() < 2.0 ** -16          # far below bf16's resolution (2^-8)
    assert np.all(np.abs(got[tiny] - ref[tiny]) < 2.0 ** -110)


def test_gelu_bf16_matches_torch_tanh_gelu(orc):
    """On bf16 inputs, bf16(GELU) equals torch's tanh GELU (in float64) rounded to bf16,
    except within one bf16 step where the value sits on a rounding tie."""
    # |x| < 5 keeps torch's 0.5 x (1 + tanh(u)) free of cancellation in float64
    x = ALL_BF16_F32[np.isfinite(ALL_BF16_F32) & (np.abs(ALL_BF16_F32) < 5)]
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    _, y, _ = orc.gelu_quantize_amax(xb, E4M3FN, 1.0)
    ref = torch.nn.functional.gelu(torch.from_numpy(x.astype(np.float64)), approximate="tanh")
    refb = ref.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    same = y == refb
    assert same.mean() > 0.995  # ties: |error| < 2^-16 relative against bf16 steps of 2^-8
    yf = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rf = (refb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    step = np.maximum(np.abs(rf), 2.0 ** -126) * 2.0 ** -7
    assert np.all(np.abs(yf - rf)[~same] <= step[~same])


def test_gelu_special_values(orc):
    assert orc.gelu_f32(0.0) == 0.0
    assert orc.gelu_f32(np.inf) == np.inf
    g = orc.gelu_f32(-np.inf)
    assert g == 0.0 and math.copysign(1, g) < 0
    g = orc.gelu_f32(-1e30)
    assert g == 0.0 and math.copysign(1, g) < 0
    assert orc.gelu_f32(1e30) == np.float32(1e30)
    assert np.isnan(orc.gelu_f32(np.nan))


@pytest.mark.parametrize("fmt", [E4M3FN, E5M2])
def test_fused_gelu_quantize_is_quantize_of_the_bf16_gelu(orc, fmt):
    rng = np.random.default_rng(33)
    h = (rng.normal(0, 2, 5000).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    for s in (1.0, 0.0123, 2.0 ** -70):
        q, y, a = orc.gelu_quantize_amax(h, fmt, s)
        q2, a2 = orc.quantize_amax(y, fmt, s)
        assert np.array_equal(q, q2) and a == a2
        yf = (y.astype(np.uint32) << 16).view(np.float32)
        assert a == np.max(np.abs(yf)) == orc.gelu_amax(h)


# --------------------------------------------------------------------------- LayerNorm producer fused with Q

def _ln_rows(rng, rows, H, spread=1.0):
    x = (rng.normal(0, spread, (rows, H)) + rng.normal(0, 2 * spread, (rows, 1))).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16)


@pytest.mark.parametrize("H", [16, 272, 4096, 16384])
def test_layernorm_stats_close_to_float64(orc, H):
    rng = np.random.default_rng(H)
    x = _ln_rows(rng, 6, H)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    x64 = x.double().numpy()
    for r in range(6):
        mean, rstd = orc.layernorm_stats(xb[r])
        m64 = x64[r].mean()
        v64 = x64[r].var()
        assert abs(mean - m64) <= 2.0 ** -18 * np.abs(x64[r]).max()
        assert abs(rstd * math.sqrt(v64 + 1e-6) - 1.0) <= 2.0 ** -14


def test_layernorm_output_close_to_torch(orc):
    rng = np.random.default_rng(41)
    H = 4096
    x = _ln_rows(rng, 16, H)
    g = rng.uniform(0.5, 1.5, H).astype(np.float32)
    b = rng.normal(0, 0.2, H).astype(np.float32)
    _, y, a = orc.layernorm_quantize_amax(x.view(torch.int16).numpy().view(np.uint16), H, g, b, E4M3FN, 1.0)
    ref = torch.nn.functional.layer_norm(x.double(), (H,), torch.from_numpy(g).double(),
                                         torch.from_numpy(b).double(), eps=1e-6)
    refb = ref.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).reshape(-1)
    same = y == refb
    assert same.mean() > 0.99                      # the rest: bf16 rounding ties
    yf = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rf = ref.numpy().reshape(-1)
    assert np.all(np.abs(yf - rf) <= 2.0 ** -8 * np.abs(rf) + 2.0 ** -14)
    assert a == np.max(np.abs(yf))


def test_layernorm_constant_rows_give_beta(orc):
    H = 64
    x = torch.full((3, H), 2.5).to(torch.bfloat16)
    g = np.full(H, 3.0, np.float32)
    b = np.linspace(-1, 1, H).astype(np.float32)
    _, y, _ = orc.layernorm_quantize_amax(x.view(torch.int16).numpy().view(np.uint16), H, g, b, E4M3FN, 1.0)
    want = torch.from_numpy(np.tile(b, 3)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(y, want)


@pytest.mark.parametrize("fmt", [E4M3FN, E5M2])
def test_fused_layernorm_quantize_is_quantize_of_its_output(orc, fmt):
    rng = np.random.default_rng(42)
    H = 1024
    x = _ln_rows(rng, 5, H, 3.0)
    g = rng.uniform(0.5, 1.5, H).astype(np.float32)
    b = rng.normal(0, 0.2, H).astype(np.float32)
    for s in (1.0, 0.0123, 7.5):
        q, y, a = orc.layernorm_quantize_amax(x.view(torch.int16).numpy().view(np.uint16), H, g, b, fmt, s)
        q2, a2 = orc.quantize_amax(y, fmt, s)
        assert np.array_equal(q, q2) and a == a2
