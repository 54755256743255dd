/*
 * fp8q_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU definition of every result the FP8
 * delayed-scaling path computes.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the product library never does and
 * shares no code, header, table or constant with it.
 *
 * Sources (web pages, cited by title and section):
 *   [XLA-FP8]  NVIDIA JAX-Toolbox, "User Guide on Native XLA-FP8":
 *              opening section (E4M3/E5M2 formats, quantization Q and
 *              de-quantization DQ), section "JAX" (the delayed-scaling example:
 *              Q = cast(A / A_scale), DQ = cast(a_fp8) * a_scale,
 *              A_scale = max|A| / E4M3_MAX), section "Gradient accumulation of
 *              FP8 params" (FP8 meta accumulates with max; zero history and
 *              unit scale as the initial state).
 *   [XLA-7432] openxla/xla issue "Fusion of Fp8 quantization and amax
 *              reduction kernels": the amax reduction = max|x| per tensor,
 *              fused with the quantization.
 *   [TE-593]   NVIDIA/TransformerEngine PR "Implement fused kernel for FP8
 *              scale update": amax_and_scale_update = amax-history roll,
 *              amax selection from the history, scale and scale_inv, in place,
 *              batched over all layers.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - Q divides by scale in fp32 (IEEE, round to nearest even), then rounds
 *     once more to the FP8 grid (nearest, ties to the even code), saturating
 *     to +-448 (e4m3fn) or +-57344 (e5m2); +-inf saturates too.  A NaN input
 *     gives the code 0x7F (any NaN code is accepted by the parity tests).
 *   - amax = max|x| in fp32; any NaN makes it NaN; it is max-accumulated into
 *     the caller's value, which must start non-negative.
 *   - DQ = RNE_bf16(RN_f32(decode(q) * scale)); a NaN result is any NaN.
 *   - History: row 0 is the newest; the roll moves every row one step older,
 *     drops the oldest and inserts the new amax as row 0 before selection.
 *     Selection "max" is the max over the rolled window (NaN propagates),
 *     "most_recent" is row 0.  scale = RN(a / FP8_MAX) * 2^margin and
 *     scale_inv = RN(1 / scale) are written only when a is finite and > 0 and
 *     the new scale is a normal float; otherwise both pass through unchanged.
 *
 * Build: plain C11, no intrinsics, -ffp-contract=off, no fast-math, so float
 * arithmetic is IEEE binary32 with round-to-nearest-even on x86-64 and
 * AArch64 alike.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "fp8q_oracle.h"

/* ----------------------------------------------------------------------- */
/* bf16 and fp32 bit views.                                                 */

static float bits_to_f32(uint32_t b) {
    float f;
    memcpy(&f, &b, sizeof f);
    return f;
}

static uint32_t f32_to_bits(float f) {
    uint32_t b;
    memcpy(&b, &f, sizeof b);
    return b;
}

/* bf16 is the upper half of a binary32: widening is exact. */
float orc_bf16_to_f32(uint16_t h) { return bits_to_f32((uint32_t)h << 16); }

/*
 * Round a binary32 value to the nearest bf16, ties to the even bf16 (the one
 * whose last mantissa bit is 0).  Written as the definition: the two bf16
 * neighbours of |f| are the truncation `lo` and the next value up `hi`; pick
 * the nearer by comparing |f| with their midpoint, which is exact in double.
 * A value at or above the midpoint between the largest finite bf16 and 2^128
 * rounds to infinity, as IEEE rounding to a narrower format does.
 */
uint16_t orc_f32_to_bf16(float f) {
    if (isnan(f)) return 0x7FC0;
    uint32_t b = f32_to_bits(f);
    uint32_t sign = b & 0x80000000u;
    uint32_t mag = b & 0x7FFFFFFFu;
    uint32_t lo = mag & 0xFFFF0000u;
    if (lo == mag) return (uint16_t)(b >> 16); /* already a bf16 (or inf) */
    uint32_t hi = lo + 0x10000u;               /* next bf16 up in magnitude */
    double dlo = (double)bits_to_f32(lo);
    double dhi = (hi == 0x7F800000u) ? ldexp(1.0, 128) : (double)bits_to_f32(hi);
    double a = (double)bits_to_f32(mag);
    double mid = 0.5 * (dlo + dhi);
    uint32_t pick;
    if (a < mid) pick = lo;
    else if (a > mid) pick = hi;
    else pick = ((lo >> 16) & 1u) ? hi : lo;
    return (uint16_t)((sign | pick) >> 16);
}

/* ----------------------------------------------------------------------- */
/* FP8 formats ([XLA-FP8] opening section: E4M3 has one more mantissa bit,  */
/* E5M2 one more exponent bit).                                             */
/*   e4m3fn: 1 sign, 4 exponent (bias 7), 3 mantissa; no infinity; S.1111.111 */
/*           is NaN; largest finite 0x7E = 448.                             */
/*   e5m2:   1 sign, 5 exponent (bias 15), 2 mantissa; exponent 31 is inf   */
/*           (mantissa 0) or NaN; largest finite 0x7B = 57344.              */

static int fmt_exp_bits(int fmt) { return fmt == ORC_E4M3FN ? 4 : 5; }
static int fmt_bias(int fmt) { return fmt == ORC_E4M3FN ? 7 : 15; }

int orc_fp8_max_code(int fmt) { return fmt == ORC_E4M3FN ? 0x7E : 0x7B; }

/* Exact value of an FP8 code, decoded from its bit fields. */
double orc_fp8_decode(uint8_t code, int fmt) {
    int ebits = fmt_exp_bits(fmt);
    int mbits = 7 - ebits;
    int bias = fmt_bias(fmt);
    int sign = code >> 7;
    int e = (code >> mbits) & ((1 << ebits) - 1);
    int m = code & ((1 << mbits) - 1);
    double v;
    if (fmt == ORC_E4M3FN && e == 15 && m == 7) return NAN;
    if (fmt == ORC_E5M2 && e == 31) {
        if (m != 0) return NAN;
        return sign ? -INFINITY : INFINITY;
    }
    if (e == 0)
        v = ldexp((double)m, 1 - bias - mbits); /* subnormal: 0.m * 2^(1-bias) */
    else
        v = ldexp((double)((1 << mbits) + m), e - bias - mbits); /* 1.m * 2^(e-bias) */
    return sign ? -v : v;
}

double orc_fp8_max(int fmt) { return orc_fp8_decode((uint8_t)orc_fp8_max_code(fmt), fmt); }

/*
 * Nearest FP8 code to a binary32 value: saturating, ties to the even code.
 * The non-negative finite codes 0..max_code decode to strictly increasing
 * values, so a binary search finds the largest code not above |y|; the answer
 * is that code or the next one, whichever is nearer (midpoint exact in double).
 */
uint8_t orc_fp8_encode(float y, int fmt) {
    if (isnan(y)) return 0x7F;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    int maxc = orc_fp8_max_code(fmt);
    if (a >= orc_fp8_decode((uint8_t)maxc, fmt)) return (uint8_t)(sign | maxc);
    int lo = 0, hi = maxc; /* decode(lo) <= a < decode(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (orc_fp8_decode((uint8_t)mid, fmt) <= a) lo = mid;
        else hi = mid;
    }
    double vlo = orc_fp8_decode((uint8_t)lo, fmt);
    double vhi = orc_fp8_decode((uint8_t)hi, fmt);
    double midv = 0.5 * (vlo + vhi);
    int code;
    if (a < midv) code = lo;
    else if (a > midv) code = hi;
    else code = (lo % 2 == 0) ? lo : hi;
    return (uint8_t)(sign | code);
}

/* ----------------------------------------------------------------------- */
/* Quantize + amax ([XLA-FP8] "JAX": A_fp8 = (A / A_scale).astype(fp8);     */
/* [XLA-7432]: amax reduction max|x| over the same tensor).                 */

/* amax accumulation: max that lets a NaN win over every number. */
static float amax_combine(float acc, float v) {
    if (isnan(acc)) return acc;
    if (isnan(v)) return v;
    return v > acc ? v : acc;
}

void orc_quantize_amax(const uint16_t* x_bf16, int64_t n, int fmt, float scale,
                       uint8_t* q, float* amax_inout) {
    float m = *amax_inout;
    for (int64_t i = 0; i < n; ++i) {
        float x = orc_bf16_to_f32(x_bf16[i]);
        float y = x / scale; /* one IEEE binary32 division, RN */
        q[i] = orc_fp8_encode(y, fmt);
        m = amax_combine(m, fabsf(x));
    }
    if (n > 0) *amax_inout = m;
}

/* A ragged list is each tensor on its own, with its own scale and amax. */
void orc_multi_quantize_amax(const orc_tensor* list, int32_t count, int fmt) {
    for (int32_t t = 0; t < count; ++t)
        orc_quantize_amax(list[t].x_bf16, list[t].n, fmt, list[t].scale, list[t].q,
                          list[t].amax);
}

/* amax alone (used by the workload recipes' "previous step" scales). */
float orc_amax(const uint16_t* x_bf16, int64_t n) {
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) m = amax_combine(m, fabsf(orc_bf16_to_f32(x_bf16[i])));
    return m;
}

/* ----------------------------------------------------------------------- */
/* Dequantize ([XLA-FP8] "JAX": a = a_fp8.astype(bf16) * a_scale, computed  */
/* here as an fp32 product rounded once to bf16).                           */

void orc_dequantize(const uint8_t* q, int64_t n, int fmt, float scale, uint16_t* y_bf16) {
    for (int64_t i = 0; i < n; ++i) {
        float v = (float)orc_fp8_decode(q[i], fmt); /* exact: every FP8 value is a binary32 */
        float p = v * scale;                        /* one binary32 multiply, RN */
        y_bf16[i] = orc_f32_to_bf16(p);
    }
}

/* ----------------------------------------------------------------------- */
/* Fused quantize-then-dequantize ("fake quant") with amax ([XLA-FP8]       */
/* section "Gradient accumulation of FP8 params": in_qdq passes a value     */
/* through Q and DQ with the tensor's scale).  Each element is exactly      */
/* DQ(Q(x)) of the two definitions above.                                   */

void orc_qdq_amax(const uint16_t* x_bf16, int64_t n, int fmt, float scale, uint16_t* y_bf16,
                  float* amax_inout) {
    float m = *amax_inout;
    for (int64_t i = 0; i < n; ++i) {
        float x = orc_bf16_to_f32(x_bf16[i]);
        uint8_t code = orc_fp8_encode(x / scale, fmt);
        float p = (float)orc_fp8_decode(code, fmt) * scale;
        y_bf16[i] = orc_f32_to_bf16(p);
        m = amax_combine(m, fabsf(x));
    }
    if (n > 0) *amax_inout = m;
}

/* ----------------------------------------------------------------------- */
/* GELU producer fused with the quantization ([XLA-7432], test.py: the MLP  */
/* applies nn.gelu, the tanh form, to the first dense layer's output and    */
/* feeds it to an FP8 dense layer; the issue asks for the quantization to   */
/* be fused with what produces its input).                                  */
/*                                                                          */
/* GELU(tanh) = 0.5 x (1 + tanh(u)) = x / (1 + exp(-2u)),                   */
/* u = sqrt(2/pi) (x + 0.044715 x^3).  So that a GPU and a CPU agree bit for */
/* bit, exp is evaluated by additive range reduction (W. J. Cody and W.     */
/* Waite, "Software Manual for the Elementary Functions", 1980) and a        */
/* degree-6 Taylor polynomial of e^r, each step one correctly rounded       */
/* binary32 operation (fmaf where written), in a fixed order.  The constants */
/* are the binary32 roundings of ln 2 split in two (the high part to 16      */
/* significant bits, so k * LN2_HI is exact for |k| < 2^8), of 1 / ln 2, of   */
/* -2 sqrt(2/pi), of 0.044715 and of 1/k!.                                   */

static const float EXP_LN2_HI = 0x1.62e4p-1f;
static const float EXP_LN2_LO = 0x1.7f7d1cp-20f;
static const float EXP_INV_LN2 = 0x1.715476p+0f;
static const float EXP_ROUNDER = 0x1.8p23f;   /* 1.5 * 2^23: adding it rounds to an integer */
static const float GELU_K = -0x1.988454p+0f;  /* -2 sqrt(2/pi) */
static const float GELU_C = 0x1.6e4e26p-5f;   /* 0.044715 */

/* e^v for the GELU below.  v is clamped to [-20, 89]: under -20, 1 + e^v
 * rounds to exactly 1 in binary32 whatever e^v is; over 88.73, e^v
 * overflows to +inf.  k = round(v / ln 2) comes from one fused multiply-add
 * with 1.5 * 2^23 (the sum's last bit is then the integer), r = v - k ln 2 in
 * two parts, e^r by a degree-6 Taylor polynomial (Horner, fused), and
 * e^v = (e^r * 2^(k-1)) * 2: the first product is exact, the second rounds
 * once (to +inf past the largest float). */
float orc_exp_f32(float v) {
    if (v > 89.0f) v = 89.0f;
    if (!(v >= -20.0f)) v = -20.0f;                /* also NaN: GELU returns x * 1 = NaN */
    float t = fmaf(v, EXP_INV_LN2, EXP_ROUNDER);   /* rounds v / ln 2 to the nearest integer */
    float k = t - EXP_ROUNDER;                     /* exact */
    float r = fmaf(-k, EXP_LN2_HI, v);
    r = fmaf(-k, EXP_LN2_LO, r);
    float p = 0x1.6c16c2p-10f;                     /* 1/720 */
    p = fmaf(p, r, 0x1.111112p-7f);                /* 1/120 */
    p = fmaf(p, r, 0x1.555556p-5f);                /* 1/24 */
    p = fmaf(p, r, 0x1.555556p-3f);                /* 1/6 */
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int ki = (int)k;                               /* in [-29, 128] */
    return (p * ldexpf(1.0f, ki - 1)) * 2.0f;
}

float orc_gelu_f32(float x) {
    if (x == -INFINITY) return -0.0f;              /* the limit; x * 0 would be NaN */
    float x2 = x * x;
    float s = x * fmaf(GELU_C, x2, 1.0f);          /* x (1 + 0.044715 x^2) */
    float d = 1.0f + orc_exp_f32(GELU_K * s);      /* 1 + exp(-2u) */
    return x * (1.0f / d);
}

/* y = bf16(GELU(h)); q = FP8(y / scale); amax = max(amax, |y|).  The codes
 * and the amax are those fp8q's quantize gives for the bf16 tensor y. */
void orc_gelu_quantize_amax(const uint16_t* h_bf16, int64_t n, int fmt, float scale, uint8_t* q,
                            uint16_t* y_bf16, float* amax_inout) {
    float m = *amax_inout;
    for (int64_t i = 0; i < n; ++i) {
        uint16_t yb = orc_f32_to_bf16(orc_gelu_f32(orc_bf16_to_f32(h_bf16[i])));
        float y = orc_bf16_to_f32(yb);
        if (y_bf16) y_bf16[i] = yb;
        q[i] = orc_fp8_encode(y / scale, fmt);
        m = amax_combine(m, fabsf(y));
    }
    if (n > 0) *amax_inout = m;
}

/* max|bf16(GELU(h))| alone (the fused op's amax, without the FP8 encoding). */
float orc_gelu_amax(const uint16_t* h_bf16, int64_t n) {
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float y = orc_bf16_to_f32(orc_f32_to_bf16(orc_gelu_f32(orc_bf16_to_f32(h_bf16[i]))));
        m = amax_combine(m, fabsf(y));
    }
    return m;
}

/* ----------------------------------------------------------------------- */
/* LayerNorm producer fused with the quantization ([XLA-7432], test.py: the */
/* transformer block applies nn.LayerNorm() to its input and feeds the      */
/* MLP's first FP8 dense layer; the issue asks for the quantization to be   */
/* fused with what produces its input).                                     */
/*                                                                          */
/* Per row of H elements (H a multiple of 16), in binary32, Flax's defaults: */
/*   mean = S / H, m2 = Q / H with S = sum x, Q = sum x^2,                   */
/*   var = max(0, m2 - mean^2), rstd = 1 / sqrt(var + eps),                 */
/*   y = (x - mean) * (rstd * gamma) + beta, then rounded to bf16.          */
/* S and Q are summed in one fixed association so that any implementation  */
/* can reproduce them bit for bit: the row is cut into vectors of 16        */
/* elements and vector v belongs to lane v mod 256; each lane adds its      */
/* elements in index order (s = s + x, q = fma(x, x, q)); within each group */
/* of 32 lanes the partial sums are folded pairwise, lanes j and j + o for  */
/* o = 16, 8, 4, 2, 1; the 8 group totals are then added left to right.     */

static float row_sum_fixed_order(float* lane) {
    for (int w = 0; w < 8; ++w)
        for (int o = 16; o >= 1; o /= 2)
            for (int j = 0; j < o; ++j) lane[32 * w + j] = lane[32 * w + j] + lane[32 * w + j + o];
    float t = lane[0];
    for (int w = 1; w < 8; ++w) t = t + lane[32 * w];
    return t;
}

void orc_layernorm_stats(const uint16_t* row, int32_t H, float eps, float* mean_out, float* rstd_out) {
    float s[256], q[256];
    for (int l = 0; l < 256; ++l) s[l] = q[l] = 0.0f;
    for (int32_t v = 0; v < H / 16; ++v) {
        int l = v % 256;
        for (int e = 0; e < 16; ++e) {
            float x = orc_bf16_to_f32(row[16 * v + e]);
            s[l] = s[l] + x;
            q[l] = fmaf(x, x, q[l]);
        }
    }
    float S = row_sum_fixed_order(s), Q = row_sum_fixed_order(q);
    float mean = S / (float)H;
    float m2 = Q / (float)H;
    float var = m2 - mean * mean;
    if (!(var > 0.0f)) var = 0.0f;
    *mean_out = mean;
    *rstd_out = 1.0f / sqrtf(var + eps);
}

/* y = bf16(LayerNorm(x) * gamma + beta) row by row; q = FP8(y / scale);
 * amax = max(amax, |y|).  gamma and beta are float[H]; y may be NULL. */
void orc_layernorm_quantize_amax(const uint16_t* x_bf16, int64_t rows, int32_t H, const float* gamma,
                                 const float* beta, float eps, int fmt, float scale, uint8_t* q,
                                 uint16_t* y_bf16, float* amax_inout) {
    float m = *amax_inout;
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* row = x_bf16 + r * H;
        float mean, rstd;
        orc_layernorm_stats(row, H, eps, &mean, &rstd);
        for (int32_t i = 0; i < H; ++i) {
            float x = orc_bf16_to_f32(row[i]);
            float mul = rstd * gamma[i];
            float yf = (x - mean) * mul + beta[i];
            uint16_t yb = orc_f32_to_bf16(yf);
            float y = orc_bf16_to_f32(yb);
            if (y_bf16) y_bf16[r * H + i] = yb;
            q[r * H + i] = orc_fp8_encode(y / scale, fmt);
            m = amax_combine(m, fabsf(y));
        }
    }
    if (rows > 0 && H > 0) *amax_inout = m;
}

/* ----------------------------------------------------------------------- */
/* amax_and_scale_update ([TE-593]; scale formula from [XLA-FP8] "JAX":     */
/* scale = max|A| / E4M3_MAX, times 2^margin).                              */

/* Scale and scale_inv of one slot from its selected amax, or pass-through. */
static void slot_scale(float a, int f, int32_t margin, float* scale, float* scale_inv) {
    if (f != ORC_E4M3FN && f != ORC_E5M2) return; /* unknown format: leave the slot */
    if (!(isfinite(a) && a > 0.0f)) return;
    float fp8max = (float)orc_fp8_max(f);
    float sc = a / fp8max;      /* RN binary32 */
    sc = ldexpf(sc, margin);    /* times 2^margin, one rounding */
    if (!isnormal(sc)) return;
    *scale = sc;
    *scale_inv = 1.0f / sc;     /* RN binary32 */
}

void orc_amax_scale_update(float* hist, int32_t H, int32_t S, const float* amax_new,
                           float* scale, float* scale_inv, const uint8_t* slot_format,
                           int fmt, int algo, int32_t margin) {
    for (int32_t s = 0; s < S; ++s) {
        /* 1. roll: every entry one step older, the oldest dropped */
        for (int32_t h = H - 1; h >= 1; --h) hist[(int64_t)h * S + s] = hist[(int64_t)(h - 1) * S + s];
        hist[s] = amax_new[s];

        /* 2. select */
        float a = hist[s];
        if (algo == ORC_ALGO_MAX)
            for (int32_t h = 1; h < H; ++h) a = amax_combine(a, hist[(int64_t)h * S + s]);

        /* 3. scale and its inverse, or pass-through */
        slot_scale(a, slot_format ? slot_format[s] : fmt, margin, &scale[s], &scale_inv[s]);
    }
}

/*
 * The same update over a ring buffer (a NEXT item beyond the roll: the window
 * is kept in place and only the oldest entry is overwritten).  Slot s keeps
 * its own position head[s] = the physical row of its newest entry; logical
 * row r (0 = newest) is physical row (head[s] - r) mod H, so after the same
 * sequence of calls the window holds exactly what the rolled history holds.
 * A head outside [0, H) leaves the whole slot unchanged.
 */
void orc_amax_scale_update_ring(float* hist, int32_t* head, int32_t H, int32_t S,
                                const float* amax_new, float* scale, float* scale_inv,
                                const uint8_t* slot_format, int fmt, int algo, int32_t margin) {
    for (int32_t s = 0; s < S; ++s) {
        int32_t h = head[s];
        if (h < 0 || h >= H) continue;
        h = (h + 1) % H;                   /* the oldest entry's row */
        hist[(int64_t)h * S + s] = amax_new[s];
        head[s] = h;
        float a = hist[(int64_t)h * S + s];
        if (algo == ORC_ALGO_MAX)
            for (int32_t r = 0; r < H; ++r) a = amax_combine(a, hist[(int64_t)r * S + s]);
        slot_scale(a, slot_format ? slot_format[s] : fmt, margin, &scale[s], &scale_inv[s]);
    }
}
