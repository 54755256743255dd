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
/* The producers fused with the quantization ([XLA-7432], test.py: the      */
/* transformer block applies nn.LayerNorm() to its input, and the MLP       */
/* applies nn.gelu to the first dense layer's output; each result feeds an  */
/* FP8 dense layer, and the issue asks for the quantization to be fused     */
/* with what produces its input).                                           */
/*                                                                          */
/* The producers are defined here by their plain formulas in float64.  The  */
/* fused operation's output is y = bf16(producer(x)); a binary32            */
/* implementation reaches the float64 value only up to its own rounding,    */
/* so y is accepted within a tolerance derived from that arithmetic (the    */
/* Python side of this oracle states it).  The FP8 codes and the amax are   */
/* then exactly orc_quantize_amax of that y.                                */

/* Nearest bf16 to a float64 value, ties to the even bf16, in ONE rounding  */
/* (rounding to binary32 first could round twice).  The two bf16 neighbours */
/* of |g| are multiples of the bf16 spacing at |g| (2^(e-7) for |g| in      */
/* [2^e, 2^(e+1)), 2^-133 below 2^-126), so they and their midpoint are     */
/* exact in double.  At or beyond the midpoint between the largest finite   */
/* bf16 and 2^128 the result is infinity.                                    */
uint16_t orc_f64_to_bf16(double g) {
    if (isnan(g)) return 0x7FC0;
    uint16_t sign = signbit(g) ? 0x8000 : 0x0000;
    double a = fabs(g);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int e;
    (void)frexp(a, &e);                          /* a in [2^(e-1), 2^e) */
    int q = (e - 1 >= -126) ? (e - 1) - 7 : -133; /* exponent of the spacing */
    double ulp = ldexp(1.0, q);
    double m = floor(a / ulp);                   /* a / ulp is exact: a power-of-two scaling */
    double lo = m * ulp, hi = lo + ulp, mid = lo + 0.5 * ulp;
    double pick;
    if (a < mid) pick = lo;
    else if (a > mid) pick = hi;
    else pick = (fmod(m, 2.0) == 0.0) ? lo : hi; /* the even last mantissa bit */
    if (pick >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    return (uint16_t)(sign | (f32_to_bits((float)pick) >> 16)); /* exact: pick is a bf16 value */
}

/* orc_f64_to_bf16 over an array. */
void orc_f64_to_bf16_array(const double* g, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16(g[i]);
}

/* GELU, tanh form (Flax's nn.gelu, approximate=True):                      */
/*   GELU(x) = 0.5 x (1 + tanh(u)),  u = sqrt(2/pi) (x + 0.044715 x^3).      */
/* Since 1 + tanh(u) = 2 / (1 + e^(-2u)), this is x / (1 + e^(-2u)), which   */
/* float64 evaluates without the cancellation that 1 + tanh(u) suffers for */
/* u << 0 (there the result is tiny but still far inside bf16's range).     */
/* At +-inf the value is the limit: +inf and -0.                            */
double orc_gelu_ref(double x) {
    if (isnan(x)) return x;
    if (isinf(x)) return x > 0 ? x : -0.0;
    const double k = sqrt(2.0 / acos(-1.0));
    const double u = k * (x + 0.044715 * x * x * x);
    return x / (1.0 + exp(-2.0 * u));
}

/* GELU(h) in float64 for n bf16 inputs. */
void orc_gelu_ref_array(const uint16_t* h_bf16, int64_t n, double* g) {
    for (int64_t i = 0; i < n; ++i) g[i] = orc_gelu_ref((double)orc_bf16_to_f32(h_bf16[i]));
}

/* LayerNorm with Flax's defaults (nn.LayerNorm(): statistics over the last  */
/* axis, epsilon 1e-6 unless given, learned scale gamma and bias beta),     */
/* row by row in float64:                                                   */
/*   mean = (1/H) sum x,   var = max(0, (1/H) sum x^2 - mean^2),            */
/*   y = (x - mean) * (gamma / sqrt(var + eps)) + beta.                     */
/* The sums run left to right.  mean_out and rstd_out (1/sqrt(var + eps))   */
/* may be NULL.  A NaN or infinite input makes the row's y NaN.             */
void orc_layernorm_ref(const uint16_t* x_bf16, int64_t rows, int32_t H, const float* gamma,
                       const float* beta, double eps, double* y, double* mean_out, double* rstd_out) {
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* row = x_bf16 + r * H;
        double s = 0.0, s2 = 0.0;
        for (int32_t i = 0; i < H; ++i) {
            double v = (double)orc_bf16_to_f32(row[i]);
            s += v;
            s2 += v * v;
        }
        double mean = s / H;
        double var = s2 / H - mean * mean;
        if (var < 0.0) var = 0.0;                  /* a NaN stays NaN */
        double rstd = 1.0 / sqrt(var + eps);
        for (int32_t i = 0; i < H; ++i) {
            double v = (double)orc_bf16_to_f32(row[i]);
            y[r * H + i] = (v - mean) * (rstd * (double)gamma[i]) + (double)beta[i];
        }
        if (mean_out) mean_out[r] = mean;
        if (rstd_out) rstd_out[r] = rstd;
    }
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
