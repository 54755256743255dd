/*
 * gelu_sequence.c -- TEST INFRASTRUCTURE: a determinism check, not the oracle.
 *
 * The library's GELU producer evaluates the tanh-form GELU by one fixed
 * sequence of correctly rounded binary32 operations, so that its direct
 * kernel and its table kernel (which tabulates the same arithmetic for every
 * bf16 input) give the same bits on every GB300.  This file restates that
 * sequence on the CPU so that a test can confirm the bits are reproducible.
 * Parity with the definition is a separate matter: the oracle defines GELU in
 * float64 and the tests accept the kernel's bf16 result within a tolerance
 * derived from this arithmetic.
 *
 * The sequence: s = x (1 + 0.044715 x^2), v = -2 sqrt(2/pi) s, clamped to
 * [-20, 89]; e^v by additive range reduction (W. J. Cody and W. Waite,
 * "Software Manual for the Elementary Functions", 1980): k = round(v / ln 2)
 * from one fused multiply-add with 1.5 * 2^23, r = v - k ln 2 with ln 2 split
 * in two (high part to 16 significant bits, so k * LN2_HI is exact), a
 * degree-6 Taylor polynomial of e^r (Horner, fused), and (p * 2^(k-1)) * 2;
 * then 1 / (1 + e^v), times x.  GELU(-inf) = -0.  Build with
 * -ffp-contract=off so that every line is the operation it shows.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static const float LN2_HI = 0x1.62e4p-1f;
static const float LN2_LO = 0x1.7f7d1cp-20f;
static const float INV_LN2 = 0x1.715476p+0f;
static const float ROUNDER = 0x1.8p23f;
static const float NEG_2_SQRT_2_OVER_PI = -0x1.988454p+0f;
static const float C3 = 0x1.6e4e26p-5f; /* 0.044715 */

float seq_exp_f32(float v) {
    if (v > 89.0f) v = 89.0f;
    if (!(v >= -20.0f)) v = -20.0f;
    float t = fmaf(v, INV_LN2, ROUNDER);
    float k = t - ROUNDER;
    float r = fmaf(-k, LN2_HI, v);
    r = fmaf(-k, LN2_LO, r);
    float p = 0x1.6c16c2p-10f;      /* 1/720 */
    p = fmaf(p, r, 0x1.111112p-7f); /* 1/120 */
    p = fmaf(p, r, 0x1.555556p-5f); /* 1/24 */
    p = fmaf(p, r, 0x1.555556p-3f); /* 1/6 */
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    return (p * ldexpf(1.0f, (int)k - 1)) * 2.0f;
}

float seq_gelu_f32(float x) {
    if (x == -INFINITY) return -0.0f;
    float x2 = x * x;
    float s = x * fmaf(C3, x2, 1.0f);
    float d = 1.0f + seq_exp_f32(NEG_2_SQRT_2_OVER_PI * s);
    return x * (1.0f / d);
}

/* bf16 bits of RN_bf16(seq_gelu_f32(h)) for n bf16 inputs. */
void seq_gelu_bf16(const uint16_t* h, int64_t n, uint16_t* y) {
    for (int64_t i = 0; i < n; ++i) {
        uint32_t b = (uint32_t)h[i] << 16;
        float x;
        memcpy(&x, &b, 4);
        float g = seq_gelu_f32(x);
        uint32_t gb;
        memcpy(&gb, &g, 4);
        if (isnan(g)) {
            y[i] = 0x7FC0;
            continue;
        }
        /* round to nearest bf16, ties to even (binary32 -> bf16) */
        uint32_t lsb = (gb >> 16) & 1u;
        y[i] = (uint16_t)((gb + 0x7FFFu + lsb) >> 16);
    }
}
