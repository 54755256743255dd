/*
 * Exhaustive check of the quantize kernel's division method against IEEE
 * binary32 division, on the host (C99 fmaf is a correctly rounded fused
 * multiply-add; -ffp-contract=off keeps every other operation separate).
 *
 * Method (Markstein's correction step, P. Markstein, IBM J. Res. Dev. 34(1),
 * 1990): r = RN(1/s); y0 = RN(x*r); e = fma(y0, s, -x); y = fma(-e, r, y0).
 *
 * Part 1: every bf16 significand (x in [1,2), 128 values) against every
 * binary32 significand of s (s in [1,2), 2^23 values) -- y must equal x/s
 * bit for bit.  While no intermediate leaves the normal range, scaling x and
 * s by powers of two scales every step exactly, so this covers the band the
 * kernel uses the method in.
 * Part 2: the band edges -- random bf16 x (all exponents, both signs, zeros,
 * subnormals) with random s in [2^-60, 2^60]: wherever |x/s| is in
 * [2^-18, 2^17] the result must equal x/s; below it, |y| <= 2^-17 with the
 * sign of x; above it (after the clamp to RU_bf16(s*2^17)), y >= 2^17.
 * Prints "mismatches <n>" and exits 0 only when n == 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float f32(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
static uint32_t b32(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }

static float method(float x, float s, float r) {
    float y0 = x * r;
    float e = fmaf(y0, s, -x);
    return fmaf(-e, r, y0);
}

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static uint64_t next_u64(void) { /* splitmix64 */
    uint64_t z = (rng_state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

int main(void) {
    long bad = 0;
#pragma omp parallel for reduction(+ : bad) schedule(static)
    for (int32_t ms = 0; ms < (1 << 23); ++ms) {
        float s = f32(0x3F800000u | (uint32_t)ms);
        float r = 1.0f / s;
        for (uint32_t mx = 0; mx < 128; ++mx) {
            float x = f32(0x3F800000u | (mx << 16));
            if (b32(method(x, s, r)) != b32(x / s)) bad++;
        }
    }
    long bad2 = 0;
    for (int i = 0; i < 20000000; ++i) {
        uint64_t u = next_u64();
        float x = f32((uint32_t)(u & 0xFFFF) << 16);
        if (isnan(x) || isinf(x)) continue;
        float s = ldexpf(1.0f + (float)((u >> 16) & 0x7FFFFF) * 0x1p-23f, (int)((u >> 40) % 121) - 60);
        float r = 1.0f / s;
        float t = f32((b32(s * 131072.0f) + 0xFFFFu) & 0xFFFF0000u); /* RU_bf16(s * 2^17) */
        float xc = fabsf(x) > t ? copysignf(t, x) : x;
        float y = method(xc, s, r);
        float q = x / s;
        float aq = fabsf(q);
        if (aq >= 0x1p-18f && aq <= 0x1p17f) {
            if (b32(y) != b32(q)) bad2++;
        } else if (aq < 0x1p-18f) {
            if (!(fabsf(y) <= 0x1p-17f) || signbit(y) != signbit(x)) bad2++;
        } else {
            if (!(fabsf(y) >= 0x1p17f) || signbit(y) != signbit(x)) bad2++;
        }
    }
    printf("mismatches %ld (significand sweep) %ld (band edges)\n", bad, bad2);
    return (bad == 0 && bad2 == 0) ? 0 : 1;
}
