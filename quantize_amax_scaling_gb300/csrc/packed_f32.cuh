// packed_f32.cuh -- two-lane binary32 arithmetic (PTX f32x2, sm_100 and later)
// and a correctly rounded two-lane reciprocal, for the producer kernels.
//
// Every two-lane operation rounds each lane exactly like its scalar form.

#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace {

// Two-lane binary32 add and multiply (PTX f32x2, sm_100 and later), each lane
// rounded to nearest even exactly like add.rn.f32 / mul.rn.f32.  A two-lane
// multiply whose result feeds a two-lane add was measured to come out as one
// fused multiply-add (a single rounding) on sm_103a even with the explicit
// rounding mode (and so did a two-lane fma with a -0 addend followed by a
// two-lane add), so a product that is then added is formed with the scalar
// __fmul_rn / __fadd_rn pair, which is never contracted.
__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// RN(1/d) for d in [1, 2^126), where 1/d is a normal number: the hardware
// approximation y0 refined by one correction step, r = 1 - d*y0 and
// y = y0 + y0*r, each a fused multiply-add (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990).  tests/csrc/reciprocal_check.cu compares it bit for bit
// with the IEEE reciprocal for every binary32 d in [1, 2^126).  Larger d
// (1/d subnormal or zero, and +inf) take the IEEE reciprocal instead.
__device__ __forceinline__ float rcp_approx_ftz(float d) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(d));
    return y;
}

__device__ __forceinline__ float2 rcp2_rn(float2 d) {
    if (fmaxf(d.x, d.y) >= 0x1p126f) return make_float2(__frcp_rn(d.x), __frcp_rn(d.y));
    const float2 y0 = make_float2(rcp_approx_ftz(d.x), rcp_approx_ftz(d.y));
    const float2 r = fma2_rn(mul2_rn(d, splat2(-1.0f)), y0, splat2(1.0f));
    return fma2_rn(y0, r, y0);
}

}  // namespace
