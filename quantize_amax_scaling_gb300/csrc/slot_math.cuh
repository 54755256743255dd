// slot_math.cuh -- per-slot arithmetic of the scale update, shared by the
// update kernels and by the update fused with a quantize (whose quantizing
// CTAs recompute one slot's new scale and must get the same bits).

#pragma once

#include "fp8q_common.cuh"

namespace {

// Order-preserving integer key of a non-NaN float (so an integer max is a
// float max); NaN is tracked separately.
__device__ __forceinline__ int float_key(float f) {
    const int b = __float_as_int(f);
    return b ^ ((b >> 31) & 0x7FFFFFFF);
}

__device__ __forceinline__ float key_float(int k) { return __int_as_float(k ^ ((k >> 31) & 0x7FFFFFFF)); }

// The new scale of a slot from its selected amax: RN(amax / FP8_MAX) * 2^margin
// for a known format, a finite amax > 0 and a normal, finite result; false
// (the slot keeps its scale and scale_inv) otherwise.
__device__ __forceinline__ bool new_slot_scale(float amax, int f, int margin, float* sc) {
    if ((f == FP8Q_E4M3FN || f == FP8Q_E5M2) && isfinite(amax) && amax > 0.0f) {
        const float fp8max = (f == FP8Q_E4M3FN) ? 448.0f : 57344.0f;
        const float pow2m = __uint_as_float((uint32_t)(127 + margin) << 23);  // exact 2^margin
        const float s = __fmul_rn(__fdiv_rn(amax, fp8max), pow2m);
        if (s >= 0x1p-126f && s <= 0x1.fffffep127f) {  // normal and finite
            *sc = s;
            return true;
        }
    }
    return false;
}

// Scale and scale_inv of one slot from its selected amax, or pass-through.
__device__ __forceinline__ void slot_scale(float amax, int f, int margin, float* scale, float* scale_inv) {
    float sc;
    if (new_slot_scale(amax, f, margin, &sc)) {
        *scale = sc;
        *scale_inv = __frcp_rn(sc);
    }
}

}  // namespace
