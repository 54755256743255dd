// reciprocal_check.cu -- rcp2_rn (the producers' two-lane reciprocal) against
// CUDA's IEEE reciprocal __frcp_rn, bit for bit, for every binary32 d in
// [1, 2^128) and for +inf.  Lane 0 walks binade k and lane 1 binade 127 - k
// with a scrambled significand, so every call mixes two different values (and
// pairs that take the fallback with pairs that do not).  Prints one line per
// binade with a mismatch count, then the total; exits 1 on any mismatch or
// CUDA error.
#include <cstdint>
#include <cstdio>

#include <cuda_runtime.h>

#include "packed_f32.cuh"

__global__ void check(unsigned long long* bad) {
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;  // significand
    if (i >= (1u << 23)) return;
    const uint32_t j = (i * 2654435761u) & 0x7FFFFFu;          // a permutation of the significands
    for (int k = 0; k < 128; ++k) {
        const float d0 = __uint_as_float(((uint32_t)(k + 127) << 23) | i);
        const float d1 = __uint_as_float(((uint32_t)(127 - k + 127) << 23) | j);
        const float2 y = rcp2_rn(make_float2(d0, d1));
        if (__float_as_uint(y.x) != __float_as_uint(__frcp_rn(d0))) atomicAdd(&bad[k], 1ull);
        if (__float_as_uint(y.y) != __float_as_uint(__frcp_rn(d1))) atomicAdd(&bad[127 - k], 1ull);
    }
    if (i == 0) {  // +inf in either lane
        const float2 y = rcp2_rn(make_float2(__int_as_float(0x7F800000), 3.0f));
        if (__float_as_uint(y.x) != 0u || __float_as_uint(y.y) != __float_as_uint(__frcp_rn(3.0f)))
            atomicAdd(&bad[128], 1ull);
    }
}

int main() {
    unsigned long long* bad = nullptr;
    if (cudaMalloc(&bad, 129 * sizeof(unsigned long long)) != cudaSuccess) return 1;
    cudaMemset(bad, 0, 129 * sizeof(unsigned long long));
    check<<<(1u << 23) / 256, 256>>>(bad);
    cudaError_t err = cudaDeviceSynchronize();
    if (err != cudaSuccess) {
        std::printf("CUDA error: %s\n", cudaGetErrorString(err));
        return 1;
    }
    unsigned long long h[129];
    cudaMemcpy(h, bad, sizeof h, cudaMemcpyDeviceToHost);
    cudaFree(bad);
    unsigned long long total = 0;
    for (int k = 0; k < 129; ++k) {
        if (h[k]) std::printf("%s %d: %llu mismatches\n", k < 128 ? "binade" : "inf case", k, h[k]);
        total += h[k];
    }
    std::printf("checked %llu values, mismatches: %llu\n", 2ull * 128ull * (1ull << 23) + 2ull, total);
    return total == 0 ? 0 : 1;
}
