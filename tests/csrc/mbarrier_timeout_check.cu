// mbarrier_timeout_check.cu -- the bounded mbarrier wait the LayerNorm producer
// uses (mbarrier.cuh), on the GPU, without any fault: a bulk copy that arrives
// completes its wait, and a wait on an mbarrier that nothing ever completes
// gives up after about one second and reports it, so the kernel can return.
// Prints the outcome; exits 1 if either case misbehaves or CUDA reports an
// error.
#include <cstdint>
#include <cstdio>

#include <cuda_runtime.h>

#include "mbarrier.cuh"

constexpr int kN = 1024;

__global__ void waits(const float* src, float* dst, unsigned long long* out) {
    __shared__ __align__(128) float buf[kN];
    __shared__ uint64_t bar[2];
    if (threadIdx.x == 0) {
        mbar_init(&bar[0]);
        mbar_init(&bar[1]);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) bulk_load(buf, src, sizeof buf, &bar[0]);
    const bool got = mbar_wait(&bar[0], 0);  // the copy arrives
    if (got)
        for (int i = threadIdx.x; i < kN; i += blockDim.x) dst[i] = 2.0f * buf[i];
    const uint64_t t0 = global_ns();
    const bool none = mbar_wait(&bar[1], 0);  // nothing ever arrives on bar[1]
    const uint64_t t1 = global_ns();
    if (threadIdx.x == 0) {
        out[0] = got;
        out[1] = none;
        out[2] = t1 - t0;
    }
}

int main() {
    float h[kN], r[kN];
    for (int i = 0; i < kN; ++i) h[i] = (float)i - 100.0f;
    float *src = nullptr, *dst = nullptr;
    unsigned long long* out = nullptr;
    if (cudaMalloc(&src, sizeof h) != cudaSuccess || cudaMalloc(&dst, sizeof h) != cudaSuccess ||
        cudaMalloc(&out, 3 * sizeof(unsigned long long)) != cudaSuccess)
        return 1;
    cudaMemcpy(src, h, sizeof h, cudaMemcpyHostToDevice);
    cudaMemset(dst, 0, sizeof h);
    waits<<<1, 256>>>(src, dst, out);
    const cudaError_t err = cudaDeviceSynchronize();
    if (err != cudaSuccess) {
        std::printf("CUDA error: %s\n", cudaGetErrorString(err));
        return 1;
    }
    unsigned long long o[3];
    cudaMemcpy(o, out, sizeof o, cudaMemcpyDeviceToHost);
    cudaMemcpy(r, dst, sizeof r, cudaMemcpyDeviceToHost);
    int bad = 0;
    for (int i = 0; i < kN; ++i) bad += r[i] != 2.0f * h[i];
    std::printf("arrived wait: %llu, data mismatches: %d; empty wait: %llu after %.3f s\n", o[0], bad, o[1],
                o[2] * 1e-9);
    cudaFree(src);
    cudaFree(dst);
    cudaFree(out);
    const bool ok = o[0] == 1 && bad == 0 && o[1] == 0 && o[2] >= 1000000000ull && o[2] < 3000000000ull;
    std::printf("%s\n", ok ? "OK" : "FAILED");
    return ok ? 0 : 1;
}
