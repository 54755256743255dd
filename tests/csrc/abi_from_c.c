/*
 * Calls libfp8q through its C header only (no Python, no torch).
 *   ./abi_from_c args  -- argument checking, no GPU needed
 *   ./abi_from_c gpu   -- quantize / dequantize / scale update on device
 *                         buffers; expected values are hand-derived from the
 *                         FP8 and bf16 definitions (see tests/golden)
 * Prints "OK" and exits 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "fp8q.h"

#ifdef WITH_CUDA
#include <cuda_runtime.h>
#endif

static int fails = 0;
#define CHECK(c) do { if (!(c)) { printf("FAIL line %d: %s\n", __LINE__, #c); ++fails; } } while (0)

static int args_mode(void) {
    void* p = (void*)0x10000;
    CHECK(fp8q_quantize_amax(NULL, NULL, 0, FP8Q_E4M3FN, NULL, NULL, NULL) == FP8Q_OK);
    CHECK(fp8q_quantize_amax(p, p, -1, FP8Q_E4M3FN, p, p, NULL) == FP8Q_ERR_INVALID_ARG);
    CHECK(fp8q_quantize_amax(p, p, 4, (fp8q_format)9, p, p, NULL) == FP8Q_ERR_INVALID_ARG);
    CHECK(fp8q_dequantize(NULL, p, 4, FP8Q_E5M2, p, NULL) == FP8Q_ERR_INVALID_ARG);
    CHECK(fp8q_multi_quantize_amax(NULL, FP8Q_MAX_TENSORS + 1, FP8Q_E4M3FN, NULL) == FP8Q_ERR_TOO_MANY_TENSORS);
    CHECK(fp8q_amax_scale_update(p, 0, 4, p, p, p, NULL, FP8Q_E4M3FN, FP8Q_ALGO_MAX, 0, NULL) ==
          FP8Q_ERR_INVALID_ARG);
    CHECK(fp8q_amax_scale_update_ring(p, p, 4, 4, p, p, p, NULL, FP8Q_E4M3FN, FP8Q_ALGO_MAX, 65, NULL) ==
          FP8Q_ERR_INVALID_ARG);
    CHECK(fp8q_qdq_amax(p, (char*)p + 1, 4, FP8Q_E4M3FN, p, p, NULL) == FP8Q_ERR_INVALID_ARG);
    CHECK(fp8q_gelu_quantize_amax(p, NULL, NULL, 4, FP8Q_E4M3FN, p, p, NULL) == FP8Q_ERR_INVALID_ARG);
    CHECK(strcmp(fp8q_status_string(FP8Q_ERR_CUDA), "FP8Q_ERR_CUDA") == 0);
    CHECK(strcmp(fp8q_last_cuda_error(), "") == 0);
    return fails;
}

#ifdef WITH_CUDA
static int gpu_mode(void) {
    /* bf16 inputs and their e4m3fn codes at scale 1 (round to nearest, ties to even, saturating) */
    const uint16_t x[8] = {0x3F80 /* 1 */, 0xBF88 /* -1.0625: tie -> even */, 0x43E0 /* 448 */,
                           0x4600 /* 8192: saturates */, 0x3A80 /* 2^-10: tie -> 0 */,
                           0x3B40 /* 3*2^-10: tie -> 2^-8 */, 0x0000, 0x8000};
    const uint8_t want_q[8] = {0x38, 0xB8, 0x7E, 0x7E, 0x00, 0x02, 0x00, 0x80};
    /* dequantized at scale 2: 2, -2, 896, 896, 0, 2^-7, 0, -0 */
    const uint16_t want_y[8] = {0x4000, 0xC000, 0x4460, 0x4460, 0x0000, 0x3C00, 0x0000, 0x8000};
    void *dx, *dq, *dy, *ds, *da, *dh, *dn, *dsc, *dsi;
    CHECK(cudaMalloc(&dx, 16) == cudaSuccess);
    CHECK(cudaMalloc(&dq, 8) == cudaSuccess);
    CHECK(cudaMalloc(&dy, 16) == cudaSuccess);
    CHECK(cudaMalloc(&ds, 8) == cudaSuccess);   /* [0] = 1, [1] = 2 */
    CHECK(cudaMalloc(&da, 4) == cudaSuccess);
    CHECK(cudaMalloc(&dh, 4 * 2 * 4) == cudaSuccess);
    CHECK(cudaMalloc(&dn, 2 * 4) == cudaSuccess);
    CHECK(cudaMalloc(&dsc, 2 * 4) == cudaSuccess);
    CHECK(cudaMalloc(&dsi, 2 * 4) == cudaSuccess);
    if (fails) return fails;
    const float scales[2] = {1.0f, 2.0f}, zero = 0.0f;
    cudaMemcpy(dx, x, 16, cudaMemcpyHostToDevice);
    cudaMemcpy(ds, scales, 8, cudaMemcpyHostToDevice);
    cudaMemcpy(da, &zero, 4, cudaMemcpyHostToDevice);
    CHECK(fp8q_quantize_amax(dx, (uint8_t*)dq, 8, FP8Q_E4M3FN, (const float*)ds, (float*)da, NULL) == FP8Q_OK);
    CHECK(fp8q_dequantize((const uint8_t*)dq, dy, 8, FP8Q_E4M3FN, (const float*)ds + 1, NULL) == FP8Q_OK);
    /* one update from a zero history of 4: slot 0 sees amax 896 -> scale 2; slot 1 sees 0 -> unchanged */
    float hist[8] = {0}, news[2] = {896.0f, 0.0f}, ones[2] = {1.0f, 1.0f};
    cudaMemcpy(dh, hist, sizeof hist, cudaMemcpyHostToDevice);
    cudaMemcpy(dn, news, sizeof news, cudaMemcpyHostToDevice);
    cudaMemcpy(dsc, ones, sizeof ones, cudaMemcpyHostToDevice);
    cudaMemcpy(dsi, ones, sizeof ones, cudaMemcpyHostToDevice);
    CHECK(fp8q_amax_scale_update((float*)dh, 4, 2, (const float*)dn, (float*)dsc, (float*)dsi, NULL,
                                 FP8Q_E4M3FN, FP8Q_ALGO_MAX, 0, NULL) == FP8Q_OK);
    CHECK(cudaDeviceSynchronize() == cudaSuccess);
    uint8_t q[8];
    uint16_t y[8];
    float amax, sc[2], si[2], h[8];
    cudaMemcpy(q, dq, 8, cudaMemcpyDeviceToHost);
    cudaMemcpy(y, dy, 16, cudaMemcpyDeviceToHost);
    cudaMemcpy(&amax, da, 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(sc, dsc, 8, cudaMemcpyDeviceToHost);
    cudaMemcpy(si, dsi, 8, cudaMemcpyDeviceToHost);
    cudaMemcpy(h, dh, sizeof h, cudaMemcpyDeviceToHost);
    for (int i = 0; i < 8; ++i) {
        if (q[i] != want_q[i]) { printf("q[%d] = 0x%02x, want 0x%02x\n", i, q[i], want_q[i]); ++fails; }
        if (y[i] != want_y[i]) { printf("y[%d] = 0x%04x, want 0x%04x\n", i, y[i], want_y[i]); ++fails; }
    }
    CHECK(amax == 8192.0f);
    CHECK(sc[0] == 2.0f && si[0] == 0.5f && sc[1] == 1.0f && si[1] == 1.0f);
    CHECK(h[0] == 896.0f && h[1] == 0.0f && h[2] == 0.0f);
    cudaFree(dx); cudaFree(dq); cudaFree(dy); cudaFree(ds); cudaFree(da);
    cudaFree(dh); cudaFree(dn); cudaFree(dsc); cudaFree(dsi);
    return fails;
}
#endif

int main(int argc, char** argv) {
    int r = 1;
    if (argc > 1 && strcmp(argv[1], "args") == 0) r = args_mode();
#ifdef WITH_CUDA
    else if (argc > 1 && strcmp(argv[1], "gpu") == 0) r = gpu_mode();
#endif
    puts(r == 0 ? "OK" : "FAILED");
    return r == 0 ? 0 : 1;
}
