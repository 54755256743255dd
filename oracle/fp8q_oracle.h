/*
 * fp8q_oracle.h -- TEST INFRASTRUCTURE ONLY: the CPU oracle's own interface.
 * Shared with nothing on the CUDA path.  Arrays are host memory owned by the
 * caller; bf16 values are passed as their 16-bit patterns.
 */
#ifndef FP8Q_ORACLE_H
#define FP8Q_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_E4M3FN = 0, ORC_E5M2 = 1 };
enum { ORC_ALGO_MAX = 0, ORC_ALGO_MOST_RECENT = 1 };

typedef struct {
    const uint16_t* x_bf16;
    uint8_t* q;
    int64_t n;
    float scale;
    float* amax;
} orc_tensor;

float orc_bf16_to_f32(uint16_t h);
uint16_t orc_f32_to_bf16(float f);

int orc_fp8_max_code(int fmt);
double orc_fp8_decode(uint8_t code, int fmt);
double orc_fp8_max(int fmt);
uint8_t orc_fp8_encode(float y, int fmt);

void orc_quantize_amax(const uint16_t* x_bf16, int64_t n, int fmt, float scale, uint8_t* q,
                       float* amax_inout);
void orc_multi_quantize_amax(const orc_tensor* list, int32_t count, int fmt);
float orc_amax(const uint16_t* x_bf16, int64_t n);
void orc_dequantize(const uint8_t* q, int64_t n, int fmt, float scale, uint16_t* y_bf16);
void orc_qdq_amax(const uint16_t* x_bf16, int64_t n, int fmt, float scale, uint16_t* y_bf16,
                  float* amax_inout);
uint16_t orc_f64_to_bf16(double g);
void orc_f64_to_bf16_array(const double* g, int64_t n, uint16_t* out);
double orc_gelu_ref(double x);
void orc_gelu_ref_array(const uint16_t* h_bf16, int64_t n, double* g);
void orc_layernorm_ref(const uint16_t* x_bf16, int64_t rows, int32_t H, const float* gamma,
                       const float* beta, double eps, double* y, double* mean_out, double* rstd_out);
void orc_amax_scale_update(float* hist, int32_t H, int32_t S, const float* amax_new,
                           float* scale, float* scale_inv, const uint8_t* slot_format,
                           int fmt, int algo, int32_t margin);
void orc_amax_scale_update_ring(float* hist, int32_t* head, int32_t H, int32_t S,
                                const float* amax_new, float* scale, float* scale_inv,
                                const uint8_t* slot_format, int fmt, int algo, int32_t margin);

#ifdef __cplusplus
}
#endif

#endif
