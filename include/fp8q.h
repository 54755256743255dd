/*
 * fp8q.h -- C ABI of libfp8q: FP8 delayed-scaling quantization on one GPU.
 *
 * Nine operations, each one kernel launch on the caller's stream:
 *   fp8q_quantize_amax        bf16 -> FP8 bytes, fused with amax = max|x|
 *   fp8q_multi_quantize_amax  the same over a ragged list of tensors
 *   fp8q_dequantize           FP8 bytes -> bf16
 *   fp8q_amax_scale_update    amax-history roll + amax selection + scale and
 *                             scale_inv, for many FP8 metadata slots at once
 *   fp8q_qdq_amax             quantize then dequantize (bf16 -> bf16) + amax
 *   fp8q_amax_scale_update_ring  the update over a ring buffer (no roll)
 *   fp8q_gelu_quantize_amax   GELU producer fused with quantize + amax
 *   fp8q_layernorm_quantize_amax  LayerNorm producer fused with quantize + amax
 *   fp8q_amax_scale_update_ring_quantize  the ring update fused with the next
 *                             step's first quantize
 *
 * Sources (web pages, by title and section):
 *   "User Guide on Native XLA-FP8" (NVIDIA JAX-Toolbox): opening section
 *     (E4M3 / E5M2 formats, quantization Q and de-quantization DQ); section
 *     "JAX" (Q = cast(A / A_scale), DQ = cast(a_fp8) * a_scale, delayed
 *     scaling A_scale = max|A| / E4M3_MAX); section "Gradient accumulation of
 *     FP8 params" (FP8 meta accumulates with max, not add).
 *   "Fusion of Fp8 quantization and amax reduction kernels" (openxla/xla
 *     issue): quantization and the amax reduction are memory bound and
 *     belong in one pass over the tensor.
 *   "Implement fused kernel for FP8 scale update" (NVIDIA/TransformerEngine
 *     PR): amax_and_scale_update (history roll, amax selection, scale,
 *     scale_inv) as one in-place kernel in a framework-agnostic library,
 *     batched over all layers.
 *
 * Conventions shared by every call:
 *   - Data pointers are DEVICE memory of the calling thread's current CUDA
 *     device, owned by the caller.  The library allocates nothing, frees
 *     nothing and keeps no per-call state.  Inputs and outputs must not
 *     overlap unless a call says it works in place.
 *   - bf16 tensors are contiguous arrays of 16-bit patterns (any 2-byte
 *     aligned address); FP8 tensors are contiguous byte arrays.  Any
 *     alignment works; tensors whose bf16 and FP8 pointers are aligned alike
 *     (as allocators return them) take the vectorised path.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     return once the kernel is enqueued; results are ready when the stream
 *     reaches that point.
 *   - Errors are returned as fp8q_status, never raised or aborted.  Argument
 *     errors are detected before anything is launched.  FP8Q_ERR_CUDA means
 *     the launch itself failed; fp8q_last_cuda_error() (per thread) then
 *     describes it, and the error has been taken off the CUDA runtime's
 *     per-thread last error (cudaGetLastError) so that it is reported once.
 *     Each call checks only its own launch: a runtime error that an earlier,
 *     unrelated call left pending is neither reported nor cleared.
 *     A zero-sized call succeeds and launches nothing.
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8Q_E4M3FN = 0, /* 1-4-3, bias 7, no inf, max 448 (forward pass) */
    FP8Q_E5M2 = 1    /* 1-5-2, bias 15, IEEE inf/NaN, max 57344 (gradients) */
} fp8q_format;

typedef enum {
    FP8Q_ALGO_MAX = 0,        /* amax = max over the (rolled) history window */
    FP8Q_ALGO_MOST_RECENT = 1 /* amax = the newest entry */
} fp8q_amax_algo;

typedef enum {
    FP8Q_OK = 0,
    FP8Q_ERR_INVALID_ARG = 1,
    FP8Q_ERR_UNSUPPORTED = 2,
    FP8Q_ERR_CUDA = 3,
    FP8Q_ERR_TOO_MANY_TENSORS = 4
} fp8q_status;

/* Largest tensor count of one fp8q_multi_quantize_amax call (descriptors
 * travel inside the kernel's parameter block). */
#define FP8Q_MAX_TENSORS 512

/*
 * Fused quantize + amax of one bf16 tensor ("User Guide on Native XLA-FP8",
 * section "JAX", the quantization step; "Fusion of Fp8 quantization and amax
 * reduction kernels": amax fused into the same pass).
 *
 *   q[i]  = FP8(x[i] / *scale)   quotient in binary32, rounded to nearest even;
 *                                then rounded to the FP8 grid (nearest, ties
 *                                to even), saturating to +-448 / +-57344;
 *                                +-inf saturates; NaN gives a NaN code.
 *   *amax = max(*amax, max_i |x[i]|)   max-accumulated (not overwritten); a
 *                                NaN input makes it NaN; +-inf gives +inf.
 *
 * x_bf16: n bf16 values (device).  q: n bytes (device, written).
 * scale:  one float (device, read); any value, positive normal scales in
 *         [2^-60, 2^60] take the fast exact path.
 * amax:   one float (device, read-modify-write).  Start it at +0 (or any
 *         non-negative value) before the first tensor of a step.
 * Errors: INVALID_ARG for n < 0, an unknown fmt, a NULL pointer with n > 0
 *         or an odd x_bf16 address.
 */
fp8q_status fp8q_quantize_amax(const void* x_bf16, uint8_t* q, int64_t n, fp8q_format fmt,
                               const float* scale, float* amax, void* stream);

/* One tensor of a ragged list: its own size, scale and amax. */
typedef struct {
    const void* x_bf16; /* n bf16 values (device) */
    uint8_t* q;         /* n bytes (device, written) */
    int64_t n;          /* elements; 0 is allowed (pointers then unused) */
    const float* scale; /* one float (device) */
    float* amax;        /* one float (device), max-accumulated */
} fp8q_tensor;

/*
 * fp8q_quantize_amax over `count` tensors in ONE launch ("Fusion of Fp8
 * quantization and amax reduction kernels": weights and activations all need
 * Q + amax; "Implement fused kernel for FP8 scale update": batch the per-layer
 * work).  Each tensor gets exactly the result fp8q_quantize_amax would give.
 *
 * list:   `count` descriptors in HOST memory, read during the call only.
 * Errors: TOO_MANY_TENSORS for count > FP8Q_MAX_TENSORS; INVALID_ARG for
 *         count < 0, list == NULL with count > 0, or any descriptor that
 *         fp8q_quantize_amax would reject.  Two tensors may share an amax or
 *         a scale; outputs must not overlap.
 */
fp8q_status fp8q_multi_quantize_amax(const fp8q_tensor* list, int32_t count, fp8q_format fmt,
                                     void* stream);

/*
 * Dequantize ("User Guide on Native XLA-FP8", section "JAX": up-cast the FP8
 * value and multiply by the scale):
 *   y[i] = bf16_rne( float(q[i]) * *scale )   product in binary32 (RN), then
 *                                             rounded to nearest-even bf16;
 *                                             NaN codes give a NaN.
 * q: n bytes (device).  y_bf16: n bf16 (device, written).  scale: one float
 * (device).  Errors: INVALID_ARG for n < 0, unknown fmt, NULL with n > 0, odd
 * y_bf16 address.
 */
fp8q_status fp8q_dequantize(const uint8_t* q, void* y_bf16, int64_t n, fp8q_format fmt,
                            const float* scale, void* stream);

/*
 * amax_and_scale_update for `num_slots` FP8 metadata slots in ONE launch,
 * in place ("Implement fused kernel for FP8 scale update"; scale formula from
 * "User Guide on Native XLA-FP8", section "JAX", delayed scaling).  Per slot s:
 *   1. roll:   hist[h][s] <- hist[h-1][s] for h = H-1 .. 1 (oldest dropped);
 *              hist[0][s] <- amax_new[s]
 *   2. select: a = max_h hist[h][s] (ALGO_MAX; NaN wins) or hist[0][s]
 *              (ALGO_MOST_RECENT)
 *   3. scale:  if a is finite and > 0 and sc = RN(a / FP8_MAX) * 2^margin is
 *              a normal float: scale[s] = sc, scale_inv[s] = RN(1 / sc);
 *              otherwise scale[s] and scale_inv[s] are left unchanged.
 * FP8_MAX = 448 (e4m3fn) or 57344 (e5m2): from slot_format[s] when it is not
 * NULL (0 = e4m3fn, 1 = e5m2, any other code leaves that slot's scale alone),
 * else from fmt for every slot.
 *
 * amax_history: float[history_len][num_slots], row-major, row 0 newest
 * (device, updated in place).  amax_new: float[num_slots] (device, read).
 * scale, scale_inv: float[num_slots] (device, updated in place).
 * slot_format: uint8[num_slots] (device) or NULL.
 * Errors: INVALID_ARG for history_len < 1, num_slots < 1, a NULL or
 *         misaligned float pointer, unknown fmt or algo, margin outside
 *         [-64, 64].  amax_new must not overlap the history.
 */
fp8q_status fp8q_amax_scale_update(float* amax_history, int32_t history_len, int32_t num_slots,
                                   const float* amax_new, float* scale, float* scale_inv,
                                   const uint8_t* slot_format, fp8q_format fmt,
                                   fp8q_amax_algo algo, int32_t margin, void* stream);

/*
 * Fused quantize -> dequantize ("fake quant") with amax, in one pass
 * ("User Guide on Native XLA-FP8", section "Gradient accumulation of FP8
 * params": in_qdq passes a value through Q and DQ with its scale):
 *   y[i]  = bf16_rne( float(FP8(x[i] / *scale)) * *scale )   exactly
 *           fp8q_dequantize(fp8q_quantize_amax(x)), without the FP8 bytes
 *   *amax = max(*amax, max_i |x[i]|)
 * x_bf16: n bf16 (device).  y_bf16: n bf16 (device, written); y_bf16 may equal
 * x_bf16 (in place) but must not partially overlap it.  scale, amax: as for
 * fp8q_quantize_amax.  Errors: as for fp8q_quantize_amax, plus an odd y_bf16.
 */
fp8q_status fp8q_qdq_amax(const void* x_bf16, void* y_bf16, int64_t n, fp8q_format fmt,
                          const float* scale, float* amax, void* stream);

/*
 * amax_and_scale_update over a ring buffer: the same window, selection and
 * scale as fp8q_amax_scale_update, without moving the history.  Each slot's
 * oldest entry is overwritten in place instead of every entry shifting by one
 * row, so a call reads the history and writes one row.  (Window and scale:
 * "Implement fused kernel for FP8 scale update"; "User Guide on Native
 * XLA-FP8", section "JAX", delayed scaling.)  Per slot s, with h = head[s]:
 *   1. h' = (h + 1) mod H;  hist[h'][s] <- amax_new[s];  head[s] <- h'
 *   2. select: a = max over all H rows (ALGO_MAX; NaN wins) or amax_new[s]
 *   3. scale / scale_inv exactly as fp8q_amax_scale_update.
 * Logical row r (0 = newest) of slot s is physical row (head[s] - r) mod H,
 * so after any sequence of calls the window and the scales equal those of the
 * rolled form.  Start with head[s] = H - 1 to fill rows 0, 1, 2, ... in order.
 * A head outside [0, H) leaves that slot's history, head and scales untouched.
 *
 * amax_history: float[H][num_slots] row-major (device, one row per slot
 * written).  head: int32[num_slots] (device, read and advanced).  Other
 * arguments and errors: as for fp8q_amax_scale_update (head is checked like
 * the float pointers).
 */
fp8q_status fp8q_amax_scale_update_ring(float* amax_history, int32_t* head, int32_t history_len,
                                        int32_t num_slots, const float* amax_new, float* scale,
                                        float* scale_inv, const uint8_t* slot_format,
                                        fp8q_format fmt, fp8q_amax_algo algo, int32_t margin,
                                        void* stream);

/*
 * GELU producer fused with quantize + amax: the first MLP layer's output goes
 * through GELU and straight into FP8 for the next FP8 dense layer ("Fusion of
 * Fp8 quantization and amax reduction kernels": the reproducer's
 * dense -> gelu -> dense pattern, with quantization fused into what produces
 * its input), in one pass:
 *   y[i]  = bf16_rne(GELU(h[i]))        tanh form x / (1 + exp(-2u)),
 *                                        u = sqrt(2/pi)(x + 0.044715 x^3)
 *   q[i]  = FP8(y[i] / *scale)           exactly fp8q_quantize_amax of y
 *   *amax = max(*amax, max_i |y[i]|)
 * GELU is evaluated by a fixed sequence of correctly rounded binary32
 * operations (exp by additive range reduction and a degree-6 Taylor
 * polynomial), so it is reproducible bit for bit: y is the bf16 rounding of a
 * value within (6|v| + 10) 2^-24 relative of the exact tanh-form GELU, with
 * v = 2 sqrt(2/pi) x (1 + 0.044715 x^2) (and within 2^-122 absolute where
 * |GELU| < 2^-122).  The codes and the amax are exactly those of quantizing
 * the y returned.
 * h_bf16: n bf16 (device).  y_bf16: n bf16 (device, written) or NULL when only
 * the FP8 codes are wanted.  q, scale, amax: as for fp8q_quantize_amax.
 * Large tensors go through a table of every bf16 input built by thread-block
 * clusters; on a device where no such cluster can be resident (a partitioned
 * or shared GPU) the call takes the element-by-element kernel, with the same
 * results.  The first large call on a device queries how many clusters fit
 * (host-side calls, allowed during graph capture).
 * Errors: as for fp8q_quantize_amax, plus an odd y_bf16.
 */
fp8q_status fp8q_gelu_quantize_amax(const void* h_bf16, void* y_bf16, uint8_t* q, int64_t n,
                                    fp8q_format fmt, const float* scale, float* amax, void* stream);

/*
 * LayerNorm producer fused with quantize + amax: the transformer block of the
 * reproducer in "Fusion of Fp8 quantization and amax reduction kernels"
 * (test.py) normalises its input with a LayerNorm and feeds the MLP's first
 * FP8 dense layer; this computes that layer's FP8 input in one pass over x.
 * Row by row (rows x hidden, row-major), in binary32 with Flax's defaults:
 *   mean = S / H, var = max(0, Q / H - mean^2), rstd = 1 / sqrt(var + eps)
 *   y[i]  = bf16_rne((x[i] - mean) * (rstd * gamma[i]) + beta[i])
 *   q[i]  = FP8(y[i] / *scale)           exactly fp8q_quantize_amax of y
 *   *amax = max(*amax, max |y|)          over every row
 * with S = sum x and Q = sum x^2.  Precision: y is the bf16 rounding of a
 * value within a stated bound of the exact (float64) LayerNorm; the bound
 * follows binary32 error analysis with row sums whose longest chain of
 * additions is at most hidden / 128 + 32 (rows are summed in a fixed order, so
 * a call is reproducible bit for bit), and y is that exact value rounded once to bf16
 * unless it lies close to a bf16 rounding boundary.  The codes and the amax
 * are always exactly those of quantizing the y returned.  A NaN or infinite
 * x makes its row's y NaN.
 * The kernel stages rows of x in shared memory with asynchronous bulk copies
 * and waits for each copy at most one second.  Should a wait ever run out
 * (correct operation never gets there), the call stops early, leaving the
 * outputs incomplete and *amax holding the bit pattern 0x7FFFFFFF: a NaN that
 * no bf16 data can produce (a NaN input gives the canonical 0x7FC00000 or
 * another pattern below 0x7FFFFFFF).  A caller that must tell this apart reads
 * *amax's bits after the stream has reached the call.
 * x_bf16: rows * hidden bf16 (device).  y_bf16: the same (device, written)
 * or NULL when only the FP8 codes are wanted.  q: rows * hidden bytes
 * (device).  gamma, beta: hidden floats each (device).  These five must be
 * 16-byte aligned.  scale, amax: as for fp8q_quantize_amax.  hidden: a
 * multiple of 16 from 16 to 32768.  Rows longer than 4096 run on
 * thread-block clusters of ceil(hidden / 4096) CTAs, each CTA a column slice
 * (up to 96 KB of shared memory); where no cluster of that size fits on the
 * device, one CTA takes each batch of rows instead (rows longer than 16384
 * then take 4 * hidden bytes of shared memory, one CTA per SM).  Both give y
 * within the same bound, not always the same bits.
 * The first call on a device also sets the kernel's shared-memory limit
 * (cudaFuncSetAttribute) and reads its occupancy.  Those are host-side calls,
 * not stream work, so that first call may itself be captured in a CUDA graph.
 * Errors: FP8Q_ERR_INVALID_ARG for a bad fmt, rows < 0, hidden < 16 or not a
 * multiple of 16, a NULL pointer (other than y_bf16) with rows > 0, or a
 * misaligned scale/amax; FP8Q_ERR_UNSUPPORTED for hidden > 32768 or a
 * misaligned x_bf16, y_bf16, q, gamma or beta; FP8Q_ERR_CUDA if the launch
 * or its first-call set-up fails.  rows == 0 launches nothing.
 */
fp8q_status fp8q_layernorm_quantize_amax(const void* x_bf16, void* y_bf16, uint8_t* q, int64_t rows,
                                         int32_t hidden, const float* gamma, const float* beta,
                                         float eps, fp8q_format fmt, const float* scale, float* amax,
                                         void* stream);

/*
 * The ring-buffer update fused with the quantize that follows it, in one
 * launch: the update sits between one step's amax and the next step's casts
 * ("Implement fused kernel for FP8 scale update": one launch per update; the
 * next quantize then needs its new scale), so this call does both:
 *   fp8q_amax_scale_update_ring(history, heads, ...)   for every slot, then
 *   fp8q_quantize_amax(x, q, n, fmt, &scale[slot], amax)
 * with identical results.  The heads come in through head_in (read only) and
 * go out through head_out (written for every slot; swap the two arrays between
 * steps).  The quantizing CTAs compute slot `slot`'s new scale themselves from
 * its history column (without the row the update overwrites) and amax_new,
 * with the update's own arithmetic, so no CTA waits for another.
 * amax_history, history_len, num_slots, amax_new, scale, scale_inv,
 * slot_format, algo, margin: as fp8q_amax_scale_update_ring.  fmt: the FP8
 * format of q, and the format of slots without slot_format (give slot `slot`
 * the format of q).  x_bf16, q, n, amax: as fp8q_quantize_amax; amax must not
 * alias amax_new or the history.  slot: 0 <= slot < num_slots.
 * Errors: those of both calls, plus FP8Q_ERR_INVALID_ARG for a slot out of
 * range or head_out equal to head_in.  n == 0 runs only the update.
 */
fp8q_status fp8q_amax_scale_update_ring_quantize(float* amax_history, const int32_t* head_in,
                                                 int32_t* head_out, int32_t history_len, int32_t num_slots,
                                                 const float* amax_new, float* scale, float* scale_inv,
                                                 const uint8_t* slot_format, fp8q_format fmt,
                                                 fp8q_amax_algo algo, int32_t margin, const void* x_bf16,
                                                 uint8_t* q, int64_t n, int32_t slot, float* amax,
                                                 void* stream);

/* Static, human-readable name of a status. */
const char* fp8q_status_string(fp8q_status status);

/* Text of the calling thread's last FP8Q_ERR_CUDA ("" if none). */
const char* fp8q_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H */
