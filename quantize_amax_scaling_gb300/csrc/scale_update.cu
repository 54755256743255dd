// scale_update.cu -- the batched amax-history update and scale
// computation, rolled and ring-buffer forms.

#include "fp8q_common.cuh"

namespace {

// ----------------------------------------------------------------------------
// amax history roll + amax selection + scale update

constexpr int kUpdThreads = 256;
constexpr int kUpdCols = 4;                           // slot columns per CTA
constexpr int kUpdRows = 4;                           // rows per thread per chunk
constexpr int kUpdChunk = kUpdThreads * kUpdRows;     // 1024 history rows per chunk

struct UpdArgs {
    float* hist;
    const float* amax_new;
    float* scale;
    float* scale_inv;
    const uint8_t* slot_format;
    int32_t H, S;
    int32_t fmt, algo, margin;
};

// Order-preserving integer key of a non-NaN float (so an integer max is a
// float max); NaN is tracked separately.
__device__ __forceinline__ int float_key(float f) {
    const int b = __float_as_int(f);
    return b ^ ((b >> 31) & 0x7FFFFFFF);
}

__device__ __forceinline__ float key_float(int k) { return __int_as_float(k ^ ((k >> 31) & 0x7FFFFFFF)); }

template <bool VEC4>
__device__ __forceinline__ float4 load_row(const UpdArgs& a, int64_t row, int c0, int ncols) {
    const float* p = a.hist + row * a.S + c0;
    if (VEC4) return *reinterpret_cast<const float4*>(p);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ncols > 0) v.x = p[0];
    if (ncols > 1) v.y = p[1];
    if (ncols > 2) v.z = p[2];
    if (ncols > 3) v.w = p[3];
    return v;
}

template <bool VEC4>
__device__ __forceinline__ void store_row(const UpdArgs& a, int64_t row, int c0, int ncols, float4 v) {
    float* p = a.hist + row * a.S + c0;
    if (VEC4) {
        *reinterpret_cast<float4*>(p) = v;
        return;
    }
    if (ncols > 0) p[0] = v.x;
    if (ncols > 1) p[1] = v.y;
    if (ncols > 2) p[2] = v.z;
    if (ncols > 3) p[3] = v.w;
}

__device__ __forceinline__ void fold(int (&key)[4], bool (&nan)[4], float4 v) {
    const float c[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        nan[j] |= isnan(c[j]);
        key[j] = max(key[j], float_key(c[j]));
    }
}

// Scale and scale_inv of one slot from its selected amax, or pass-through.
__device__ __forceinline__ void slot_scale(float amax, int f, int margin, float* scale, float* scale_inv) {
    if ((f == FP8Q_E4M3FN || f == FP8Q_E5M2) && isfinite(amax) && amax > 0.0f) {
        const float fp8max = (f == FP8Q_E4M3FN) ? 448.0f : 57344.0f;
        const float pow2m = __uint_as_float((uint32_t)(127 + margin) << 23);  // exact 2^margin
        const float sc = __fmul_rn(__fdiv_rn(amax, fp8max), pow2m);
        if (sc >= 0x1p-126f && sc <= 0x1.fffffep127f) {  // normal and finite
            *scale = sc;
            *scale_inv = __frcp_rn(sc);
        }
    }
}

template <bool VEC4>
__global__ void __launch_bounds__(kUpdThreads) amax_scale_update_kernel(const UpdArgs a) {
    __shared__ int s_key[kUpdThreads / 32][kUpdCols];
    __shared__ int s_nan[kUpdThreads / 32][kUpdCols];
    const int c0 = blockIdx.x * kUpdCols;
    const int ncols = min(kUpdCols, a.S - c0);
    const int64_t H = a.H;
    const bool want_max = (a.algo == FP8Q_ALGO_MAX);

    int key[4] = {INT_MIN, INT_MIN, INT_MIN, INT_MIN};
    bool nan[4] = {false, false, false, false};

    // The per-slot inputs are fetched first so their latency overlaps the
    // history loads instead of adding round trips after the barrier.
    float newest = 0.0f;
    int slot_fmt = a.fmt;
    if (threadIdx.x < ncols) {
        newest = a.amax_new[c0 + threadIdx.x];
        if (a.slot_format) slot_fmt = a.slot_format[c0 + threadIdx.x];
    }

    float4 cur[kUpdRows], nxt[kUpdRows];
#pragma unroll
    for (int k = 0; k < kUpdRows; ++k) {
        const int64_t r = threadIdx.x + (int64_t)k * kUpdThreads;
        if (r < H) cur[k] = load_row<VEC4>(a, r, c0, ncols);
    }
    for (int64_t base = 0; base < H; base += kUpdChunk) {
        const bool more = base + kUpdChunk < H;
        if (more) {
#pragma unroll
            for (int k = 0; k < kUpdRows; ++k) {
                const int64_t r = base + kUpdChunk + threadIdx.x + (int64_t)k * kUpdThreads;
                if (r < H) nxt[k] = load_row<VEC4>(a, r, c0, ncols);
            }
        }
        if (want_max) {
            // old rows 0..H-2 survive the roll; row H-1 drops out of the window
#pragma unroll
            for (int k = 0; k < kUpdRows; ++k) {
                const int64_t r = base + threadIdx.x + (int64_t)k * kUpdThreads;
                if (r + 1 < H) fold(key, nan, cur[k]);
            }
        }
        __syncthreads();  // every read of rows <= base + 2*chunk - 1 precedes the writes below
#pragma unroll
        for (int k = 0; k < kUpdRows; ++k) {
            const int64_t r = base + threadIdx.x + (int64_t)k * kUpdThreads;
            if (r + 1 < H) store_row<VEC4>(a, r + 1, c0, ncols, cur[k]);
        }
        if (more) {
#pragma unroll
            for (int k = 0; k < kUpdRows; ++k) cur[k] = nxt[k];
        }
    }
    // Row 0 was read before the first barrier; now it receives the new amax.
    if (threadIdx.x < ncols) a.hist[c0 + threadIdx.x] = newest;

    if (want_max) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int kw = __reduce_max_sync(0xFFFFFFFFu, key[j]);
            const bool nw = __any_sync(0xFFFFFFFFu, nan[j]);
            if (lane == 0) {
                s_key[warp][j] = kw;
                s_nan[warp][j] = nw;
            }
        }
        __syncthreads();
    }
    if (threadIdx.x < ncols) {
        const int j = threadIdx.x;
        const int s = c0 + j;
        float amax = newest;
        if (want_max) {
            int kb = INT_MIN;
            bool nb = isnan(newest);
            for (int w = 0; w < kUpdThreads / 32; ++w) {
                kb = max(kb, s_key[w][j]);
                nb |= (s_nan[w][j] != 0);
            }
            if (H > 1) amax = fmaxf(amax, key_float(kb));
            if (nb) amax = __int_as_float(0x7FC00000);
        }
        slot_scale(amax, slot_fmt, a.margin, a.scale + s, a.scale_inv + s);
    }
}

// Ring-buffer form of the update: the window stays where it is and only each
// slot's oldest row is overwritten.  head[s] is the physical row of slot s's
// newest entry.  Same CTA layout as the rolled kernel (4 slot columns per CTA,
// all their rows), so each CTA reads and advances only its own heads; nothing
// is shifted, so there is no barrier between the reads and the writes.
template <bool VEC4>
__global__ void __launch_bounds__(kUpdThreads) amax_scale_update_ring_kernel(const UpdArgs a,
                                                                            int32_t* head) {
    __shared__ int s_key[kUpdThreads / 32][kUpdCols];
    __shared__ int s_nan[kUpdThreads / 32][kUpdCols];
    const int c0 = blockIdx.x * kUpdCols;
    const int ncols = min(kUpdCols, a.S - c0);
    const int64_t H = a.H;
    const bool want_max = (a.algo == FP8Q_ALGO_MAX);

    // the row each column's new entry goes to (-1: corrupt head, slot untouched)
    int hn[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int h = j < ncols ? head[c0 + j] : -1;
        hn[j] = (h >= 0 && h < a.H) ? (h + 1 == a.H ? 0 : h + 1) : -1;
    }
    float newest = 0.0f;
    int slot_fmt = a.fmt;
    if (threadIdx.x < ncols) {
        newest = a.amax_new[c0 + threadIdx.x];
        if (a.slot_format) slot_fmt = a.slot_format[c0 + threadIdx.x];
    }

    int key[4] = {INT_MIN, INT_MIN, INT_MIN, INT_MIN};
    bool nan[4] = {false, false, false, false};
    if (want_max) {
        for (int64_t base = 0; base < H; base += kUpdChunk) {
            float4 v[kUpdRows];
#pragma unroll
            for (int k = 0; k < kUpdRows; ++k) {
                const int64_t r = base + threadIdx.x + (int64_t)k * kUpdThreads;
                if (r < H) v[k] = load_row<VEC4>(a, r, c0, ncols);
            }
#pragma unroll
            for (int k = 0; k < kUpdRows; ++k) {
                const int64_t r = base + threadIdx.x + (int64_t)k * kUpdThreads;
                if (r < H) {
                    // the oldest entry (row hn) leaves the window
                    const float c[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (r == hn[j]) continue;
                        nan[j] |= isnan(c[j]);
                        key[j] = max(key[j], float_key(c[j]));
                    }
                }
            }
        }
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int kw = __reduce_max_sync(0xFFFFFFFFu, key[j]);
            const bool nw = __any_sync(0xFFFFFFFFu, nan[j]);
            if (lane == 0) {
                s_key[warp][j] = kw;
                s_nan[warp][j] = nw;
            }
        }
        __syncthreads();  // every row has been read; only now is the oldest one replaced
    }
    const int j = threadIdx.x;
    const int my_hn = j == 0 ? hn[0] : j == 1 ? hn[1] : j == 2 ? hn[2] : hn[3];
    if (j < ncols && my_hn >= 0) {
        const int s = c0 + j;
        float amax = newest;
        if (want_max) {
            int kb = INT_MIN;
            bool nb = isnan(newest);
            for (int w = 0; w < kUpdThreads / 32; ++w) {
                kb = max(kb, s_key[w][j]);
                nb |= (s_nan[w][j] != 0);
            }
            if (H > 1) amax = fmaxf(amax, key_float(kb));
            if (nb) amax = __int_as_float(0x7FC00000);
        }
        a.hist[(int64_t)my_hn * a.S + s] = newest;
        head[s] = my_hn;
        slot_scale(amax, slot_fmt, a.margin, a.scale + s, a.scale_inv + s);
    }
}

}  // namespace

// ----------------------------------------------------------------------------
// C ABI

extern "C" {

fp8q_status fp8q_amax_scale_update(float* amax_history, int32_t history_len, int32_t num_slots,
                                   const float* amax_new, float* scale, float* scale_inv,
                                   const uint8_t* slot_format, fp8q_format fmt,
                                   fp8q_amax_algo algo, int32_t margin, void* stream) {
    if (history_len < 1 || num_slots < 1 || !valid_fmt(fmt)) return FP8Q_ERR_INVALID_ARG;
    if (algo != FP8Q_ALGO_MAX && algo != FP8Q_ALGO_MOST_RECENT) return FP8Q_ERR_INVALID_ARG;
    if (margin < -64 || margin > 64) return FP8Q_ERR_INVALID_ARG;
    const void* fp[4] = {amax_history, amax_new, scale, scale_inv};
    for (const void* p : fp)
        if (!p || ((uintptr_t)p & 3u)) return FP8Q_ERR_INVALID_ARG;
    UpdArgs a;
    a.hist = amax_history;
    a.amax_new = amax_new;
    a.scale = scale;
    a.scale_inv = scale_inv;
    a.slot_format = slot_format;
    a.H = history_len;
    a.S = num_slots;
    a.fmt = fmt;
    a.algo = algo;
    a.margin = margin;
    const int grid = (num_slots + kUpdCols - 1) / kUpdCols;
    const bool vec4 = ((uintptr_t)amax_history & 15u) == 0 && (num_slots % kUpdCols) == 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (vec4) amax_scale_update_kernel<true><<<grid, kUpdThreads, 0, s>>>(a);
    else      amax_scale_update_kernel<false><<<grid, kUpdThreads, 0, s>>>(a);
    return after_launch("amax_scale_update_kernel");
}

fp8q_status fp8q_amax_scale_update_ring(float* amax_history, int32_t* head, int32_t history_len,
                                        int32_t num_slots, const float* amax_new, float* scale,
                                        float* scale_inv, const uint8_t* slot_format, fp8q_format fmt,
                                        fp8q_amax_algo algo, int32_t margin, void* stream) {
    if (history_len < 1 || num_slots < 1 || !valid_fmt(fmt)) return FP8Q_ERR_INVALID_ARG;
    if (algo != FP8Q_ALGO_MAX && algo != FP8Q_ALGO_MOST_RECENT) return FP8Q_ERR_INVALID_ARG;
    if (margin < -64 || margin > 64) return FP8Q_ERR_INVALID_ARG;
    const void* fp[5] = {amax_history, head, amax_new, scale, scale_inv};
    for (const void* p : fp)
        if (!p || ((uintptr_t)p & 3u)) return FP8Q_ERR_INVALID_ARG;
    UpdArgs a;
    a.hist = amax_history;
    a.amax_new = amax_new;
    a.scale = scale;
    a.scale_inv = scale_inv;
    a.slot_format = slot_format;
    a.H = history_len;
    a.S = num_slots;
    a.fmt = fmt;
    a.algo = algo;
    a.margin = margin;
    const int grid = (num_slots + kUpdCols - 1) / kUpdCols;
    const bool vec4 = ((uintptr_t)amax_history & 15u) == 0 && (num_slots % kUpdCols) == 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (vec4) amax_scale_update_ring_kernel<true><<<grid, kUpdThreads, 0, s>>>(a, head);
    else      amax_scale_update_ring_kernel<false><<<grid, kUpdThreads, 0, s>>>(a, head);
    return after_launch("amax_scale_update_ring_kernel");
}

}  // extern "C"
