// scale_update.cu -- the batched amax-history update and scale
// computation, rolled and ring-buffer forms.

#include "fp8q_common.cuh"
#include "quant_tile.cuh"
#include "slot_math.cuh"

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

// Column j's selected amax -- the new entry and, for max, the warps' maxima of
// the rows that survive the roll -- and its scale.
__device__ __forceinline__ void finish_slot(const UpdArgs& a, int c0, int j, float newest, int slot_fmt,
                                            bool want_max, const int (&s_key)[kUpdThreads / 32][kUpdCols],
                                            const int (&s_nan)[kUpdThreads / 32][kUpdCols]) {
    float amax = newest;
    if (want_max) {
        int kb = INT_MIN;
        bool nb = isnan(newest);
        for (int w = 0; w < kUpdThreads / 32; ++w) {
            kb = max(kb, s_key[w][j]);
            nb |= (s_nan[w][j] != 0);
        }
        if (a.H > 1) amax = fmaxf(amax, key_float(kb));
        if (nb) amax = __int_as_float(0x7FC00000);
    }
    slot_scale(amax, slot_fmt, a.margin, a.scale + c0 + j, a.scale_inv + c0 + j);
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

    if (H <= kUpdChunk) {
        // One chunk, in blocks: thread t holds rows kUpdRows t ... kUpdRows t + kUpdRows - 1.
        // The roll moves each of them one row older.  All but the last land in rows of the
        // same block, which only this thread reads, so they are stored as soon as they
        // are loaded; the last lands in the first row of the next thread's block and
        // waits for the barrier below, by which time every row has been read.
        float4 v[kUpdRows];
        const int64_t r0 = (int64_t)threadIdx.x * kUpdRows;
#pragma unroll
        for (int k = 0; k < kUpdRows; ++k)
            if (r0 + k < H) v[k] = load_row<VEC4>(a, r0 + k, c0, ncols);
        if (want_max) {
            // old rows 0..H-2 survive the roll; row H-1 drops out of the window
#pragma unroll
            for (int k = 0; k < kUpdRows; ++k)
                if (r0 + k + 1 < H) fold(key, nan, v[k]);
        }
#pragma unroll
        for (int k = 0; k + 1 < kUpdRows; ++k)
            if (r0 + k + 1 < H) store_row<VEC4>(a, r0 + k + 1, c0, ncols, v[k]);
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
        }
        __syncthreads();  // every row has been read; the warps' maxima are in shared memory
        if (r0 + kUpdRows < H) store_row<VEC4>(a, r0 + kUpdRows, c0, ncols, v[kUpdRows - 1]);
        // row 0 (read above by thread 0) receives the new amax
        if (threadIdx.x < ncols) a.hist[c0 + threadIdx.x] = newest;
        if (threadIdx.x < ncols) finish_slot(a, c0, threadIdx.x, newest, slot_fmt, want_max, s_key, s_nan);
        return;
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
    if (threadIdx.x < ncols) finish_slot(a, c0, threadIdx.x, newest, slot_fmt, want_max, s_key, s_nan);
}

// Ring-buffer form of the update: the window stays where it is and only each
// slot's oldest row is overwritten.  head[s] is the physical row of slot s's
// newest entry.  Same CTA layout as the rolled kernel (4 slot columns per CTA,
// all their rows), so each CTA reads and advances only its own heads; nothing
// is shifted, so there is no barrier between the reads and the writes.
//
// head_in is read, head_out written (the same array for the in-place call):
// a slot with a head outside [0, H) is left alone and its head copied.
template <bool VEC4>
__device__ __forceinline__ void ring_update_cols(const UpdArgs& a, const int32_t* head_in, int32_t* head_out,
                                                 int c0) {
    __shared__ int s_key[kUpdThreads / 32][kUpdCols];
    __shared__ int s_nan[kUpdThreads / 32][kUpdCols];
    const int ncols = min(kUpdCols, a.S - c0);
    const int64_t H = a.H;
    const bool want_max = (a.algo == FP8Q_ALGO_MAX);

    // the row each column's new entry goes to (-1: corrupt head, slot untouched)
    int hn[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int h = j < ncols ? head_in[c0 + j] : -1;
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
    if (j < ncols && my_hn < 0 && head_out != head_in) head_out[c0 + j] = head_in[c0 + j];
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
        head_out[s] = my_hn;
        slot_scale(amax, slot_fmt, a.margin, a.scale + s, a.scale_inv + s);
    }
}

template <bool VEC4>
__global__ void __launch_bounds__(kUpdThreads) amax_scale_update_ring_kernel(const UpdArgs a,
                                                                            int32_t* head) {
    ring_update_cols<VEC4>(a, head, head, blockIdx.x * kUpdCols);
}

// ----------------------------------------------------------------------------
// The ring-buffer update fused with the next quantize, in one launch.
//
// The first ceil(S / 4) CTAs run the ring update of their slot columns, as
// above, with the heads read from head_in and written to head_out.  Every
// other CTA quantizes tiles of x with slot `slot`'s new scale, which it
// computes itself from what the update reads: the slot's history column
// without the row the update overwrites (the oldest), and amax_new.  So no
// CTA reads anything another CTA of the launch writes, except scale[slot] in
// the pass-through case, which the update then leaves untouched; no CTA waits
// for another.  new_slot_scale is the update's own arithmetic, so the scale
// the quantize uses has the same bits as the one the update stores.

// Slot `slot`'s scale after the update (block-wide: every thread calls it).
__device__ __forceinline__ float scale_after_update(const UpdArgs& a, const int32_t* head_in, int slot,
                                                    int* s_key, int* s_nan) {
    const int h = head_in[slot];
    const bool valid = h >= 0 && h < a.H;
    const int hn = valid ? (h + 1 == a.H ? 0 : h + 1) : -1;
    const float newest = a.amax_new[slot];
    const int f = a.slot_format ? (int)a.slot_format[slot] : a.fmt;
    float amax = newest;
    if (a.algo == FP8Q_ALGO_MAX) {
        int key = INT_MIN;
        bool nan = false;
        for (int64_t r = threadIdx.x; r < a.H; r += kThreads) {
            if (r == hn) continue;  // the oldest entry leaves the window
            const float v = a.hist[r * a.S + slot];
            nan |= isnan(v);
            key = max(key, float_key(v));
        }
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        key = __reduce_max_sync(0xFFFFFFFFu, key);
        nan = __any_sync(0xFFFFFFFFu, nan);
        if (lane == 0) {
            s_key[warp] = key;
            s_nan[warp] = nan;
        }
        __syncthreads();
        int kb = INT_MIN;
        bool nb = isnan(newest);
        for (int w = 0; w < kThreads / 32; ++w) {
            kb = max(kb, s_key[w]);
            nb |= (s_nan[w] != 0);
        }
        if (a.H > 1) amax = fmaxf(amax, key_float(kb));
        if (nb) amax = __int_as_float(0x7FC00000);
    }
    float sc;
    if (valid && new_slot_scale(amax, f, a.margin, &sc)) return sc;
    return a.scale[slot];  // unchanged: the update does not write it
}

// Most quantizing CTAs (152 SMs x 16): each reads the slot's history column
// once, so fewer CTAs looping over tiles beat one CTA per tile here (measured
// on 8192x16384 with 1024 rows: 65.3 us, against 74.0 us with one CTA per
// tile and 71.4 us with 608 CTAs).
constexpr int64_t kFusedQuantCtas = 2432;

template <int FMT, bool VEC4>
__global__ void __launch_bounds__(kThreads, 4) ring_update_quantize_kernel(const UpdArgs a, const int32_t* head_in,
                                                                        int32_t* head_out, int n_upd,
                                                                        const QTensor t, int slot, int64_t tiles) {
    static_assert(kUpdThreads == kThreads, "one block size for both roles");
    if ((int)blockIdx.x < n_upd) {
        ring_update_cols<VEC4>(a, head_in, head_out, blockIdx.x * kUpdCols);
        return;
    }
    __shared__ uint32_t red[kThreads / 32];
    __shared__ int s_key[kThreads / 32];
    __shared__ int s_nan[kThreads / 32];
    const int64_t stride = (int64_t)gridDim.x - n_upd;
    int64_t tile = (int64_t)blockIdx.x - n_upd;
    QCursor k = make_cursor_with<kOutFp8>(t, 0, QScale{});
    TileRegs<kOutFp8> r;
    if (tile < tiles && k.mode == kModeVec) quant_vec_load<kOutFp8>(k, tile, r);  // in flight meanwhile
    k.c = make_qscale_value(scale_after_update(a, head_in, slot, s_key, s_nan));
    uint32_t m2 = 0, ms = 0;
    for (bool first = true; tile < tiles; tile += stride, first = false) {
        if (!first && k.mode == kModeVec) quant_vec_load<kOutFp8>(k, tile, r);
        if (k.c.fast) {
            if (k.mode == kModeVec) quant_vec_store<FMT, true, kOutFp8>(k, tile, r, m2);
            quant_scalars<FMT, true, kOutFp8>(k, tile, ms);
        } else {
            if (k.mode == kModeVec) quant_vec_store<FMT, false, kOutFp8>(k, tile, r, m2);
            quant_scalars<FMT, false, kOutFp8>(k, tile, ms);
        }
    }
    flush_amax(m2, ms, t.amax, red);
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
    return vec4 ? launch_kernel(amax_scale_update_kernel<true>, dim3(grid), dim3(kUpdThreads), 0, s,
                                "amax_scale_update_kernel", a)
                : launch_kernel(amax_scale_update_kernel<false>, dim3(grid), dim3(kUpdThreads), 0, s,
                                "amax_scale_update_kernel", a);
}

fp8q_status fp8q_amax_scale_update_ring_quantize(float* amax_history, const int32_t* head_in,
                                                 int32_t* head_out, int32_t history_len, int32_t num_slots,
                                                 const float* amax_new, float* scale, float* scale_inv,
                                                 const uint8_t* slot_format, fp8q_format fmt,
                                                 fp8q_amax_algo algo, int32_t margin, const void* x_bf16,
                                                 uint8_t* q, int64_t n, int32_t slot, float* amax,
                                                 void* stream) {
    if (history_len < 1 || num_slots < 1 || !valid_fmt(fmt)) return FP8Q_ERR_INVALID_ARG;
    if (algo != FP8Q_ALGO_MAX && algo != FP8Q_ALGO_MOST_RECENT) return FP8Q_ERR_INVALID_ARG;
    if (margin < -64 || margin > 64) return FP8Q_ERR_INVALID_ARG;
    if (slot < 0 || slot >= num_slots) return FP8Q_ERR_INVALID_ARG;
    const void* fp[6] = {amax_history, head_in, head_out, amax_new, scale, scale_inv};
    for (const void* p : fp)
        if (!p || ((uintptr_t)p & 3u)) return FP8Q_ERR_INVALID_ARG;
    if ((const void*)head_in == (const void*)head_out) return FP8Q_ERR_INVALID_ARG;
    const fp8q_tensor ft = {x_bf16, q, n, scale + slot, amax};
    const fp8q_status st = check_tensor(ft);
    if (st != FP8Q_OK) return st;
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
    QTensor t;
    t.x = static_cast<const uint16_t*>(x_bf16);
    t.q = q;
    t.scale = scale + slot;
    t.amax = amax;
    t.n = n;
    t.tile_end = 0;
    const Split sp = split_tensor<QuantGeom>((uintptr_t)x_bf16, (uintptr_t)q, n);
    const int n_upd = (num_slots + kUpdCols - 1) / kUpdCols;
    const int64_t max_q = kFusedQuantCtas;
    const int grid = n_upd + (int)(sp.tiles < max_q ? sp.tiles : max_q);
    const bool vec4 = ((uintptr_t)amax_history & 15u) == 0 && (num_slots % kUpdCols) == 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto kern = fmt == FP8Q_E4M3FN ? (vec4 ? ring_update_quantize_kernel<FP8Q_E4M3FN, true>
                                           : ring_update_quantize_kernel<FP8Q_E4M3FN, false>)
                                    : (vec4 ? ring_update_quantize_kernel<FP8Q_E5M2, true>
                                           : ring_update_quantize_kernel<FP8Q_E5M2, false>);
    return launch_kernel(kern, dim3(grid), dim3(kThreads), 0, s, "ring_update_quantize_kernel", a, head_in, head_out,
                         n_upd, t, slot, sp.tiles);
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
    return launch_kernel(vec4 ? amax_scale_update_ring_kernel<true> : amax_scale_update_ring_kernel<false>, dim3(grid),
                         dim3(kUpdThreads), 0, s, "amax_scale_update_ring_kernel", a, head);
}

}  // extern "C"
