// quantize.cu -- quantize + amax (single and ragged multi-tensor),
// the fused quantize -> dequantize, and dequantize.

#include "fp8q_common.cuh"
#include "quant_tile.cuh"

#include <mutex>

namespace {

template <int FMT, int MAXT, int OUT>
__global__ void __launch_bounds__(kThreads) quantize_amax_kernel(const __grid_constant__ QList<MAXT> L) {
    __shared__ uint32_t red[kThreads / 32];
    int64_t tile = blockIdx.x;
    if (tile >= L.total_tiles) return;
    // first tensor whose tiles end after this tile (binary search: a CTA starts cold)
    int lo = 0, hi = L.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (tile < L.t[mid].tile_end) hi = mid;
        else lo = mid + 1;
    }
    int ti = lo;
    QCursor k = make_cursor<OUT>(L.t[ti], ti ? L.t[ti - 1].tile_end : 0);
    uint32_t m2 = 0, ms = 0;
    for (; tile < L.total_tiles; tile += gridDim.x) {
        if (tile >= L.t[ti].tile_end) {  // uniform across the CTA
            flush_amax(m2, ms, k.amax, red);
            m2 = 0;
            ms = 0;
            do { ++ti; } while (tile >= L.t[ti].tile_end);
            k = make_cursor<OUT>(L.t[ti], L.t[ti - 1].tile_end);
        }
        quant_tile<FMT, OUT>(k, tile - k.tile_begin, m2, ms);
    }
    flush_amax(m2, ms, k.amax, red);
}

// ----------------------------------------------------------------------------
// Quantize + amax of one tensor by a persistent grid: the tensor's 16-element
// vectors in chunks of kStreamUnroll * kThreads, CTA b taking chunks b, b + G,
// b + 2G, ... (G CTAs), each thread keeping its next two vectors loading while
// it converts the current two.  With one CTA per tile, a tensor of a few waves
// of tiles ends on a partial wave that leaves most SMs idle (2048 tiles over
// 608 resident CTAs is 3.4 waves); here every CTA streams within one chunk of
// the same amount, and at any moment the CTAs work on one window of the tensor
// (measured on 8192x4096 from a cold L2: as fast as contiguous balanced ranges
// per CTA from a clean L2, 4% faster after dirty writes).  The launcher picks
// it for vector-path tensors of at most kStreamMaxTiles tiles (2560: 41.9 M
// elements).

constexpr int kStreamCtasPerSm = 4;
constexpr int kStreamUnroll = 2;

template <int FMT, bool FAST>
__device__ __forceinline__ void stream_range(const QCursor& k, int64_t v0, int64_t end, uint4 (&a)[kStreamUnroll],
                                             uint4 (&b)[kStreamUnroll], uint32_t& m2) {
    const uint16_t* xb = k.x + k.head;
    const int64_t cstride = (int64_t)gridDim.x * kStreamUnroll * kThreads;
    for (; v0 < end; v0 += cstride) {
        uint4 na[kStreamUnroll], nb[kStreamUnroll];
#pragma unroll
        for (int u = 0; u < kStreamUnroll; ++u) {
            const int64_t v = v0 + cstride + u * kThreads;
            if (v < end) ld_stream_v8(xb + v * QuantGeom::kVecElems, na[u], nb[u]);
        }
#pragma unroll
        for (int u = 0; u < kStreamUnroll; ++u) {
            const int64_t v = v0 + u * kThreads;
            if (v < end) quant_vec1<FMT, FAST, kOutFp8>(k, v, a[u], b[u], m2);
        }
#pragma unroll
        for (int u = 0; u < kStreamUnroll; ++u) {
            a[u] = na[u];
            b[u] = nb[u];
        }
    }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, kStreamCtasPerSm) quantize_amax_stream_kernel(const QTensor t) {
    __shared__ uint32_t red[kThreads / 32];
    const Split sp = split_tensor<QuantGeom>((uintptr_t)t.x, (uintptr_t)t.q, t.n);  // the vector path
    const int64_t beg = (int64_t)blockIdx.x * (kStreamUnroll * kThreads);  // this CTA's first chunk
    const int64_t end = sp.nvec;
    uint4 a[kStreamUnroll], b[kStreamUnroll];
    const int64_t v0 = beg + threadIdx.x;
#pragma unroll
    for (int u = 0; u < kStreamUnroll; ++u) {  // loads first: nothing here waits on the scale
        const int64_t v = v0 + u * kThreads;
        if (v < end) ld_stream_v8(t.x + sp.head + v * QuantGeom::kVecElems, a[u], b[u]);
    }
    const QCursor k = make_cursor<kOutFp8>(t, 0);
    uint32_t m2 = 0, ms = 0;
    if (k.c.fast) {
        stream_range<FMT, true>(k, v0, end, a, b, m2);
        if (blockIdx.x == 0) quant_scalars<FMT, true, kOutFp8>(k, 0, ms);  // scalar head and tail
    } else {
        stream_range<FMT, false>(k, v0, end, a, b, m2);
        if (blockIdx.x == 0) quant_scalars<FMT, false, kOutFp8>(k, 0, ms);
    }
    flush_amax(m2, ms, t.amax, red);
}

// ----------------------------------------------------------------------------
// Dequantize


template <int FMT>
__global__ void __launch_bounds__(kThreads)
    dequantize_kernel(const uint8_t* __restrict__ q, uint16_t* __restrict__ y, int64_t n,
                      const float* __restrict__ scale, int64_t tiles) {
    const float s = __ldg(scale);
    const Split sp = split_tensor<DequantGeom>((uintptr_t)y, (uintptr_t)q, n);
    constexpr int E = DequantGeom::kVecElems, U = DequantGeom::kVecPerThread;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        if (sp.mode == kModeVec) {
            const uint8_t* qb = q + sp.head;
            uint16_t* yb = y + sp.head;
            const int64_t v0 = tile * Tile<DequantGeom>::kVecs + threadIdx.x;
            uint2 w[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + (int64_t)u * kThreads;
                if (v < sp.nvec) w[u] = ld_stream_v2(qb + v * E);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + (int64_t)u * kThreads;
                if (v < sp.nvec) {
                    uint4 o;
                    o.x = dequant_pair<FMT>(w[u].x & 0xFFFFu, s);
                    o.y = dequant_pair<FMT>(w[u].x >> 16, s);
                    o.z = dequant_pair<FMT>(w[u].y & 0xFFFFu, s);
                    o.w = dequant_pair<FMT>(w[u].y >> 16, s);
                    st_v4(yb + v * E, o);
                }
            }
            if (tile == 0) {
                const int64_t tail0 = sp.head + sp.nvec * E;
                const int64_t nscalar = sp.head + (n - tail0);
                for (int64_t j = threadIdx.x; j < nscalar; j += kThreads) {
                    const int64_t i = j < sp.head ? j : tail0 + (j - sp.head);
                    y[i] = (uint16_t)(dequant_pair<FMT>(q[i], s) & 0xFFFFu);
                }
            }
        } else {
            const int64_t base = tile * Tile<DequantGeom>::kElems;
            const int64_t end = min(base + (int64_t)Tile<DequantGeom>::kElems, n);
            for (int64_t i = base + threadIdx.x; i < end; i += kThreads)
                y[i] = (uint16_t)(dequant_pair<FMT>(q[i], s) & 0xFFFFu);
        }
    }
}

// ----------------------------------------------------------------------------
// Host side: quantize launchers

// `list[i].q` is the FP8 output, or (OUT == kOutBf16) the bf16 output.
template <int FMT, int MAXT, int OUT = kOutFp8>
fp8q_status launch_quantize(const fp8q_tensor* list, int32_t count, cudaStream_t stream) {
    QList<MAXT> L;
    int64_t tiles = 0;
    int m = 0;
    for (int32_t i = 0; i < count; ++i) {
        const fp8q_tensor& t = list[i];
        const Split sp =
            split_tensor<typename GeomOf<OUT>::type>((uintptr_t)t.x_bf16, (uintptr_t)t.q, t.n);
        if (sp.tiles == 0) continue;  // empty tensors take no tiles and are skipped
        QTensor& d = L.t[m++];
        d.x = static_cast<const uint16_t*>(t.x_bf16);
        d.q = t.q;
        d.scale = t.scale;
        d.amax = t.amax;
        d.n = t.n;
        tiles += sp.tiles;
        d.tile_end = tiles;
    }
    if (tiles == 0) return FP8Q_OK;
    L.total_tiles = tiles;
    L.count = m;
    L.pad = 0;
    // One CTA per tile (16384 elements for quantize, 8192 for the fused
    // quantize -> dequantize); each CTA flushes its amax once.  Measured on
    // GB300 against a persistent grid-stride loop: quantize 61.9 vs 65.9 us and
    // quantize -> dequantize 82.6 vs 110.6 us on 8192x16384.  The kernel's
    // grid-stride loop still covers tile counts beyond the grid limit.
    const int grid = (int)(tiles < 0x7FFFFFFF ? tiles : 0x7FFFFFFF);
    return launch_kernel(quantize_amax_kernel<FMT, MAXT, OUT>, dim3((unsigned)grid), dim3(kThreads), 0, stream,
                         "quantize_amax_kernel", L);
}

// Most tiles (16384 elements each) of a tensor that takes the persistent
// grid; larger tensors run one CTA per tile.  Measured on GB300 (means of 40
// launches): at 2048 tiles the persistent grid takes 16.5 us from a cold,
// clean L2 against 18.5 us (a median), and 14.3 us back to back against 16.3;
// from 3072 tiles up it is faster from a clean L2 (22.5 against 24.7 us at
// 3072) but slower after 256 MB of dirty writes (30.9 against 29.5 us).
constexpr int64_t kStreamMaxTiles = 2560;

// Resident CTAs of the persistent grid per device (multiprocessors x
// kStreamCtasPerSm), read on the first call there.
std::mutex g_sm_mu;
int g_sm_count[64] = {};

cudaError_t sm_count(int* sms) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(g_sm_mu);
    if (dev < 0 || dev >= 64) return cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_sm_count[dev] == 0) {
        err = cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess) return err;
    }
    *sms = g_sm_count[dev];
    return cudaSuccess;
}

template <int FMT>
fp8q_status launch_quantize_one(const fp8q_tensor& t, cudaStream_t stream) {
    const Split sp = split_tensor<QuantGeom>((uintptr_t)t.x_bf16, (uintptr_t)t.q, t.n);
    if (sp.mode != kModeVec || sp.tiles < 2 || sp.tiles > kStreamMaxTiles)
        return launch_quantize<FMT, 1>(&t, 1, stream);
    int sms = 0;
    const cudaError_t err = sm_count(&sms);
    if (err != cudaSuccess) return cuda_fail(err, "quantize_amax_stream_kernel setup");
    const int64_t ctas = (int64_t)sms * kStreamCtasPerSm;
    const int64_t chunks = (sp.nvec + kStreamUnroll * kThreads - 1) / (kStreamUnroll * kThreads);
    const int64_t grid = chunks < ctas ? chunks : ctas;
    QTensor d;
    d.x = static_cast<const uint16_t*>(t.x_bf16);
    d.q = t.q;
    d.scale = t.scale;
    d.amax = t.amax;
    d.n = t.n;
    d.tile_end = 0;
    return launch_kernel(quantize_amax_stream_kernel<FMT>, dim3((unsigned)grid), dim3(kThreads), 0, stream,
                         "quantize_amax_stream_kernel", d);
}

template <int FMT>
fp8q_status dispatch_quantize(const fp8q_tensor* list, int32_t count, cudaStream_t stream) {
    int32_t live = 0;
    for (int32_t i = 0; i < count; ++i) live += list[i].n > 0;
    if (live <= 1) return launch_quantize<FMT, 1>(list, count, stream);
    if (live <= 8) return launch_quantize<FMT, 8>(list, count, stream);
    if (live <= 64) return launch_quantize<FMT, 64>(list, count, stream);
    return launch_quantize<FMT, FP8Q_MAX_TENSORS>(list, count, stream);
}

template <int FMT>
fp8q_status launch_dequantize(const uint8_t* q, void* y, int64_t n, const float* scale,
                              cudaStream_t stream) {
    const Split sp = split_tensor<DequantGeom>((uintptr_t)y, (uintptr_t)q, n);
    // One CTA per tile: for this write-heavy stream (1 byte read, 2 written)
    // the hardware's in-order CTA dispatch keeps the writes more sequential
    // than a persistent grid-stride loop does (measured ~12% faster on GB300).
    // The kernel's loop still covers any tile count beyond the grid limit.
    const int64_t kMaxGrid = 0x7FFFFFFF;
    const int grid = (int)(sp.tiles < kMaxGrid ? sp.tiles : kMaxGrid);
    return launch_kernel(dequantize_kernel<FMT>, dim3((unsigned)grid), dim3(kThreads), 0, stream, "dequantize_kernel",
                         q, static_cast<uint16_t*>(y), n, scale, sp.tiles);
}

}  // namespace

// ----------------------------------------------------------------------------
// C ABI

extern "C" {

fp8q_status fp8q_quantize_amax(const void* x_bf16, uint8_t* q, int64_t n, fp8q_format fmt,
                               const float* scale, float* amax, void* stream) {
    if (!valid_fmt(fmt)) return FP8Q_ERR_INVALID_ARG;
    const fp8q_tensor t = {x_bf16, q, n, scale, amax};
    fp8q_status st = check_tensor(t);
    if (st != FP8Q_OK || n == 0) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return fmt == FP8Q_E4M3FN ? launch_quantize_one<FP8Q_E4M3FN>(t, s) : launch_quantize_one<FP8Q_E5M2>(t, s);
}

fp8q_status fp8q_multi_quantize_amax(const fp8q_tensor* list, int32_t count, fp8q_format fmt,
                                     void* stream) {
    if (!valid_fmt(fmt) || count < 0) return FP8Q_ERR_INVALID_ARG;
    if (count > FP8Q_MAX_TENSORS) return FP8Q_ERR_TOO_MANY_TENSORS;
    if (count == 0) return FP8Q_OK;
    if (!list) return FP8Q_ERR_INVALID_ARG;
    for (int32_t i = 0; i < count; ++i) {
        fp8q_status st = check_tensor(list[i]);
        if (st != FP8Q_OK) return st;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return fmt == FP8Q_E4M3FN ? dispatch_quantize<FP8Q_E4M3FN>(list, count, s)
                              : dispatch_quantize<FP8Q_E5M2>(list, count, s);
}

fp8q_status fp8q_qdq_amax(const void* x_bf16, void* y_bf16, int64_t n, fp8q_format fmt,
                          const float* scale, float* amax, void* stream) {
    if (!valid_fmt(fmt)) return FP8Q_ERR_INVALID_ARG;
    const fp8q_tensor t = {x_bf16, static_cast<uint8_t*>(y_bf16), n, scale, amax};
    fp8q_status st = check_tensor(t);
    if (st != FP8Q_OK || n == 0) return st;
    if ((uintptr_t)y_bf16 & 1u) return FP8Q_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return fmt == FP8Q_E4M3FN ? launch_quantize<FP8Q_E4M3FN, 1, kOutBf16>(&t, 1, s)
                              : launch_quantize<FP8Q_E5M2, 1, kOutBf16>(&t, 1, s);
}

fp8q_status fp8q_dequantize(const uint8_t* q, void* y_bf16, int64_t n, fp8q_format fmt,
                            const float* scale, void* stream) {
    if (!valid_fmt(fmt) || n < 0) return FP8Q_ERR_INVALID_ARG;
    if (n == 0) return FP8Q_OK;
    if (!q || !y_bf16 || !scale || ((uintptr_t)y_bf16 & 1u) || ((uintptr_t)scale & 3u))
        return FP8Q_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return fmt == FP8Q_E4M3FN ? launch_dequantize<FP8Q_E4M3FN>(q, y_bf16, n, scale, s)
                              : launch_dequantize<FP8Q_E5M2>(q, y_bf16, n, scale, s);
}

}  // extern "C"
