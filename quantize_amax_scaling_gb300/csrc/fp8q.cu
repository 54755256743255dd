// fp8q.cu -- sm_103a kernels and the C ABI of libfp8q (see include/fp8q.h).
//
// Sources (web pages, by title and section):
//   "User Guide on Native XLA-FP8" (NVIDIA JAX-Toolbox), section "JAX":
//     Q = cast(A / A_scale), DQ = cast(a_fp8) * a_scale, delayed scaling
//     A_scale = max|A| / E4M3_MAX.
//   "Fusion of Fp8 quantization and amax reduction kernels" (openxla/xla
//     issue): Q and the amax reduction are memory bound; fuse them.
//   "Implement fused kernel for FP8 scale update" (TransformerEngine PR):
//     the whole amax_and_scale_update in one in-place kernel, all layers.
//
// Every kernel here streams HBM; none is a contraction, so there are no
// tensor-core instructions.  Design points:
//   * quantize+amax reads each bf16 once (32-byte vector loads), writes each
//     FP8 byte once (16-byte stores), and reduces |x| with packed
//     NaN-propagating bf16x2 max, then one warp redux and one atomic per CTA
//     and tensor.  Each tile's loads are issued before anything waits on the
//     scale's own load.
//   * every streaming kernel launches one CTA per tile (16 KB to 32 KB of
//     input); on GB300 this beat a persistent grid-stride loop for all three,
//     most of all for the write-heavy dequantize and quantize -> dequantize.
//   * the division x / scale is exact IEEE binary32 (round to nearest even)
//     without a per-element divide: with r = RN(1/s) computed once per CTA,
//     y0 = RN(x*r), e = fma(y0, s, -x), y = fma(-e, r, y0) is the correctly
//     rounded quotient (Markstein's correction step, P. Markstein, "Computation
//     of elementary functions on the IBM RISC System/6000 processor", IBM J.
//     Res. Dev. 34(1), 1990).  This was checked for every bf16 significand
//     against every binary32 scale significand; it is used for positive scales
//     in [2^-60, 2^60], where no intermediate leaves the normal range while the
//     quotient lies in [2^-18, 2^17] (outside that band the FP8 result is a
//     signed zero or saturated, and the error there cannot change it).  Inputs
//     are clamped to |x| <= RU_bf16(s * 2^17) first (NaN kept), so x*r cannot
//     overflow and +-inf saturates.  Other scales use __fdiv_rn per element.
//   * the ragged multi-tensor launch numbers the tiles of all its tensors in
//     one sequence; a CTA finds its tensor by binary search over the
//     descriptors, which travel by value in the kernel parameters, so the
//     launch needs no host-to-device copy.
//   * the scale update gives each CTA four slot columns and every history row
//     of them, reads all rows into registers, synchronises, then writes the
//     rows shifted by one; no other CTA touches those columns, so the in-place
//     roll needs no grid-wide synchronisation.  The ring-buffer form keeps the
//     same layout, overwrites only each slot's oldest row and advances a
//     per-slot head that only the owning CTA touches.
//   * no kernel waits on another CTA, a flag or an mbarrier: the only waits are
//     __syncthreads in uniform control flow.

#include "fp8q.h"

#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstdio>

namespace {

// ----------------------------------------------------------------------------
// Error reporting

thread_local char g_last_error[256] = "";

fp8q_status cuda_fail(cudaError_t e, const char* where) {
    std::snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", where, cudaGetErrorName(e),
                  cudaGetErrorString(e));
    return FP8Q_ERR_CUDA;
}

fp8q_status after_launch(const char* where) {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? FP8Q_OK : cuda_fail(e, where);
}

// ----------------------------------------------------------------------------
// Launch geometry

constexpr int kThreads = 256;  // threads per CTA (streaming kernels)

// Vector geometry of the streaming kernels.  A thread moves vectors of
// kVecElems elements; a tile is kVecPerThread vectors per thread.  The "wide"
// side is the bf16 input (quantize) or output (dequantize); the "narrow" side
// is the other tensor, with kNarrowBytes per element, and must be
// kNarrowAlign-byte aligned wherever the wide side is kWideAlign-aligned.
//   quantize:   16 bf16 (one 32-byte load) -> 16 codes (one 16-byte store), 4 per thread
//   dequantize: 8 codes (one 8-byte load)  -> 8 bf16 (one 16-byte store)
//   fused Q->DQ: 16 bf16 (one 32-byte load) -> 16 bf16 (two 16-byte stores)
struct QuantGeom {
    static constexpr int kVecElems = 16;
    static constexpr int kVecPerThread = 4;
    static constexpr int kWideAlign = 32;
    static constexpr int kNarrowBytes = 1;
    static constexpr int kNarrowAlign = 16;
};
struct DequantGeom {
    static constexpr int kVecElems = 8;
    static constexpr int kVecPerThread = 4;
    static constexpr int kWideAlign = 16;
    static constexpr int kNarrowBytes = 1;
    static constexpr int kNarrowAlign = 8;
};
struct QdqGeom {
    static constexpr int kVecElems = 16;
    static constexpr int kVecPerThread = 2;
    static constexpr int kWideAlign = 32;
    static constexpr int kNarrowBytes = 2;
    static constexpr int kNarrowAlign = 16;
};
template <class G>
struct Tile {
    static constexpr int kVecs = kThreads * G::kVecPerThread;
    static constexpr int kElems = kVecs * G::kVecElems;  // 8192 for both kernels
};

enum : int { kModeVec = 0, kModeScalar = 1 };

// How a tensor is split: `head` scalar elements until the wide pointer is
// G::kWideAlign-byte aligned, then `nvec` vectors, then a scalar tail shorter
// than one vector.  The narrow pointer must then be G::kNarrowAlign-byte
// aligned at the same element; otherwise the whole tensor is processed element
// by element.  Host and device both call this, so they agree on the tile count.
struct Split {
    int64_t head, nvec, tiles;
    int mode;
};

template <class G>
__host__ __device__ inline Split split_tensor(uintptr_t wide, uintptr_t narrow, int64_t n) {
    Split s;
    if (n <= 0) {
        s.head = 0; s.nvec = 0; s.tiles = 0; s.mode = kModeVec;
        return s;
    }
    const unsigned wa = G::kWideAlign;
    int64_t h = (int64_t)(((wa - (unsigned)(wide & (wa - 1))) & (wa - 1)) >> 1);
    if (h > n) h = n;
    if (((narrow + (uintptr_t)h * G::kNarrowBytes) & (uintptr_t)(G::kNarrowAlign - 1)) == 0) {
        s.mode = kModeVec;
        s.head = h;
        s.nvec = (n - h) / G::kVecElems;
        int64_t t = (s.nvec + Tile<G>::kVecs - 1) / Tile<G>::kVecs;
        s.tiles = t > 0 ? t : 1;  // tile 0 also carries the scalar head and tail
    } else {
        s.mode = kModeScalar;
        s.head = n;
        s.nvec = 0;
        s.tiles = (n + Tile<G>::kElems - 1) / Tile<G>::kElems;
    }
    return s;
}

// ----------------------------------------------------------------------------
// Device helpers (inline PTX: documented instructions only).  Inputs are read
// once: loads skip L1 and ask L2 to fetch whole 256-byte blocks; outputs
// are written once: stores are marked streaming (evict-first) so L2 drains them
// to HBM early instead of holding them against the next kernel.

__device__ __forceinline__ void ld_stream_v8(const void* p, uint4& a, uint4& b) {
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                 : "l"(p));
}

__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// max(|a|, |b|) per bf16 lane; NaN in either gives the canonical NaN.  The
// result's sign is sign(a) ^ sign(b) and is ignored by every caller.
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// sign(a) * min(|a|, t) per bf16 lane for t >= 0; NaN stays NaN.
__device__ __forceinline__ uint32_t bf16x2_clamp(uint32_t a, uint32_t t2) {
    uint32_t d;
    asm("min.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(t2));
    return d;
}

// Two binary32 values -> two saturated, RNE FP8 codes; `lo` lands in the low byte.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_fp8x2(float lo, float hi) {
    uint16_t d;
    if (FMT == FP8Q_E4M3FN)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// Two FP8 codes (low byte first) -> two half values, exact.
template <int FMT>
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint32_t pair) {
    uint32_t d;
    if (FMT == FP8Q_E4M3FN) {
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"((uint16_t)pair));
    } else {
        // an e5m2 code is the upper byte of the half with the same value
        d = __byte_perm(pair, 0u, 0x1404);  // bytes: [0]=0, [1]=b0, [2]=0, [3]=b1
    }
    return d;
}

__device__ __forceinline__ float f16_lo(uint32_t h2) {
    float f;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.f32.f16 %0, l; }" : "=f"(f) : "r"(h2));
    return f;
}

__device__ __forceinline__ float f16_hi(uint32_t h2) {
    float f;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.f32.f16 %0, h; }" : "=f"(f) : "r"(h2));
    return f;
}

// Two binary32 -> packed bf16x2, round to nearest even; `lo` in the low half.
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Two FP8 codes (one 16-bit pair, low byte first) -> two bf16 (one word):
// exact widening, one binary32 multiply each, round to nearest-even bf16.
template <int FMT>
__device__ __forceinline__ uint32_t dequant_pair(uint32_t pair, float s) {
    const uint32_t h2 = fp8x2_to_f16x2<FMT>(pair);
    return cvt_bf16x2(__fmul_rn(f16_lo(h2), s), __fmul_rn(f16_hi(h2), s));
}

// ----------------------------------------------------------------------------
// Quantize + amax (and the fused quantize -> dequantize, which shares it)

enum : int { kOutFp8 = 0, kOutBf16 = 1 };  // what the quantize kernel writes
template <int OUT>
struct GeomOf { using type = QuantGeom; };
template <>
struct GeomOf<kOutBf16> { using type = QdqGeom; };

// Per-tensor constants a CTA derives from the scale.
struct QScale {
    float s;      // the scale
    float r;      // RN(1 / s)
    uint32_t t2;  // clamp bound RU_bf16(s * 2^17), in both bf16 lanes
    bool fast;    // s in [2^-60, 2^60]
};

__device__ __forceinline__ QScale make_qscale(const float* scale) {
    QScale q;
    q.s = __ldg(scale);
    q.fast = (q.s >= 0x1p-60f) && (q.s <= 0x1p60f);  // false for NaN, <= 0, inf, tiny
    q.r = q.fast ? __frcp_rn(q.s) : 1.0f;
    uint32_t tb = q.fast ? __float_as_uint(q.s * 131072.0f) : 0u;  // exact: s * 2^17
    tb = (tb + 0xFFFFu) & 0xFFFF0000u;                                 // round up to bf16
    q.t2 = (tb >> 16) | tb;
    return q;
}

template <bool FAST>
__device__ __forceinline__ float divide(float x, const QScale& c) {
    if (FAST) {
        float y0 = __fmul_rn(x, c.r);
        float e = __fmaf_rn(y0, c.s, -x);
        return __fmaf_rn(-e, c.r, y0);
    }
    return __fdiv_rn(x, c.s);
}

// Two bf16 (one 32-bit word, element 0 in the low half) -> two FP8 codes.
template <int FMT, bool FAST>
__device__ __forceinline__ uint32_t quant_pair(uint32_t w, const QScale& c) {
    if (FAST) w = bf16x2_clamp(w, c.t2);
    const float f0 = __uint_as_float(w << 16);
    const float f1 = __uint_as_float(w & 0xFFFF0000u);
    return cvt_fp8x2<FMT>(divide<FAST>(f0, c), divide<FAST>(f1, c));
}

// |x| bits of one bf16 (low half of w), as a binary32 bit pattern.
__device__ __forceinline__ uint32_t abs_bits_lo(uint32_t w) { return (w & 0x7FFFu) << 16; }

struct QTensor {
    const uint16_t* x;
    uint8_t* q;  // FP8 codes, or the bf16 output of the fused quantize -> dequantize
    const float* scale;
    float* amax;
    int64_t n;
    int64_t tile_end;  // exclusive end of this tensor's tiles in the global numbering
};

template <int MAXT>
struct QList {
    int64_t total_tiles;
    int32_t count;
    int32_t pad;
    QTensor t[MAXT];
};

struct QCursor {
    const uint16_t* x;
    uint8_t* q;
    float* amax;
    int64_t n, head, nvec, tile_begin;
    int mode;
    QScale c;
};

template <int OUT>
__device__ __forceinline__ QCursor make_cursor(const QTensor& t, int64_t tile_begin) {
    QCursor k;
    Split sp = split_tensor<typename GeomOf<OUT>::type>((uintptr_t)t.x, (uintptr_t)t.q, t.n);
    k.x = t.x;
    k.q = t.q;
    k.amax = t.amax;
    k.n = t.n;
    k.head = sp.head;
    k.nvec = sp.nvec;
    k.mode = sp.mode;
    k.tile_begin = tile_begin;
    k.c = make_qscale(t.scale);
    return k;
}

// CTA-wide max of the per-thread |x| bits, then one atomic into *amax.
// Every thread of the CTA must call it (it synchronises).
__device__ __forceinline__ void flush_amax(uint32_t m2, uint32_t ms, float* amax, uint32_t* red) {
    uint32_t m = max(max(abs_bits_lo(m2), m2 & 0x7FFF0000u), ms);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t b = red[0];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) b = max(b, red[w]);
        // |x| bit patterns order like the values (NaN above +inf); a signed
        // compare also lets any non-negative result beat a negative seed.
        atomicMax(reinterpret_cast<int*>(amax), (int)b);
    }
    __syncthreads();  // `red` is reused by the next flush
}

// Four bf16 (two words) -> four FP8 codes in one word.
template <int FMT, bool FAST>
__device__ __forceinline__ uint32_t quant_quad(uint32_t w0, uint32_t w1, const QScale& c) {
    return quant_pair<FMT, FAST>(w0, c) | (quant_pair<FMT, FAST>(w1, c) << 16);
}

// A tile's vectors, loaded before anything depends on the scale, so the loads
// and the scale's own load are in flight together.
template <int OUT>
struct TileRegs {
    uint4 a[GeomOf<OUT>::type::kVecPerThread], b[GeomOf<OUT>::type::kVecPerThread];
};

template <int OUT>
__device__ __forceinline__ void quant_vec_load(const QCursor& k, int64_t local, TileRegs<OUT>& r) {
    using G = typename GeomOf<OUT>::type;
    const uint16_t* xb = k.x + k.head;
    const int64_t v0 = local * Tile<G>::kVecs + threadIdx.x;
#pragma unroll
    for (int u = 0; u < G::kVecPerThread; ++u) {
        const int64_t v = v0 + (int64_t)u * kThreads;
        if (v < k.nvec) ld_stream_v8(xb + v * G::kVecElems, r.a[u], r.b[u]);
    }
}

template <int FMT, bool FAST, int OUT>
__device__ __forceinline__ void quant_vec_store(const QCursor& k, int64_t local, const TileRegs<OUT>& r,
                                                uint32_t& m2) {
    using G = typename GeomOf<OUT>::type;
    constexpr int E = G::kVecElems, U = G::kVecPerThread;
    uint8_t* qb = k.q + k.head;
    const int64_t v0 = local * Tile<G>::kVecs + threadIdx.x;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t v = v0 + (int64_t)u * kThreads;
        if (v < k.nvec) {
            const uint4& a = r.a[u];
            const uint4& b = r.b[u];
            m2 = bf16x2_absmax(m2, bf16x2_absmax(bf16x2_absmax(bf16x2_absmax(a.x, a.y), bf16x2_absmax(a.z, a.w)),
                                                 bf16x2_absmax(bf16x2_absmax(b.x, b.y), bf16x2_absmax(b.z, b.w))));
            uint4 o;
            o.x = quant_quad<FMT, FAST>(a.x, a.y, k.c);
            o.y = quant_quad<FMT, FAST>(a.z, a.w, k.c);
            o.z = quant_quad<FMT, FAST>(b.x, b.y, k.c);
            o.w = quant_quad<FMT, FAST>(b.z, b.w, k.c);
            if (OUT == kOutFp8) {
                st_v4(qb + v * E, o);
            } else {  // widen the fresh codes straight back: y = DQ(Q(x))
                uint16_t* yb = reinterpret_cast<uint16_t*>(k.q) + k.head + v * E;
                const float s = k.c.s;
                st_v4(yb, make_uint4(dequant_pair<FMT>(o.x & 0xFFFFu, s), dequant_pair<FMT>(o.x >> 16, s),
                                     dequant_pair<FMT>(o.y & 0xFFFFu, s), dequant_pair<FMT>(o.y >> 16, s)));
                st_v4(yb + 8, make_uint4(dequant_pair<FMT>(o.z & 0xFFFFu, s), dequant_pair<FMT>(o.z >> 16, s),
                                         dequant_pair<FMT>(o.w & 0xFFFFu, s), dequant_pair<FMT>(o.w >> 16, s)));
            }
        }
    }
}

template <int FMT, bool FAST, int OUT>
__device__ __forceinline__ void quant_scalar(const QCursor& k, int64_t i, uint32_t& ms) {
    const uint32_t w = k.x[i];
    ms = max(ms, abs_bits_lo(w));
    const uint32_t code = quant_pair<FMT, FAST>(w, k.c) & 0xFFu;
    if (OUT == kOutFp8)
        k.q[i] = (uint8_t)code;
    else
        reinterpret_cast<uint16_t*>(k.q)[i] = (uint16_t)(dequant_pair<FMT>(code, k.c.s) & 0xFFFFu);
}

template <int FMT, bool FAST, int OUT>
__device__ __forceinline__ void quant_scalars(const QCursor& k, int64_t local, uint32_t& ms) {
    using G = typename GeomOf<OUT>::type;
    if (k.mode == kModeVec) {
        if (local == 0) {  // scalar head and tail, each shorter than one vector
            const int64_t tail0 = k.head + k.nvec * G::kVecElems;
            const int64_t nscalar = k.head + (k.n - tail0);
            for (int64_t j = threadIdx.x; j < nscalar; j += kThreads)
                quant_scalar<FMT, FAST, OUT>(k, j < k.head ? j : tail0 + (j - k.head), ms);
        }
    } else {
        const int64_t base = local * Tile<G>::kElems;
        const int64_t end = min(base + (int64_t)Tile<G>::kElems, k.n);
        for (int64_t i = base + threadIdx.x; i < end; i += kThreads) quant_scalar<FMT, FAST, OUT>(k, i, ms);
    }
}

template <int FMT, int OUT>
__device__ __forceinline__ void quant_tile(const QCursor& k, int64_t local, uint32_t& m2, uint32_t& ms) {
    TileRegs<OUT> r;
    if (k.mode == kModeVec) quant_vec_load<OUT>(k, local, r);
    if (k.c.fast) {
        if (k.mode == kModeVec) quant_vec_store<FMT, true, OUT>(k, local, r, m2);
        quant_scalars<FMT, true, OUT>(k, local, ms);
    } else {
        if (k.mode == kModeVec) quant_vec_store<FMT, false, OUT>(k, local, r, m2);
        quant_scalars<FMT, false, OUT>(k, local, ms);
    }
}

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
// GELU producer fused with quantize + amax
//
// y = bf16(GELU(h)) with GELU(x) = x / (1 + exp(-2u)), u = sqrt(2/pi)(x +
// 0.044715 x^3) -- the tanh form -- then exactly the quantize above applied to
// y: FP8 codes of y / scale and amax = max|y|.  exp is evaluated by additive
// range reduction (Cody and Waite, "Software Manual for the Elementary
// Functions", 1980) and a degree-6 Taylor polynomial, every step one
// correctly rounded binary32 operation written out in a fixed order (no
// contraction, no approximate instruction), so the result is reproducible bit
// for bit on any IEEE machine.  Constants: binary32 roundings of ln 2 split in
// two (high part to 16 significant bits), 1/ln 2, -2 sqrt(2/pi), 0.044715, 1/k!.

// e^v on [-20, 89]: under -20, 1 + e^v is exactly 1 in binary32 whatever e^v
// is; above 88.73 the result overflows to +inf.  k = round(v / ln 2) comes
// from one fused multiply-add with 1.5 * 2^23 (whose sum's last bit is then
// the integer, read straight from the bits), r = v - k ln 2 in two parts, e^r
// by a degree-6 Taylor polynomial, then (e^r * 2^(k-1)) * 2.
__device__ __forceinline__ float exp_rr(float v) {
    v = fminf(fmaxf(v, -20.0f), 89.0f);  // fmaxf first: a NaN becomes -20
    const float t = __fmaf_rn(v, 0x1.715476p+0f, 0x1.8p23f);
    const float k = __fsub_rn(t, 0x1.8p23f);
    float r = __fmaf_rn(-k, 0x1.62e4p-1f, v);
    r = __fmaf_rn(-k, 0x1.7f7d1cp-20f, r);
    float p = 0x1.6c16c2p-10f;
    p = __fmaf_rn(p, r, 0x1.111112p-7f);
    p = __fmaf_rn(p, r, 0x1.555556p-5f);
    p = __fmaf_rn(p, r, 0x1.555556p-3f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int ki = __float_as_int(t) - __float_as_int(0x1.8p23f);  // k, in [-29, 128]
    return __fmul_rn(__fmul_rn(p, __int_as_float((ki + 126) << 23)), 2.0f);
}

__device__ __forceinline__ float gelu_rr(float x) {
    const float x2 = __fmul_rn(x, x);
    const float sx = __fmul_rn(x, __fmaf_rn(0x1.6e4e26p-5f, x2, 1.0f));  // x (1 + 0.044715 x^2)
    const float d = __fadd_rn(1.0f, exp_rr(__fmul_rn(-0x1.988454p+0f, sx)));
    const float g = __fmul_rn(x, __frcp_rn(d));
    return x == -INFINITY ? -0.0f : g;  // the limit (x * 0 would be NaN); NaN stays NaN
}

// Two bf16 (one word) -> two bf16 of GELU (one word).
__device__ __forceinline__ uint32_t gelu_pair(uint32_t w) {
    return cvt_bf16x2(gelu_rr(__uint_as_float(w << 16)), gelu_rr(__uint_as_float(w & 0xFFFF0000u)));
}

struct GeluGeom {
    static constexpr int kVecElems = 16;  // 16 bf16 in (32 bytes) -> 16 codes (+ 16 bf16 of y)
    static constexpr int kVecPerThread = 2;
    static constexpr int kWideAlign = 32;
    static constexpr int kNarrowBytes = 1;
    static constexpr int kNarrowAlign = 16;
};

struct GeluArgs {
    const uint16_t* h;
    uint16_t* y;  // may be null
    uint8_t* q;
    const float* scale;
    float* amax;
    int64_t n, head, nvec, tiles;
    int mode;
};

template <int FMT, bool FAST, bool WRITE_Y>
__device__ __forceinline__ void gelu_vec_store(const GeluArgs& a, const QScale& c, int64_t v, const uint4& wa,
                                               const uint4& wb, uint32_t& m2) {
    constexpr int E = GeluGeom::kVecElems;
    uint4 ya, yb;
    ya.x = gelu_pair(wa.x); ya.y = gelu_pair(wa.y); ya.z = gelu_pair(wa.z); ya.w = gelu_pair(wa.w);
    yb.x = gelu_pair(wb.x); yb.y = gelu_pair(wb.y); yb.z = gelu_pair(wb.z); yb.w = gelu_pair(wb.w);
    if (WRITE_Y) {
        uint16_t* yp = a.y + a.head + v * E;
        st_v4(yp, ya);
        st_v4(yp + 8, yb);
    }
    m2 = bf16x2_absmax(m2, bf16x2_absmax(bf16x2_absmax(bf16x2_absmax(ya.x, ya.y), bf16x2_absmax(ya.z, ya.w)),
                                         bf16x2_absmax(bf16x2_absmax(yb.x, yb.y), bf16x2_absmax(yb.z, yb.w))));
    uint4 o;
    o.x = quant_quad<FMT, FAST>(ya.x, ya.y, c);
    o.y = quant_quad<FMT, FAST>(ya.z, ya.w, c);
    o.z = quant_quad<FMT, FAST>(yb.x, yb.y, c);
    o.w = quant_quad<FMT, FAST>(yb.z, yb.w, c);
    st_v4(a.q + a.head + v * E, o);
}

template <int FMT, bool FAST, bool WRITE_Y>
__device__ __forceinline__ void gelu_scalar(const GeluArgs& a, const QScale& c, int64_t i, uint32_t& ms) {
    const uint32_t yw = gelu_pair(a.h[i]) & 0xFFFFu;
    if (WRITE_Y) a.y[i] = (uint16_t)yw;
    ms = max(ms, abs_bits_lo(yw));
    a.q[i] = (uint8_t)(quant_pair<FMT, FAST>(yw, c) & 0xFFu);
}

template <int FMT, bool FAST, bool WRITE_Y>
__device__ __forceinline__ void gelu_tile(const GeluArgs& a, const QScale& c, int64_t tile, const uint4* wa,
                                          const uint4* wb, uint32_t& m2, uint32_t& ms) {
    constexpr int E = GeluGeom::kVecElems, U = GeluGeom::kVecPerThread;
    if (a.mode == kModeVec) {
        const int64_t v0 = tile * Tile<GeluGeom>::kVecs + threadIdx.x;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = v0 + (int64_t)u * kThreads;
            if (v < a.nvec) gelu_vec_store<FMT, FAST, WRITE_Y>(a, c, v, wa[u], wb[u], m2);
        }
        if (tile == 0) {
            const int64_t tail0 = a.head + a.nvec * E;
            const int64_t nscalar = a.head + (a.n - tail0);
            for (int64_t j = threadIdx.x; j < nscalar; j += kThreads)
                gelu_scalar<FMT, FAST, WRITE_Y>(a, c, j < a.head ? j : tail0 + (j - a.head), ms);
        }
    } else {
        const int64_t base = tile * Tile<GeluGeom>::kElems;
        const int64_t end = min(base + (int64_t)Tile<GeluGeom>::kElems, a.n);
        for (int64_t i = base + threadIdx.x; i < end; i += kThreads) gelu_scalar<FMT, FAST, WRITE_Y>(a, c, i, ms);
    }
}

template <int FMT, bool WRITE_Y>
__global__ void __launch_bounds__(kThreads) gelu_quantize_amax_kernel(const GeluArgs a) {
    __shared__ uint32_t red[kThreads / 32];
    constexpr int E = GeluGeom::kVecElems, U = GeluGeom::kVecPerThread;
    uint32_t m2 = 0, ms = 0;
    QScale c;
    bool have_scale = false;
    for (int64_t tile = blockIdx.x; tile < a.tiles; tile += gridDim.x) {
        uint4 wa[U], wb[U];
        if (a.mode == kModeVec) {  // loads first: nothing here waits on the scale
            const int64_t v0 = tile * Tile<GeluGeom>::kVecs + threadIdx.x;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + (int64_t)u * kThreads;
                if (v < a.nvec) ld_stream_v8(a.h + a.head + v * E, wa[u], wb[u]);
            }
        }
        if (!have_scale) {
            c = make_qscale(a.scale);
            have_scale = true;
        }
        if (c.fast) gelu_tile<FMT, true, WRITE_Y>(a, c, tile, wa, wb, m2, ms);
        else        gelu_tile<FMT, false, WRITE_Y>(a, c, tile, wa, wb, m2, ms);
    }
    flush_amax(m2, ms, a.amax, red);
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

bool valid_fmt(int fmt) { return fmt == FP8Q_E4M3FN || fmt == FP8Q_E5M2; }

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
    quantize_amax_kernel<FMT, MAXT, OUT><<<grid, kThreads, 0, stream>>>(L);
    return after_launch("quantize_amax_kernel");
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

fp8q_status check_tensor(const fp8q_tensor& t) {
    if (t.n < 0) return FP8Q_ERR_INVALID_ARG;
    if (t.n == 0) return FP8Q_OK;
    if (!t.x_bf16 || !t.q || !t.scale || !t.amax) return FP8Q_ERR_INVALID_ARG;
    if (((uintptr_t)t.x_bf16 & 1u) || ((uintptr_t)t.scale & 3u) || ((uintptr_t)t.amax & 3u))
        return FP8Q_ERR_INVALID_ARG;
    return FP8Q_OK;
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
    dequantize_kernel<FMT><<<grid, kThreads, 0, stream>>>(q, static_cast<uint16_t*>(y), n, scale, sp.tiles);
    return after_launch("dequantize_kernel");
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
    return fmt == FP8Q_E4M3FN ? launch_quantize<FP8Q_E4M3FN, 1>(&t, 1, s)
                              : launch_quantize<FP8Q_E5M2, 1>(&t, 1, s);
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

fp8q_status fp8q_gelu_quantize_amax(const void* h_bf16, void* y_bf16, uint8_t* q, int64_t n,
                                    fp8q_format fmt, const float* scale, float* amax, void* stream) {
    if (!valid_fmt(fmt)) return FP8Q_ERR_INVALID_ARG;
    const fp8q_tensor t = {h_bf16, q, n, scale, amax};
    fp8q_status st = check_tensor(t);
    if (st != FP8Q_OK || n == 0) return st;
    if ((uintptr_t)y_bf16 & 1u) return FP8Q_ERR_INVALID_ARG;
    Split sp = split_tensor<GeluGeom>((uintptr_t)h_bf16, (uintptr_t)q, n);
    // the bf16 output rides the vector path only if it is aligned like the input
    if (y_bf16 && sp.mode == kModeVec && (((uintptr_t)y_bf16 - (uintptr_t)h_bf16) & 31u) != 0) {
        sp.mode = kModeScalar;
        sp.head = n;
        sp.nvec = 0;
        sp.tiles = (n + Tile<GeluGeom>::kElems - 1) / Tile<GeluGeom>::kElems;
    }
    GeluArgs a;
    a.h = static_cast<const uint16_t*>(h_bf16);
    a.y = static_cast<uint16_t*>(y_bf16);
    a.q = q;
    a.scale = scale;
    a.amax = amax;
    a.n = n;
    a.head = sp.head;
    a.nvec = sp.nvec;
    a.tiles = sp.tiles;
    a.mode = sp.mode;
    const int grid = (int)(sp.tiles < 0x7FFFFFFF ? sp.tiles : 0x7FFFFFFF);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fmt == FP8Q_E4M3FN) {
        if (y_bf16) gelu_quantize_amax_kernel<FP8Q_E4M3FN, true><<<grid, kThreads, 0, s>>>(a);
        else        gelu_quantize_amax_kernel<FP8Q_E4M3FN, false><<<grid, kThreads, 0, s>>>(a);
    } else {
        if (y_bf16) gelu_quantize_amax_kernel<FP8Q_E5M2, true><<<grid, kThreads, 0, s>>>(a);
        else        gelu_quantize_amax_kernel<FP8Q_E5M2, false><<<grid, kThreads, 0, s>>>(a);
    }
    return after_launch("gelu_quantize_amax_kernel");
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

const char* fp8q_status_string(fp8q_status status) {
    switch (status) {
        case FP8Q_OK: return "FP8Q_OK";
        case FP8Q_ERR_INVALID_ARG: return "FP8Q_ERR_INVALID_ARG";
        case FP8Q_ERR_UNSUPPORTED: return "FP8Q_ERR_UNSUPPORTED";
        case FP8Q_ERR_CUDA: return "FP8Q_ERR_CUDA";
        case FP8Q_ERR_TOO_MANY_TENSORS: return "FP8Q_ERR_TOO_MANY_TENSORS";
    }
    return "FP8Q_ERR_UNKNOWN";
}

const char* fp8q_last_cuda_error(void) { return g_last_error; }

}  // extern "C"
