// fp8q_common.cuh -- what the kernels of libfp8q share: launch geometry,
// bf16/FP8 conversions, the exact division by the scale, the CTA-wide amax
// flush, and host-side error reporting.  The kernels and their C ABI entry
// points live in quantize.cu, producers.cu and scale_update.cu; abi.cu holds
// the status strings.
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
//   * the LayerNorm producer is a persistent kernel that stages whole rows in
//     shared memory with cp.async.bulk; its waits on those copies' mbarriers
//     give up after one second (the result is then marked, never left
//     hanging).  No kernel waits on another CTA or on a flag; every other wait
//     is a __syncthreads in uniform control flow.

#pragma once

#include "fp8q.h"

#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstdio>

// Host-side error reporting, shared by every translation unit (abi.cu).
namespace fp8q_detail {
fp8q_status cuda_fail(cudaError_t e, const char* where);   // records the text, returns FP8Q_ERR_CUDA
extern thread_local char g_last_error[256];

// Launch `kern` on `s` and report that launch's own status.  A runtime error
// that an earlier, unrelated call left pending is neither reported nor
// cleared here: only a failure of this launch becomes FP8Q_ERR_CUDA.
template <typename... KArgs, typename... Args>
fp8q_status launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          const char* where, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
    return e == cudaSuccess ? FP8Q_OK : cuda_fail(e, where);
}

inline bool valid_fmt(int fmt) { return fmt == FP8Q_E4M3FN || fmt == FP8Q_E5M2; }

// Arguments every bf16 -> FP8 tensor entry point shares.
inline fp8q_status check_tensor(const fp8q_tensor& t) {
    if (t.n < 0) return FP8Q_ERR_INVALID_ARG;
    if (t.n == 0) return FP8Q_OK;
    if (!t.x_bf16 || !t.q || !t.scale || !t.amax) return FP8Q_ERR_INVALID_ARG;
    if (((uintptr_t)t.x_bf16 & 1u) || ((uintptr_t)t.scale & 3u) || ((uintptr_t)t.amax & 3u))
        return FP8Q_ERR_INVALID_ARG;
    return FP8Q_OK;
}
}  // namespace fp8q_detail

namespace {

using namespace fp8q_detail;

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
// Dequantize: tiles of 4096 elements (two 8-element vectors per thread).  On
// 8192x16384 (means of 40 launches) 60.7 us back to back and 61.8-62.0 after a
// 268 MB copy, against 61.4-61.5 and 62.3 with four vectors per thread and
// 61.7 and 63.6-63.8 with eight; from a clean L2 all three within 1%.
struct DequantGeom {
    static constexpr int kVecElems = 8;
    static constexpr int kVecPerThread = 2;
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

__device__ __forceinline__ QScale make_qscale_value(float s) {
    QScale q;
    q.s = s;
    q.fast = (q.s >= 0x1p-60f) && (q.s <= 0x1p60f);  // false for NaN, <= 0, inf, tiny
    q.r = q.fast ? __frcp_rn(q.s) : 1.0f;
    uint32_t tb = q.fast ? __float_as_uint(q.s * 131072.0f) : 0u;  // exact: s * 2^17
    tb = (tb + 0xFFFFu) & 0xFFFF0000u;                                 // round up to bf16
    q.t2 = (tb >> 16) | tb;
    return q;
}

__device__ __forceinline__ QScale make_qscale(const float* scale) { return make_qscale_value(__ldg(scale)); }

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

// A cursor whose scale constants are given (t.scale is not read).
template <int OUT>
__device__ __forceinline__ QCursor make_cursor_with(const QTensor& t, int64_t tile_begin, const QScale& c) {
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
    k.c = c;
    return k;
}

template <int OUT>
__device__ __forceinline__ QCursor make_cursor(const QTensor& t, int64_t tile_begin) {
    return make_cursor_with<OUT>(t, tile_begin, make_qscale(t.scale));
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

}  // namespace
