// quant_tile.cuh -- one tile of the quantize (and of the fused quantize ->
// dequantize): vector loads, conversion and stores, plus the scalar head and
// tail.  Shared by the quantize kernels and the update fused with a quantize.

#pragma once

#include "fp8q_common.cuh"

namespace {

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

// Vector v of the tensor (16 bf16 in a and b): |x| into m2, the 16 codes out
// (or, for the fused quantize -> dequantize, their bf16 values).
template <int FMT, bool FAST, int OUT>
__device__ __forceinline__ void quant_vec1(const QCursor& k, int64_t v, const uint4& a, const uint4& b, uint32_t& m2) {
    constexpr int E = GeomOf<OUT>::type::kVecElems;
    m2 = bf16x2_absmax(m2, bf16x2_absmax(bf16x2_absmax(bf16x2_absmax(a.x, a.y), bf16x2_absmax(a.z, a.w)),
                                         bf16x2_absmax(bf16x2_absmax(b.x, b.y), bf16x2_absmax(b.z, b.w))));
    uint4 o;
    o.x = quant_quad<FMT, FAST>(a.x, a.y, k.c);
    o.y = quant_quad<FMT, FAST>(a.z, a.w, k.c);
    o.z = quant_quad<FMT, FAST>(b.x, b.y, k.c);
    o.w = quant_quad<FMT, FAST>(b.z, b.w, k.c);
    if (OUT == kOutFp8) {
        st_v4(k.q + k.head + v * E, o);
    } else {  // widen the fresh codes straight back: y = DQ(Q(x))
        uint16_t* yb = reinterpret_cast<uint16_t*>(k.q) + k.head + v * E;
        const float s = k.c.s;
        st_v4(yb, make_uint4(dequant_pair<FMT>(o.x & 0xFFFFu, s), dequant_pair<FMT>(o.x >> 16, s),
                             dequant_pair<FMT>(o.y & 0xFFFFu, s), dequant_pair<FMT>(o.y >> 16, s)));
        st_v4(yb + 8, make_uint4(dequant_pair<FMT>(o.z & 0xFFFFu, s), dequant_pair<FMT>(o.z >> 16, s),
                                 dequant_pair<FMT>(o.w & 0xFFFFu, s), dequant_pair<FMT>(o.w >> 16, s)));
    }
}

template <int FMT, bool FAST, int OUT>
__device__ __forceinline__ void quant_vec_store(const QCursor& k, int64_t local, const TileRegs<OUT>& r,
                                                uint32_t& m2) {
    using G = typename GeomOf<OUT>::type;
    constexpr int U = G::kVecPerThread;
    const int64_t v0 = local * Tile<G>::kVecs + threadIdx.x;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t v = v0 + (int64_t)u * kThreads;
        if (v < k.nvec) quant_vec1<FMT, FAST, OUT>(k, v, r.a[u], r.b[u], m2);
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

}  // namespace
