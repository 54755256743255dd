// producers.cu -- the producers fused with quantize + amax:
// GELU (elementwise) and LayerNorm (row-wise).

#include "fp8q_common.cuh"
#include "mbarrier.cuh"
#include "packed_f32.cuh"

#include <mutex>


namespace {

// quant_pair's fast path, two lanes at a time: y0 = RN(x r), e = fma(y0, s, -x),
// y = fma(-e, r, y0) is the correctly rounded quotient in each lane.
template <int FMT>
__device__ __forceinline__ uint32_t quant_pair_x2(uint32_t w, const QScale& c) {
    w = bf16x2_clamp(w, c.t2);
    const float2 x = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    const float2 y0 = mul2_rn(x, splat2(c.r));
    const float2 e = fma2_rn(y0, splat2(c.s), make_float2(-x.x, -x.y));
    const float2 y = fma2_rn(make_float2(-e.x, -e.y), splat2(c.r), y0);
    return cvt_fp8x2<FMT>(y.x, y.y);
}

// Four bf16 (two words) -> four FP8 codes in one word; the fast path two lanes
// at a time.
template <int FMT, bool FAST>
__device__ __forceinline__ uint32_t quant_quad_x2(uint32_t w0, uint32_t w1, const QScale& c) {
    if (FAST) return quant_pair_x2<FMT>(w0, c) | (quant_pair_x2<FMT>(w1, c) << 16);
    return quant_quad<FMT, false>(w0, w1, c);
}

// Eight bf16 of y -> eight FP8 codes.
template <int FMT, bool FAST>
__device__ __forceinline__ uint2 quant8(const uint4& y, const QScale& c) {
    return make_uint2(quant_quad_x2<FMT, FAST>(y.x, y.y, c), quant_quad_x2<FMT, FAST>(y.z, y.w, c));
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

// e^v on [-20, 89], two lanes at a time: under -20, 1 + e^v is exactly 1 in
// binary32 whatever e^v is; above 88.73 the result overflows to +inf.
// k = round(v / ln 2) comes from one fused multiply-add with 1.5 * 2^23 (whose
// sum's last bit is then the integer, read straight from the bits),
// r = v - k ln 2 in two parts (fma(k, -c, v) is fma(-k, c, v) exactly), e^r by
// a degree-6 Taylor polynomial, then (e^r * 2^(k-1)) * 2.  Every two-lane
// operation rounds each lane exactly like its scalar form; the one multiply
// whose result is then added (by 2, before 1 + e) is exact, so no fusion can
// change a bit.
__device__ __forceinline__ float2 exp2_rr(float2 v) {
    v.x = fminf(fmaxf(v.x, -20.0f), 89.0f);  // fmaxf first: a NaN becomes -20
    v.y = fminf(fmaxf(v.y, -20.0f), 89.0f);
    const float2 t = fma2_rn(v, splat2(0x1.715476p+0f), splat2(0x1.8p23f));
    const float2 k = add2_rn(t, splat2(-0x1.8p23f));
    float2 r = fma2_rn(k, splat2(-0x1.62e4p-1f), v);
    r = fma2_rn(k, splat2(-0x1.7f7d1cp-20f), r);
    float2 p = fma2_rn(splat2(0x1.6c16c2p-10f), r, splat2(0x1.111112p-7f));
    p = fma2_rn(p, r, splat2(0x1.555556p-5f));
    p = fma2_rn(p, r, splat2(0x1.555556p-3f));
    p = fma2_rn(p, r, splat2(0.5f));
    p = fma2_rn(p, r, splat2(1.0f));
    p = fma2_rn(p, r, splat2(1.0f));
    // 2^(k-1) from the bits of t: k = bits(t) - bits(1.5 * 2^23), in [-29, 128], and
    // ((k + 126) << 23) = bits(t) * 2^23 + (126 - bits(1.5 * 2^23)) * 2^23 (mod 2^32)
    constexpr uint32_t kScaleBias = (126u - 0x4B400000u) << 23;
    const float2 s = make_float2(__uint_as_float(__float_as_uint(t.x) * (1u << 23) + kScaleBias),
                                 __uint_as_float(__float_as_uint(t.y) * (1u << 23) + kScaleBias));
    return mul2_rn(mul2_rn(p, s), splat2(2.0f));
}

__device__ __forceinline__ float max_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// Two bf16 (one word) -> two bf16 of GELU (one word).
__device__ __forceinline__ uint32_t gelu_pair(uint32_t w) {
    const float2 x = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    const float2 x2 = mul2_rn(x, x);
    const float2 sx = mul2_rn(x, fma2_rn(splat2(0x1.6e4e26p-5f), x2, splat2(1.0f)));  // x (1 + 0.044715 x^2)
    const float2 d = add2_rn(splat2(1.0f), exp2_rr(mul2_rn(splat2(-0x1.988454p+0f), sx)));
    // x * (1 / d) with d >= 1.  GELU(-inf) is the limit -0: there d = inf and 1/d = 0,
    // so x is first raised to -FLT_MAX (-FLT_MAX * 0 = -0); max.NaN keeps a NaN.
    const float2 g = mul2_rn(make_float2(max_nan(x.x, -0x1.fffffep127f), max_nan(x.y, -0x1.fffffep127f)),
                             rcp2_rn(d));
    return cvt_bf16x2(g.x, g.y);
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

// The 16 results y of vector v: store y (optional), fold |y| into m2, store
// their FP8 codes.
template <int FMT, bool FAST, bool WRITE_Y>
__device__ __forceinline__ void gelu_emit(const GeluArgs& a, const QScale& c, int64_t v, const uint4& ya,
                                          const uint4& yb, uint32_t& m2) {
    constexpr int E = GeluGeom::kVecElems;
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
__device__ __forceinline__ void gelu_vec_store(const GeluArgs& a, const QScale& c, int64_t v, const uint4& wa,
                                               const uint4& wb, uint32_t& m2) {
    uint4 ya, yb;
    ya.x = gelu_pair(wa.x); ya.y = gelu_pair(wa.y); ya.z = gelu_pair(wa.z); ya.w = gelu_pair(wa.w);
    yb.x = gelu_pair(wb.x); yb.y = gelu_pair(wb.y); yb.z = gelu_pair(wb.z); yb.w = gelu_pair(wb.w);
    gelu_emit<FMT, FAST, WRITE_Y>(a, c, v, ya, yb, m2);
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

// At most 64 registers, so four CTAs share an SM: the exp chain is long, and
// the extra warps hide its latency (measured on 8192x16384 while the kernel
// still used the IEEE reciprocal: 155 us against 175 us with three).
template <int FMT, bool WRITE_Y>
__global__ void __launch_bounds__(kThreads, 4) gelu_quantize_amax_kernel(const GeluArgs a) {
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
// GELU through a table of every bf16 input
//
// y = bf16(GELU(h)), and so its FP8 code at a given scale, depends only on the
// 16 bits of h.  For large tensors each CTA first gets a table over all 65536
// inputs into shared memory; the CTAs of a thread-block cluster compute it
// once between them, every y with gelu_pair -- the arithmetic of the kernel
// above, so the same bits.  The CTA then streams its share of the tensor with
// shared-memory lookups in place of the GELU arithmetic:
//  - with y, the table holds y (128 KB) and each y is then quantized as above;
//  - for the codes alone it holds the FP8 code of every input at this launch's
//    scale (64 KB, each quantized once), so an element costs one byte lookup
//    (or, for one element in eight, the arithmetic), and amax comes from the
//    largest input (gelu_code_table_kernel).
// One CTA per SM, looping over the vectors two at a time, with the next two
// already loading while the current two are looked up, so that enough loads
// are in flight; the first two go out before the table is built.  Building
// the table costs each cluster about what 65536 elements cost the direct
// kernel, so smaller tensors, and any that take the element-by-element path,
// use the direct kernel.

// Threads per CTA: 1024 for the codes alone; 512 when y is stored too (its
// extra registers would spill at 1024).
constexpr int kGeluYTableThreads = 512;
constexpr int kGeluCodeTableThreads = 1024;
constexpr uint32_t kGeluYTableBytes = 65536u * 2u;
constexpr uint32_t kGeluCodeTableBytes = 65536u;
// Fewer elements take the direct kernel.  Measured on GB300 from a cold L2
// (direct / table, us): codes alone 12.7 / 12.7 at 2^22 elements, 16.8 / 14.8
// at 2^23, 25.3 / 19.2 at 2^24; with y 25.3 / 27.4 at 2^24, 41.7 / 39.7 at 2^25.
#ifdef FP8Q_TEST_GELU_TABLE_MIN_ELEMS  // test-only build: small tensors take the table path too
constexpr int64_t kGeluTableMinElems = FP8Q_TEST_GELU_TABLE_MIN_ELEMS;
constexpr int64_t kGeluTableMinElemsWithY = FP8Q_TEST_GELU_TABLE_MIN_ELEMS;
#else
constexpr int64_t kGeluTableMinElems = (int64_t)1 << 23;
constexpr int64_t kGeluTableMinElemsWithY = (int64_t)1 << 25;
#endif
// Vectors in flight per thread, two beyond the two being converted (with y,
// three or four measured 125-127 us on 8192x16384, against 113).
constexpr int kGeluTableUnroll = 2;
constexpr int kGeluYUnroll = 2;
// CTAs of one thread-block cluster (on as many SMs) build their tables
// together: each computes its share of the entries and stores each into the
// shared memory of every CTA of the cluster.  Larger clusters build faster
// but leave more SMs idle (the clusters that fit at once cover fewer SMs).
// Measured on GB300: with y (512 threads), clusters of 8 below 2^26 elements
// (cold L2, 2^25: 37.7 us, against 39.7 with 2 or 4), clusters of 4 from there
// (8192x16384 back to back: 112.0 us, against 114.6 with 2 and 113.3 with 8).
// Codes alone (1024 threads): clusters of 8 below 2^25 elements (cold L2: 14.8
// us at 2^23 and 18.9 at 2^24, against 16.9 and 21.1-21.2 with 2 or 4),
// clusters of 4 from there (back to back: 22.7, 38.7 and 65.6 us at 2^25,
// 2^26 and 2^27, against 24.7, 37.4 and 67.0 with 2).
constexpr int kGeluYTableClusterSmall = 8;
constexpr int kGeluYTableCluster = 4;
constexpr int64_t kGeluYTableSmallBelow = (int64_t)1 << 26;
constexpr int kGeluCodeTableClusterSmall = 8;
constexpr int kGeluCodeTableCluster = 4;
constexpr int64_t kGeluCodeTableSmallBelow = (int64_t)1 << 25;

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of the same shared-memory location in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t cta_addr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(cta_addr), "r"(rank));
    return d;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// The split cluster barrier: every thread of every CTA of the cluster arrives
// (relaxed: no memory ordering), and a later wait returns once all have
// arrived -- in particular once every CTA of the cluster is running.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// Every thread of every CTA of the cluster arrives; the stores made before
// are visible to all of them afterwards.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Fill the table of every CTA of the cluster: word p of kWords is entry(p).
// CTA rank r computes the words of its share, [r kWords / C, (r + 1) kWords / C),
// and stores each into the same place in every CTA of the cluster.  No CTA may
// touch another's shared memory before that CTA is known to be running: each
// arrives on the cluster barrier at entry and waits on it just before its
// first remote store, with its first word computed in between.  The caller
// then makes every table complete with cluster_sync_all.
template <int kCtaThreads, int kCluster, int kWords, typename Entry>
__device__ __forceinline__ void cluster_build(uint32_t* tab32, Entry entry) {
    constexpr int kShare = kWords / kCluster;
    static_assert(kShare % kCtaThreads == 0, "every thread computes the same number of words");
    cluster_arrive_relaxed();
    const uint32_t rank = cluster_ctarank();
    uint32_t dst[kCluster];
#pragma unroll
    for (int r = 0; r < kCluster; ++r) dst[r] = cluster_map(smem_addr(tab32), (uint32_t)r);
    int p = (int)rank * kShare + threadIdx.x;
    uint32_t v = entry(p);
    cluster_wait();
    for (;;) {
#pragma unroll
        for (int r = 0; r < kCluster; ++r) st_cluster_u32(dst[r] + 4u * (uint32_t)p, v);
        p += kCtaThreads;
        if (p >= ((int)rank + 1) * kShare) break;
        v = entry(p);
    }
}

// The next U vectors of 16 bf16 of a thread that visits v, v + stride, ...
template <int U>
__device__ __forceinline__ void gelu_load(const GeluArgs& a, int64_t v, int64_t stride, uint4 (&wa)[U],
                                          uint4 (&wb)[U]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t vu = v + u * stride;
        if (vu < a.nvec) ld_stream_v8(a.h + a.head + vu * GeluGeom::kVecElems, wa[u], wb[u]);
    }
}

__device__ __forceinline__ uint32_t gelu_lookup_pair(const uint16_t* tab, uint32_t w) {
    return (uint32_t)tab[w & 0xFFFFu] | ((uint32_t)tab[w >> 16] << 16);
}

__device__ __forceinline__ uint4 gelu_lookup4(const uint16_t* tab, const uint4& w) {
    return make_uint4(gelu_lookup_pair(tab, w.x), gelu_lookup_pair(tab, w.y), gelu_lookup_pair(tab, w.z),
                      gelu_lookup_pair(tab, w.w));
}

template <int FMT, int CLUSTER>
__global__ void __launch_bounds__(kGeluYTableThreads, 1) gelu_table_quantize_amax_kernel(const GeluArgs a) {
    extern __shared__ __align__(16) uint32_t tab32[];  // word p: the y of inputs 2p and 2p + 1
    __shared__ uint32_t red[kGeluYTableThreads / 32];
    constexpr int E = GeluGeom::kVecElems;
    const int64_t stride = (int64_t)gridDim.x * kGeluYTableThreads;
    uint32_t m2 = 0, ms = 0;
    int64_t v0 = (int64_t)blockIdx.x * kGeluYTableThreads + threadIdx.x;
    uint4 wa[kGeluYUnroll], wb[kGeluYUnroll];
    gelu_load(a, v0, stride, wa, wb);  // before the build, which hides their latency
    cluster_build<kGeluYTableThreads, CLUSTER, 32768>(
        tab32, [](int p) { return gelu_pair((uint32_t)(2 * p) | ((uint32_t)(2 * p + 1) << 16)); });
    const QScale c = make_qscale(a.scale);
    cluster_sync_all();  // every CTA's table is complete; no remote store comes after this
    const uint16_t* tab = reinterpret_cast<const uint16_t*>(tab32);
    for (; v0 < a.nvec; v0 += kGeluYUnroll * stride) {
        uint4 na[kGeluYUnroll], nb[kGeluYUnroll];
        gelu_load(a, v0 + kGeluYUnroll * stride, stride, na, nb);
#pragma unroll
        for (int u = 0; u < kGeluYUnroll; ++u) {
            const int64_t v = v0 + u * stride;
            if (v < a.nvec) {
                const uint4 ya = gelu_lookup4(tab, wa[u]), yb = gelu_lookup4(tab, wb[u]);
                if (c.fast) gelu_emit<FMT, true, true>(a, c, v, ya, yb, m2);
                else        gelu_emit<FMT, false, true>(a, c, v, ya, yb, m2);
            }
        }
#pragma unroll
        for (int u = 0; u < kGeluYUnroll; ++u) {
            wa[u] = na[u];
            wb[u] = nb[u];
        }
    }
    if (blockIdx.x == 0) {  // scalar head and tail, each shorter than one vector
        const int64_t tail0 = a.head + a.nvec * E;
        const int64_t nscalar = a.head + (a.n - tail0);
        for (int64_t j = threadIdx.x; j < nscalar; j += kGeluYTableThreads) {
            const int64_t i = j < a.head ? j : tail0 + (j - a.head);
            const uint32_t yw = tab[a.h[i]];
            a.y[i] = (uint16_t)yw;
            ms = max(ms, abs_bits_lo(yw));
            a.q[i] = (uint8_t)((c.fast ? quant_pair<FMT, true>(yw, c) : quant_pair<FMT, false>(yw, c)) & 0xFFu);
        }
    }
    // CTA-wide max of |y|, one atomic
    uint32_t m = max(max(abs_bits_lo(m2), m2 & 0x7FFF0000u), ms);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t b = red[0];
        for (int w = 1; w < kGeluYTableThreads / 32; ++w) b = max(b, red[w]);
        atomicMax(reinterpret_cast<int*>(a.amax), (int)b);
    }
}

// max(a, b) per bf16 lane by value (-0 and +0 either way); a NaN in either
// gives the canonical NaN.
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// The FP8 codes of four inputs (two words) from the code table, in order.
__device__ __forceinline__ uint32_t code_lookup4(const uint8_t* tab, uint32_t w0, uint32_t w1) {
    return (uint32_t)tab[w0 & 0xFFFFu] | ((uint32_t)tab[w0 >> 16] << 8) | ((uint32_t)tab[w1 & 0xFFFFu] << 16) |
           ((uint32_t)tab[w1 >> 16] << 24);
}

__device__ __forceinline__ uint32_t max8(uint32_t m, const uint4& a, const uint4& b) {
    return bf16x2_max(m, bf16x2_max(bf16x2_max(bf16x2_max(a.x, a.y), bf16x2_max(a.z, a.w)),
                                    bf16x2_max(bf16x2_max(b.x, b.y), bf16x2_max(b.z, b.w))));
}

// The codes of the thread's vectors v_first, v_first + stride, ... (the first
// two already loading in wa, wb), and the largest input into hm2.  The lookups
// keep the shared-memory pipe the busiest unit of the SM (a warp's 32 random
// byte lookups cost about 3.3 bank wavefronts), while instruction issue has
// room: so the first two elements of every vector are computed (gelu_pair and
// the quantize, the same bits as their table entries) and the other 14 looked
// up.  Measured on GB300 (8192x16384, CUDA events): 69.5 us, against 70.0-70.6
// with every element looked up and 69.7-70.0 with four of 16 computed.
template <int FMT, bool FAST>
__device__ __forceinline__ void code_table_stream(const GeluArgs& a, const uint8_t* tab, const QScale& c,
                                                  int64_t v_first, int64_t stride, uint4 (&wa)[2], uint4 (&wb)[2],
                                                  uint32_t& hm2) {
    constexpr int E = GeluGeom::kVecElems;
    for (int64_t v0 = v_first; v0 < a.nvec; v0 += kGeluTableUnroll * stride) {
        uint4 na[kGeluTableUnroll], nb[kGeluTableUnroll];
        gelu_load(a, v0 + kGeluTableUnroll * stride, stride, na, nb);
#pragma unroll
        for (int u = 0; u < kGeluTableUnroll; ++u) {
            const int64_t v = v0 + u * stride;
            if (v < a.nvec) {
                hm2 = max8(hm2, wa[u], wb[u]);
                // the first two elements computed, the other 14 looked up
                const uint32_t o0 = quant_pair<FMT, FAST>(gelu_pair(wa[u].x), c) |
                                    ((uint32_t)tab[wa[u].y & 0xFFFFu] << 16) | ((uint32_t)tab[wa[u].y >> 16] << 24);
                st_v4(a.q + a.head + v * E, make_uint4(o0, code_lookup4(tab, wa[u].z, wa[u].w),
                                                       code_lookup4(tab, wb[u].x, wb[u].y),
                                                       code_lookup4(tab, wb[u].z, wb[u].w)));
            }
        }
#pragma unroll
        for (int u = 0; u < kGeluTableUnroll; ++u) {
            wa[u] = na[u];
            wb[u] = nb[u];
        }
    }
}

// |y| of the low bf16 of w as a binary32 bit pattern, every NaN canonical.
__device__ __forceinline__ uint32_t gelu_abs_bits(uint32_t w) { return abs_bits_lo(bf16x2_absmax(gelu_pair(w), 0u)); }

// Every negative input (and -0, -inf) gives |y| below 0.1875 (bf16 0x3E40):
// the tanh-form GELU is smallest near x = -0.75, where it is about -0.170.
constexpr uint32_t kGeluNegativeBound = 0x3E400000u;

// Codes alone through a table of the FP8 code of every input (64 KB).
//
// amax = max|y| over the tensor without any y: the computed y is
// non-decreasing in h from +0 to +inf (and not below 0 there), and every
// negative input gives |y| below 0.1875 -- both hold for every bf16 input,
// and the tests check them.  So when the largest input hm a thread has seen
// is a NaN, or is at least +0 with |y(hm)| at least 0.1875, the largest |y|
// of its elements is |y(hm)|, computed once with gelu_pair.  A thread for
// which that fails (all of its inputs below about 0.3, or none) reads its
// elements again and takes the largest |y| of gelu_pair on each.
template <int FMT, int CLUSTER>
__global__ void __launch_bounds__(kGeluCodeTableThreads, 1) gelu_code_table_kernel(const GeluArgs a) {
    extern __shared__ __align__(16) uint32_t tab32[];  // byte h: the FP8 code of y(h) / scale
    __shared__ uint32_t red[kGeluCodeTableThreads / 32];
    constexpr int E = GeluGeom::kVecElems;
    const int64_t stride = (int64_t)gridDim.x * kGeluCodeTableThreads;
    const int64_t v_first = (int64_t)blockIdx.x * kGeluCodeTableThreads + threadIdx.x;
    uint4 wa[kGeluTableUnroll], wb[kGeluTableUnroll];
    gelu_load(a, v_first, stride, wa, wb);  // before the build, which hides their latency
    const QScale c = make_qscale(a.scale);
    // word p: the codes of inputs 4p .. 4p + 3, lowest byte first
    if (c.fast)
        cluster_build<kGeluCodeTableThreads, CLUSTER, 16384>(tab32, [&c](int p) {
            const uint32_t h = 4u * (uint32_t)p;
            return quant_quad_x2<FMT, true>(gelu_pair(h | ((h + 1u) << 16)), gelu_pair((h + 2u) | ((h + 3u) << 16)), c);
        });
    else
        cluster_build<kGeluCodeTableThreads, CLUSTER, 16384>(tab32, [&c](int p) {
            const uint32_t h = 4u * (uint32_t)p;
            return quant_quad_x2<FMT, false>(gelu_pair(h | ((h + 1u) << 16)), gelu_pair((h + 2u) | ((h + 3u) << 16)), c);
        });
    cluster_sync_all();  // every CTA's table is complete; no remote store comes after this
    const uint8_t* tab = reinterpret_cast<const uint8_t*>(tab32);
    uint32_t hm2 = 0xFF80FF80u;  // the largest input so far, per bf16 lane (-inf: none)
    if (c.fast) code_table_stream<FMT, true>(a, tab, c, v_first, stride, wa, wb, hm2);
    else        code_table_stream<FMT, false>(a, tab, c, v_first, stride, wa, wb, hm2);
    const int64_t tail0 = a.head + a.nvec * E;
    const int64_t nscalar = blockIdx.x == 0 ? a.head + (a.n - tail0) : 0;  // head and tail: CTA 0
    for (int64_t j = threadIdx.x; j < nscalar; j += kGeluCodeTableThreads) {
        const int64_t i = j < a.head ? j : tail0 + (j - a.head);
        const uint32_t hv = a.h[i];
        a.q[i] = tab[hv];
        hm2 = bf16x2_max(hm2, hv | (hv << 16));
    }
    const uint32_t hm = bf16x2_max(hm2, hm2 >> 16) & 0xFFFFu;
    uint32_t m = gelu_abs_bits(hm);
    if ((hm & 0x8000u) || m < kGeluNegativeBound) {  // read the thread's elements again
        uint32_t m2 = 0;
        for (int64_t v = v_first; v < a.nvec; v += stride) {
            uint4 x, z;
            ld_stream_v8(a.h + a.head + v * E, x, z);
            m2 = bf16x2_absmax(m2, bf16x2_absmax(
                                       bf16x2_absmax(bf16x2_absmax(gelu_pair(x.x), gelu_pair(x.y)),
                                                     bf16x2_absmax(gelu_pair(x.z), gelu_pair(x.w))),
                                       bf16x2_absmax(bf16x2_absmax(gelu_pair(z.x), gelu_pair(z.y)),
                                                     bf16x2_absmax(gelu_pair(z.z), gelu_pair(z.w)))));
        }
        m = max(abs_bits_lo(m2), m2 & 0x7FFF0000u);
        for (int64_t j = threadIdx.x; j < nscalar; j += kGeluCodeTableThreads)
            m = max(m, gelu_abs_bits(a.h[j < a.head ? j : tail0 + (j - a.head)]));
    }
    // CTA-wide max of |y|, one atomic
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t b = red[0];
        for (int w = 1; w < kGeluCodeTableThreads / 32; ++w) b = max(b, red[w]);
        atomicMax(reinterpret_cast<int*>(a.amax), (int)b);
    }
}

// ----------------------------------------------------------------------------
// LayerNorm producer fused with quantize + amax
//
// Flax's default LayerNorm in binary32, row by row (H elements, a multiple of
// 16, at most 32768): mean = S / H, var = max(0, Q / H - mean^2) (a NaN kept),
// rstd = 1 / sqrt(var + eps), y = (x - mean) * (rstd * gamma) + beta rounded
// to bf16, then the quantize path on y: FP8 codes of y / scale and
// amax = max |y|.
//
// Persistent grid (as many CTAs as fit at once, at most one per batch).  A
// batch is R consecutive rows (R a power of two up to 32, chosen so that two
// batches fit the 64 KB shared-memory ring); CTA b takes batches b, b + G, ...
// A batch arrives by one cp.async.bulk copy completing on the mbarrier of its
// ring slot, and the slot is refilled with the batch two ahead once the CTA is
// done with it, so one batch is always in flight while the CTA computes the
// other.
//
// Phase 1, statistics: all 8 warps work, 8 / R on each row (R / 8 rows each,
// one after the other, when R > 8; up to 1024 columns 8 lanes take a row, see
// ln_row_sums8).  Warp part p of a
// row sums the row's 8-element vectors p, p + 8/R, ... of its lanes in four
// chains per lane (S = sum x and Q = sum x^2, the product exact inside each
// fma), folds them and the lanes (an xor butterfly, whose two lanes per
// exchange add the same two values, so every lane gets the same bits), and
// the row's warps add their totals in warp order after a named barrier.  The
// longest chain of additions is 2 ceil(H / (256 w)) + 6 + w with w = max(1, 8 / R)
// warps a row, at most H / 128 + 32.  The row's first warp stores (-mean, rstd).
// Phase 2, output: after one CTA barrier, all 256 threads normalise, round to
// bf16, store y (optional) and quantize, two rows at a time.  Thread t owns
// the 8-element half-vectors t, t + 256, ... of every row; with H <= 4096
// those are at most two, and their gamma and beta stay in registers for the
// whole launch (longer rows take the cluster kernel below, or this one reading
// gamma and beta per row where no cluster fits).  Shared-memory reads are 16 bytes per lane at consecutive
// addresses (no bank conflicts).  The normalisation takes the bf16 operand
// straight from its word (add.f32.bf16), then rstd * gamma and the fused
// multiply-add with beta two lanes at a time.
//
// Every mbarrier wait gives up after one second (kWaitLimitNs).  The CTA
// agrees on the outcome at its phase barrier; if any thread gave up, the CTA
// stores the pattern 0x7FFFFFFF (a NaN that no bf16 input can produce) into
// *amax, waits (again bounded) for its copies still in flight and returns.
// Correct operation never gets there; a test-only build
// (FP8Q_TEST_LN_GIVE_UP_AT) makes the wait of a CTA's batch of that index
// report failure, to exercise the path without any fault.

constexpr int kLnMaxH = 32768;
constexpr int kLnMaxHalfPerThread = 16;  // the largest HPT instantiated
static_assert(kLnMaxH <= kThreads * 8 * kLnMaxHalfPerThread, "every half-vector of a row has a thread");
constexpr int kLnWarps = kThreads / 32;
constexpr int kLnMaxBatch = 4 * kLnWarps;  // single-CTA kernel: short rows, several rows a warp
constexpr int kLnClusterBatch = kLnWarps;  // cluster kernel: at most one row a warp
constexpr int kLnBufs = 2;                      // batches in the ring
constexpr uint32_t kLnRingBytes = 64u * 1024u;  // ring per CTA (both batches), rows up to 16384
// Longer rows (batches of one row) take a ring of two rows: 4 H bytes, 128 KB at most.
__host__ __device__ constexpr uint32_t ln_ring_bytes(int H) {
    return kLnBufs * 2u * (uint32_t)H > kLnRingBytes ? kLnBufs * 2u * (uint32_t)H : kLnRingBytes;
}
constexpr int kLnTimeoutBits = 0x7FFFFFFF;

struct LnArgs {
    const uint16_t* x;
    uint16_t* y;  // may be null
    uint8_t* q;
    const float* gamma;
    const float* beta;
    const float* scale;
    float* amax;
    int64_t rows;
    int32_t H;
    int32_t batch;  // rows per batch: a power of two up to 32 (cluster kernel: up to 8)
    float eps;
    int32_t slice_half;  // cluster kernel: half-vectors of 8 per CTA's column slice
};

// Streaming stores whose target this kernel never reads back: no memory
// clobber, so shared-memory loads of the next rows may be scheduled across
// them.
__device__ __forceinline__ void st_cs_v4(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
}

__device__ __forceinline__ void st_cs_v2(void* p, uint2 v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y));
}

// Named barrier `id` over `threads` threads (whole warps).
__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// s = s + x and q = fma(x, x, q) for x the low (LO) or high half of a word of
// two bf16, with the mixed-precision add.f32.bf16 / fma.f32.bf16 (PTX,
// sm_100 and later): the bf16 operand is widened exactly, so the results are
// those of the binary32 add and fma on the widened value.
template <bool LO>
__device__ __forceinline__ void acc_bf16(uint32_t w, float& s, float& q) {
    if (LO)
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.bf16 %0, lo, %0;\n\tfma.rn.f32.bf16 %1, lo, lo, %1;\n\t}"
            : "+f"(s), "+f"(q)
            : "r"(w));
    else
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.bf16 %0, hi, %0;\n\tfma.rn.f32.bf16 %1, hi, hi, %1;\n\t}"
            : "+f"(s), "+f"(q)
            : "r"(w));
}

// x + c for x the low (LO) or high bf16 half of w, widened exactly.
template <bool LO>
__device__ __forceinline__ float add_bf16(uint32_t w, float c) {
    float d;
    if (LO)
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, lo, %2;\n\t}"
            : "=f"(d)
            : "r"(w), "f"(c));
    else
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, hi, %2;\n\t}"
            : "=f"(d)
            : "r"(w), "f"(c));
    return d;
}

// One word of two bf16 of x -> one word of two bf16 of y.
__device__ __forceinline__ uint32_t ln_pair(uint32_t w, float nmean, float2 rstd2, float2 g, float2 b) {
    const float2 d = make_float2(add_bf16<true>(w, nmean), add_bf16<false>(w, nmean));
    const float2 y = fma2_rn(d, mul2_rn(rstd2, g), b);
    return cvt_bf16x2(y.x, y.y);
}

__device__ __forceinline__ float max_nan_f32(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// One half-vector of the output: y (optional), its |y| into m2, its FP8 codes.
template <int FMT, bool WRITE_Y, bool FAST>
__device__ __forceinline__ void ln_out8(const LnArgs& a, uint4 w, const float2 (&g)[4], const float2 (&b)[4],
                                        float2 stats, const QScale& c, int64_t off, uint32_t& m2) {
    const float2 rstd2 = splat2(stats.y);
    uint4 yv;
    yv.x = ln_pair(w.x, stats.x, rstd2, g[0], b[0]);
    yv.y = ln_pair(w.y, stats.x, rstd2, g[1], b[1]);
    yv.z = ln_pair(w.z, stats.x, rstd2, g[2], b[2]);
    yv.w = ln_pair(w.w, stats.x, rstd2, g[3], b[3]);
    if (WRITE_Y) st_cs_v4(a.y + off, yv);
    m2 = bf16x2_absmax(m2, bf16x2_absmax(bf16x2_absmax(yv.x, yv.y), bf16x2_absmax(yv.z, yv.w)));
    st_cs_v2(a.q + off, quant8<FMT, FAST>(yv, c));
}

__device__ __forceinline__ void load4f2(const float* p, float2 (&d)[4]) {
    const float4 u = __ldg(reinterpret_cast<const float4*>(p));
    const float4 v = __ldg(reinterpret_cast<const float4*>(p) + 1);
    d[0] = make_float2(u.x, u.y);
    d[1] = make_float2(u.z, u.w);
    d[2] = make_float2(v.x, v.y);
    d[3] = make_float2(v.z, v.w);
}

// Phase 2 over one batch: rows two at a time.  The staged rows are
// `row_bytes` apart in shared memory and hold the `nh` half-vectors that
// start at column col0 of the row (the whole row, or a cluster CTA's slice).
template <int FMT, bool WRITE_Y, int HPT, bool FAST>
__device__ __forceinline__ void ln_emit_batch(const LnArgs& a, const uint8_t* base, const float2* stats, int nr,
                                              int64_t r0, const float2 (&gr)[HPT <= 2 ? HPT : 1][4],
                                              const float2 (&br)[HPT <= 2 ? HPT : 1][4], const QScale& c,
                                              uint32_t& m2, uint32_t row_bytes, int nh, int col0) {
    constexpr bool kGammaInRegs = (HPT <= 2);
    if (HPT == 1 && 2 * nh <= kThreads) {
        // Short rows (up to 1024 columns): thread t takes half-vector t % nh of rows
        // t / nh, t / nh + P, ... (P = 256 / nh >= 2 rows a pass), so that all threads
        // work (its gamma and beta were loaded for that column).  256 columns: 40 us
        // for 2^25 elements, against 63 us with one thread a column and rows two at a
        // time; 512: 31 against 40 us; with one row a pass (1536 columns) it was 7% slower.
        const int P = kThreads / nh, u = threadIdx.x % nh;
        for (int r = threadIdx.x / nh; r < nr && threadIdx.x < P * nh; r += P) {
            const uint4 w = *reinterpret_cast<const uint4*>(base + (size_t)r * row_bytes + 16 * u);
            ln_out8<FMT, WRITE_Y, FAST>(a, w, gr[0], br[0], stats[r], c, (r0 + r) * a.H + col0 + 8 * u, m2);
        }
        return;
    }
    for (int r = 0; r < nr; r += 2) {
        const bool pair = r + 1 < nr;
        const float2 s0 = stats[r], s1 = stats[pair ? r + 1 : r];
        const uint8_t* srow = base + (size_t)r * row_bytes;
        const int64_t row_off = (r0 + r) * a.H + col0;
#pragma unroll
        for (int i = 0; i < HPT; ++i) {
            const int u = threadIdx.x + i * kThreads;
            if (u < nh) {
                const uint4 w0 = *reinterpret_cast<const uint4*>(srow + 16 * u);
                uint4 w1 = w0;
                if (pair) w1 = *reinterpret_cast<const uint4*>(srow + row_bytes + 16 * u);
                float2 g[4], b[4];
                if (kGammaInRegs) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        g[e] = gr[kGammaInRegs ? i : 0][e];
                        b[e] = br[kGammaInRegs ? i : 0][e];
                    }
                } else {
                    load4f2(a.gamma + col0 + 8 * u, g);
                    load4f2(a.beta + col0 + 8 * u, b);
                }
                const int64_t off = row_off + 8 * u;
                ln_out8<FMT, WRITE_Y, FAST>(a, w0, g, b, s0, c, off, m2);
                if (pair) ln_out8<FMT, WRITE_Y, FAST>(a, w1, g, b, s1, c, off + a.H, m2);
            }
        }
    }
}

// Phase 1 for one staged row of nv8 half-vectors: the sums S = sum x and
// Q = sum x^2 of the row's warps (group prow, wpr warps, this one ppart),
// each warp in four chains per lane, folded, then over the lanes (xor
// butterfly: every lane gets the same bits) and, for wpr > 1, the group's
// warp totals added in warp order after a named barrier.  The group's first
// warp returns the row's totals; a warp whose copy did not arrive reads nothing.
// With kGroupOk, group_ok (for the group's first warp) also says whether every
// warp of the group saw its copy arrive.
template <bool kGroupOk = false>
__device__ __forceinline__ void ln_row_sums(const uint8_t* xr, int nv8, bool warp_arrived, int lane, int warp,
                                            int prow, int ppart, int wpr, float2* part, float& S, float& Q,
                                            uint32_t* warp_ok = nullptr, bool* group_ok = nullptr) {
    float s[4] = {0.0f, 0.0f, 0.0f, 0.0f}, q[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int j = lane + 32 * ppart; warp_arrived && j < nv8; j += 32 * wpr) {
        const uint4 w = *reinterpret_cast<const uint4*>(xr + 16 * j);
        acc_bf16<true>(w.x, s[0], q[0]);
        acc_bf16<true>(w.y, s[1], q[1]);
        acc_bf16<true>(w.z, s[2], q[2]);
        acc_bf16<true>(w.w, s[3], q[3]);
        acc_bf16<false>(w.x, s[0], q[0]);
        acc_bf16<false>(w.y, s[1], q[1]);
        acc_bf16<false>(w.z, s[2], q[2]);
        acc_bf16<false>(w.w, s[3], q[3]);
    }
    S = __fadd_rn(__fadd_rn(s[0], s[1]), __fadd_rn(s[2], s[3]));
    Q = __fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        S = __fadd_rn(S, __shfl_xor_sync(0xFFFFFFFFu, S, o));
        Q = __fadd_rn(Q, __shfl_xor_sync(0xFFFFFFFFu, Q, o));
    }
    if (kGroupOk) *group_ok = warp_arrived;
    if (wpr > 1) {
        if (lane == 0) {
            part[warp] = make_float2(S, Q);
            if (kGroupOk) warp_ok[warp] = warp_arrived ? 1u : 0u;
        }
        named_sync(1 + prow, 32 * wpr);
        if (ppart == 0) {  // the row's warp totals, in warp order
            for (int p = 1; p < wpr; ++p) {
                S = __fadd_rn(S, part[warp + p].x);
                Q = __fadd_rn(Q, part[warp + p].y);
                if (kGroupOk) *group_ok = *group_ok && warp_ok[warp + p] != 0;
            }
        }
    }
}

// The same sums over 8 lanes (lane sl of its group of 8), for short rows: each
// lane sums its half-vectors sl, sl + 8, ... in four chains, folds them, and the
// group adds its lanes by an xor butterfly over 4, 2, 1 (every lane of the group
// gets the same bits).  All 32 lanes of the warp call it together; a group whose
// row does not exist or whose copy is missing reads nothing.
constexpr int kLnShortHalf = 128;  // half-vectors a row (1024 columns) up to which phase 1 uses 8 lanes a row
__device__ __forceinline__ void ln_row_sums8(const uint8_t* xr, int nv8, bool read, int sl, float& S, float& Q) {
    float s[4] = {0.0f, 0.0f, 0.0f, 0.0f}, q[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int j = sl; read && j < nv8; j += 8) {
        const uint4 w = *reinterpret_cast<const uint4*>(xr + 16 * j);
        acc_bf16<true>(w.x, s[0], q[0]);
        acc_bf16<true>(w.y, s[1], q[1]);
        acc_bf16<true>(w.z, s[2], q[2]);
        acc_bf16<true>(w.w, s[3], q[3]);
        acc_bf16<false>(w.x, s[0], q[0]);
        acc_bf16<false>(w.y, s[1], q[1]);
        acc_bf16<false>(w.z, s[2], q[2]);
        acc_bf16<false>(w.w, s[3], q[3]);
    }
    S = __fadd_rn(__fadd_rn(s[0], s[1]), __fadd_rn(s[2], s[3]));
    Q = __fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3]));
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) {
        S = __fadd_rn(S, __shfl_xor_sync(0xFFFFFFFFu, S, o));
        Q = __fadd_rn(Q, __shfl_xor_sync(0xFFFFFFFFu, Q, o));
    }
}

// (-mean, rstd) of a row of H elements from its sums.
__device__ __forceinline__ float2 ln_row_stats(float S, float Q, float Hf, float eps) {
    const float mean = __fdiv_rn(S, Hf);
    const float var = max_nan_f32(__fsub_rn(__fdiv_rn(Q, Hf), __fmul_rn(mean, mean)), 0.0f);
    return make_float2(-mean, __frsqrt_rn(__fadd_rn(var, eps)));
}

// HPT: most 8-element half-vectors a thread owns per row (ceil(H / 2048)).
template <int FMT, bool WRITE_Y, int HPT>
__global__ void __launch_bounds__(kThreads, 2) layernorm_quantize_amax_kernel(const LnArgs a) {
    extern __shared__ __align__(128) uint8_t ring[];  // kLnBufs batches of a.batch rows of 2H bytes
    __shared__ uint64_t bar[kLnBufs];
    __shared__ float2 part[kLnWarps];     // (S, Q) of each warp's part of its row
    __shared__ float2 stats[kLnMaxBatch];  // (-mean, rstd) of each row of the batch
    __shared__ uint32_t red[kLnWarps];
    constexpr bool kGammaInRegs = (HPT <= 2);
    const int nv8 = a.H / 8, nh = a.H / 8;
    const int R = a.batch;
    const int wpr = R < kLnWarps ? kLnWarps / R : 1;  // warps per row in phase 1
    const uint32_t row_bytes = 2u * (uint32_t)a.H;
    const uint32_t buf_bytes = (uint32_t)R * row_bytes;
    const int64_t nb = (a.rows + R - 1) / R;
    const int64_t G = gridDim.x;
    const int64_t n_mine = (nb - 1 - blockIdx.x) / G + 1;  // the launch keeps G <= nb
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int prow = warp / wpr, ppart = warp % wpr;        // phase 1: this warp's row and part

    if (threadIdx.x == 0) {
        for (int b = 0; b < kLnBufs; ++b) mbar_init(&bar[b]);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int64_t k = 0; k < kLnBufs && k < n_mine; ++k) {
            const int64_t r0 = (blockIdx.x + k * G) * R;
            const int64_t nr = a.rows - r0 < R ? a.rows - r0 : R;
            bulk_load(ring + (size_t)k * buf_bytes, a.x + r0 * a.H, (uint32_t)nr * row_bytes, &bar[k]);
        }
    }
    const QScale c = make_qscale(a.scale);
    const float Hf = (float)a.H;
    float2 gr[kGammaInRegs ? HPT : 1][4], br[kGammaInRegs ? HPT : 1][4];
    if (kGammaInRegs) {
#pragma unroll
        for (int i = 0; i < (kGammaInRegs ? HPT : 0); ++i) {
            // short rows (up to 1024 columns): column threadIdx.x % nh, see ln_emit_batch
            const int u = (HPT == 1 && 2 * nh <= kThreads) ? (int)threadIdx.x % nh : threadIdx.x + i * kThreads;
            if (u < nh) {
                load4f2(a.gamma + 8 * u, gr[i]);
                load4f2(a.beta + 8 * u, br[i]);
            }
        }
    }
    __syncthreads();  // barriers initialised before anyone waits on them

    uint32_t m2 = 0;
    bool ok = true;
    int64_t k = 0;
    for (; k < n_mine; ++k) {
        const int buf = (int)(k % kLnBufs);
        const uint32_t parity = (uint32_t)((k / kLnBufs) & 1);
        const int64_t r0 = (blockIdx.x + k * G) * R;
        const int nr = a.rows - r0 < R ? (int)(a.rows - r0) : R;
        const uint8_t* base = ring + (size_t)buf * buf_bytes;
        bool arrived = mbar_wait(&bar[buf], parity);
#ifdef FP8Q_TEST_LN_GIVE_UP_AT
        if (k == FP8Q_TEST_LN_GIVE_UP_AT) arrived = false;
#endif
        // Every warp of a row's group reaches the group's named barrier whatever
        // its own wait saw (a warp whose copy is missing reads nothing); the
        // CTA then agrees on the outcome at its barrier below.
        const bool warp_arrived = __all_sync(0xFFFFFFFFu, arrived);
        if (HPT == 1 && nv8 <= kLnShortHalf) {
            // Short rows (up to 1024 columns, R >= 16): 8 lanes a row, 4 rows a warp at once.
            const int sub = lane >> 3, sl = lane & 7;
            for (int base_row = 0; base_row < nr; base_row += 4 * kLnWarps) {
                const int row = base_row + 4 * warp + sub;
                float S, Q;
                ln_row_sums8(base + (size_t)row * row_bytes, nv8, warp_arrived && row < nr, sl, S, Q);
                if (sl == 0 && row < nr) stats[row] = ln_row_stats(S, Q, Hf, a.eps);
            }
        } else {
            // row prow, and with more rows than warps also prow + 8, prow + 16, ...
            for (int row = prow; row < nr; row += kLnWarps) {
                float S, Q;
                ln_row_sums(base + (size_t)row * row_bytes, nv8, warp_arrived, lane, warp, prow, ppart, wpr, part, S,
                            Q);
                if (ppart == 0 && lane == 0) stats[row] = ln_row_stats(S, Q, Hf, a.eps);
            }
        }
        ok = __syncthreads_and(arrived) != 0;
        if (!ok) break;  // uniform
        if (c.fast) ln_emit_batch<FMT, WRITE_Y, HPT, true>(a, base, stats, nr, r0, gr, br, c, m2, row_bytes, nh, 0);
        else        ln_emit_batch<FMT, WRITE_Y, HPT, false>(a, base, stats, nr, r0, gr, br, c, m2, row_bytes, nh, 0);
        __syncthreads();  // every thread is done with this slot and with stats[] and part[]
        if (threadIdx.x == 0 && k + kLnBufs < n_mine) {  // refill the slot, kLnBufs batches ahead
            const int64_t next_r0 = (blockIdx.x + (k + kLnBufs) * G) * R;
            const int64_t next_nr = a.rows - next_r0 < R ? a.rows - next_r0 : R;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            bulk_load(ring + (size_t)buf * buf_bytes, a.x + next_r0 * a.H, (uint32_t)next_nr * row_bytes, &bar[buf]);
        }
    }
    if (!ok) {
        // A copy did not arrive in time: mark the result, then wait (bounded)
        // for the copies this CTA still has in flight before leaving.
        if (threadIdx.x == 0) {
            atomicMax(reinterpret_cast<int*>(a.amax), kLnTimeoutBits);
            for (int64_t j = k; j < n_mine && j < k + kLnBufs; ++j)
                mbar_wait(&bar[j % kLnBufs], (uint32_t)((j / kLnBufs) & 1));
        }
        return;
    }
    flush_amax(m2, 0u, a.amax, red);
}

// ----------------------------------------------------------------------------
// LayerNorm rows longer than 4096, split over a thread-block cluster
//
// With H > 4096 a CTA of 256 threads cannot keep the gamma and beta of a whole
// row in registers, and reading them again for every row costs more than the
// rest of the work.  A cluster of C = ceil(H / 4096) CTAs takes each batch of
// rows together: CTA c owns the column slice of half-vectors [c hs, (c+1) hs)
// (hs = ceil(H / 8C), the last slice shorter), stages that slice of each of the
// batch's rows (one bulk copy per row, all completing on the slot's mbarrier)
// and keeps its slice's gamma and beta in registers for the whole launch.
// Phase 1 sums its slice of each row as the single-CTA kernel does.  The
// row's first lane then sends (S, Q, "every warp of the group saw its copy")
// to every CTA of the cluster, itself included, with st.async: a 16-byte store
// into the other CTA's shared memory that completes on that CTA's exchange
// mbarrier of the batch's parity, which expects C x 16 bytes per row.  The
// writer needs no fence, and no cluster barrier runs per batch.  Each CTA
// waits (bounded) for its exchange barrier; the row's first lane adds the C
// partials in rank order, so every CTA derives the same (mean, rstd) bits, and
// checks the C flags; one CTA barrier then agrees on the outcome and
// publishes the statistics.  Phase 2 is the single-CTA kernel's on the slice.
// A CTA writes a peer's slot of parity p for batch j only after its own
// exchange for batch j - 1 completed, which needed that peer's sums of batch
// j - 1, sent after the peer had read its slot for batch j - 2: one slot per
// parity is enough.  The longest chain of additions is the slice's plus C - 1,
// within H / 128 + 32.  Remote stores start after a split cluster barrier that
// every CTA enters once its mbarriers are initialised, and every CTA passes a
// last cluster barrier before it exits, so no CTA writes into one that has
// left.  A copy that never arrives clears its group's flag; every CTA then
// stops at the same batch, marks amax and drains its copies.

constexpr int kLnClusterMax = 8;
constexpr int kLnSliceHalf = kThreads * 2;  // half-vectors a CTA's slice may hold (4096 columns)
constexpr uint32_t kLnClusterRingBytes = 96u * 1024u;  // both slots at most (two CTAs an SM): batches of 8 rows up to 3072 columns

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// A 16-byte store into another CTA's shared memory that completes on an
// mbarrier there (its expected transaction bytes): no fence on the writing side.
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint4 v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     addr),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
                 : "memory");
}

// The copies of one batch: the slice of each of its nr rows, completing on bar.
__device__ __forceinline__ void ln_slice_batch_load(const LnArgs& a, uint8_t* dst, int64_t r0, int nr, int h0,
                                                    uint32_t slice_bytes, uint32_t row_stride, uint64_t* bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"((uint32_t)nr * slice_bytes)
                 : "memory");
    for (int r = 0; r < nr; ++r)
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                smem_addr(dst + (size_t)r * row_stride)),
            "l"(a.x + (r0 + r) * a.H + 8 * h0), "r"(slice_bytes), "r"(smem_addr(bar))
            : "memory");
}

template <int FMT, bool WRITE_Y>
__global__ void __launch_bounds__(kThreads, 2) layernorm_cluster_quantize_amax_kernel(const LnArgs a) {
    extern __shared__ __align__(128) uint8_t ring[];  // kLnBufs batches of a.batch slices of 16 slice_half bytes
    __shared__ uint64_t bar[kLnBufs];                        // the ring's copies
    __shared__ uint64_t xbar[2];                             // the partial sums' arrival, by batch parity
    __shared__ float2 part[kLnWarps];
    __shared__ uint32_t warp_ok[kLnWarps];
    __shared__ float2 stats[kLnClusterBatch];
    __shared__ uint4 xpart[2][kLnClusterMax][kLnClusterBatch];  // (S, Q, group arrived, 0) of every CTA, by batch parity
    __shared__ uint32_t red[kLnWarps];
    const int C = (int)cluster_nctarank(), crank = (int)cluster_ctarank();
    const int h0 = crank * a.slice_half;                        // the slice's first half-vector
    const int nhc = min(a.slice_half, a.H / 8 - h0);           // > 0: the launch keeps every slice non-empty
    const int R = a.batch;
    const int wpr = kLnWarps / R;
    const uint32_t row_stride = 16u * (uint32_t)a.slice_half;  // bytes between staged rows
    const uint32_t slice_bytes = 16u * (uint32_t)nhc;
    const uint32_t buf_bytes = (uint32_t)R * row_stride;
    const int64_t nb = (a.rows + R - 1) / R;
    const int64_t cid = blockIdx.x / C, G = gridDim.x / C;     // clusters take batches cid, cid + G, ...
    const int64_t n_mine = (nb - 1 - cid) / G + 1;             // the launch keeps G <= nb
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int prow = warp / wpr, ppart = warp % wpr;

    if (threadIdx.x == 0) {
        for (int b = 0; b < kLnBufs; ++b) mbar_init(&bar[b]);
        for (int b = 0; b < 2; ++b) mbar_init(&xbar[b]);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int64_t k = 0; k < kLnBufs && k < n_mine; ++k) {
            const int64_t r0 = (cid + k * G) * R;
            const int nr = a.rows - r0 < R ? (int)(a.rows - r0) : R;
            ln_slice_batch_load(a, ring + (size_t)k * buf_bytes, r0, nr, h0, slice_bytes, row_stride, &bar[k]);
        }
    }
    cluster_arrive_relaxed();  // after the barriers' initialisation; waited on before the first remote store
    const QScale c = make_qscale(a.scale);
    const float Hf = (float)a.H;
    float2 gr[2][4], br[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int u = threadIdx.x + i * kThreads;
        if (u < nhc) {
            load4f2(a.gamma + 8 * (h0 + u), gr[i]);
            load4f2(a.beta + 8 * (h0 + u), br[i]);
        }
    }
    __syncthreads();  // barriers initialised before anyone waits on them

    uint32_t m2 = 0;
    bool ok = true;
    int64_t k = 0;
    for (; k < n_mine; ++k) {
        const int buf = (int)(k % kLnBufs);
        const int xp = (int)(k & 1);
        const int64_t r0 = (cid + k * G) * R;
        const int nr = a.rows - r0 < R ? (int)(a.rows - r0) : R;
        const uint8_t* base = ring + (size_t)buf * buf_bytes;
        if (threadIdx.x == 0)  // the batch's partial sums from every CTA of the cluster
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&xbar[xp])),
                         "r"((uint32_t)C * 16u * (uint32_t)nr)
                         : "memory");
        bool arrived = mbar_wait(&bar[buf], (uint32_t)((k / kLnBufs) & 1));
#ifdef FP8Q_TEST_LN_GIVE_UP_AT
        if (k == FP8Q_TEST_LN_GIVE_UP_AT) arrived = false;
#endif
        const bool warp_arrived = __all_sync(0xFFFFFFFFu, arrived);
        const bool first = prow < nr && ppart == 0 && lane == 0;  // the lane that speaks for its row
        if (k == 0) cluster_wait();  // every CTA of the cluster is running, its barriers initialised
        if (prow < nr) {
            float S, Q;
            bool group_ok;
            ln_row_sums<true>(base + (size_t)prow * row_stride, nhc, warp_arrived, lane, warp, prow, ppart, wpr, part,
                              S, Q, warp_ok, &group_ok);
            if (first) {
                const uint32_t at = smem_addr(&xpart[xp][crank][prow]), xb = smem_addr(&xbar[xp]);
                const uint4 v = make_uint4(__float_as_uint(S), __float_as_uint(Q), group_ok ? 1u : 0u, 0u);
                for (int r = 0; r < C; ++r) st_async_v4(cluster_map(at, (uint32_t)r), v, cluster_map(xb, (uint32_t)r));
            }
        }
        // Every CTA gets the same C x nr partials; the row's first lane adds them in
        // rank order, and every CTA stops at the same batch if any group's copy failed.
        bool mine_ok = mbar_wait(&xbar[xp], (uint32_t)((k >> 1) & 1));
        if (first && mine_ok) {
            uint4 v = xpart[xp][0][prow];
            float Sx = __uint_as_float(v.x), Qx = __uint_as_float(v.y);
            mine_ok = v.z != 0;
            for (int r = 1; r < C; ++r) {
                v = xpart[xp][r][prow];
                Sx = __fadd_rn(Sx, __uint_as_float(v.x));
                Qx = __fadd_rn(Qx, __uint_as_float(v.y));
                mine_ok = mine_ok && v.z != 0;
            }
            stats[prow] = ln_row_stats(Sx, Qx, Hf, a.eps);
        }
        ok = __syncthreads_and(mine_ok) != 0;  // also publishes stats[]
        if (!ok) break;  // uniform over the cluster (a lost exchange only after a second)
        if (c.fast) ln_emit_batch<FMT, WRITE_Y, 2, true>(a, base, stats, nr, r0, gr, br, c, m2, row_stride, nhc, 8 * h0);
        else        ln_emit_batch<FMT, WRITE_Y, 2, false>(a, base, stats, nr, r0, gr, br, c, m2, row_stride, nhc, 8 * h0);
        __syncthreads();  // every thread is done with this slot and with stats[] and part[]
        if (threadIdx.x == 0 && k + kLnBufs < n_mine) {
            const int64_t next_r0 = (cid + (k + kLnBufs) * G) * R;
            const int next_nr = a.rows - next_r0 < R ? (int)(a.rows - next_r0) : R;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            ln_slice_batch_load(a, ring + (size_t)buf * buf_bytes, next_r0, next_nr, h0, slice_bytes, row_stride,
                                &bar[buf]);
        }
    }
    if (!ok) {
        if (threadIdx.x == 0) {
            atomicMax(reinterpret_cast<int*>(a.amax), kLnTimeoutBits);
            for (int64_t j = k; j < n_mine && j < k + kLnBufs; ++j)
                mbar_wait(&bar[j % kLnBufs], (uint32_t)((j / kLnBufs) & 1));
        }
    } else {
        flush_amax(m2, 0u, a.amax, red);
    }
    // No CTA leaves while another of its cluster may still write into its shared memory.
    cluster_arrive_relaxed();
    cluster_wait();
}

// Resident CTAs of one kernel per device, taken on the first launch there
// (the persistent LayerNorm grid and the GELU table path).
struct ResidentCache {
    std::mutex mu;
    struct Entry {
        int dev;
        int ctas;
    } e[32];
    int n = 0;
};

template <int FMT, bool WRITE_Y, int HPT>
fp8q_status launch_layernorm_hpt(LnArgs a, cudaStream_t s) {
    static ResidentCache cache;
    auto kern = layernorm_quantize_amax_kernel<FMT, WRITE_Y, HPT>;
    const uint32_t row_bytes = 2u * (uint32_t)a.H;
    uint32_t batch = ln_ring_bytes(a.H) / (kLnBufs * row_bytes);
    // a power of two: 8 / batch warps a row, or batch / 8 rows a warp
    batch = batch >= 32 ? 32 : batch >= 16 ? 16 : batch >= 8 ? 8 : batch >= 4 ? 4 : batch >= 2 ? 2 : 1;
    a.batch = (int32_t)batch;
    const uint32_t smem = kLnBufs * batch * row_bytes;
    // the most any H of this instance takes: the resident count holds for all of them
    const uint32_t smem_max = ln_ring_bytes(HPT * kThreads * 8 < kLnMaxH ? HPT * kThreads * 8 : kLnMaxH);
    int dev = 0, ctas = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) {
        std::lock_guard<std::mutex> lock(cache.mu);
        for (int k = 0; k < cache.n; ++k)
            if (cache.e[k].dev == dev) ctas = cache.e[k].ctas;
        if (ctas == 0) {
            int per_sm = 0, sms = 0;
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max);
            if (err == cudaSuccess)
                err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem_max);
            if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (err == cudaSuccess && per_sm < 1) err = cudaErrorInvalidConfiguration;
            if (err == cudaSuccess) {
                ctas = per_sm * sms;
                if (cache.n < 32) cache.e[cache.n++] = {dev, ctas};
            }
        }
    }
    if (err != cudaSuccess) return cuda_fail(err, "layernorm_quantize_amax_kernel setup");
    const int64_t batches = (a.rows + batch - 1) / batch;
    const int grid = (int)(batches < (int64_t)ctas ? batches : (int64_t)ctas);
    return launch_kernel(kern, dim3((unsigned)grid), dim3(kThreads), smem, s, "layernorm_quantize_amax_kernel", a);
}

#ifdef FP8Q_TEST_HOOKS  // test-only build: LayerNorm clusters larger than this count as not fitting (0: no limit)
int g_test_ln_max_cluster = 0;
#endif

// Rows longer than 4096 on clusters of ceil(H / 4096) CTAs, each cluster taking
// batches of rows in turn over the clusters that fit at once.  Where no cluster
// of that size fits (a partitioned or shared GPU), this returns
// FP8Q_ERR_UNSUPPORTED without recording a CUDA error, and the caller takes the
// single-CTA kernel.
template <int FMT, bool WRITE_Y>
fp8q_status launch_layernorm_cluster(LnArgs a, cudaStream_t s) {
    static ResidentCache cache[kLnClusterMax + 1];  // resident clusters x C, by cluster size C
    const int nh = a.H / 8;
    const int C = (nh + kLnSliceHalf - 1) / kLnSliceHalf;  // 2 .. 8 for 4096 < H <= 32768
    const int hs = (nh + C - 1) / C;                       // every slice non-empty: nh > 512 (C - 1) >= C (C - 1)
#ifdef FP8Q_TEST_HOOKS
    if (g_test_ln_max_cluster > 0 && C > g_test_ln_max_cluster) return FP8Q_ERR_UNSUPPORTED;
#endif
    uint32_t batch = kLnClusterRingBytes / (kLnBufs * 16u * (uint32_t)hs);
    batch = batch >= 8 ? 8 : batch >= 4 ? 4 : batch >= 2 ? 2 : 1;
    a.batch = (int32_t)batch;
    a.slice_half = hs;
    auto kern = layernorm_cluster_quantize_amax_kernel<FMT, WRITE_Y>;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kLnClusterRingBytes;  // the most any slice takes: the resident count holds for all
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int dev = 0, ctas = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) {
        ResidentCache& rc = cache[C];
        std::lock_guard<std::mutex> lock(rc.mu);
        for (int k = 0; k < rc.n; ++k)
            if (rc.e[k].dev == dev) ctas = rc.e[k].ctas;
        if (ctas == 0) {
            int clusters = 0, sms = 0;
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLnClusterRingBytes);
            if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            cfg.gridDim = dim3((unsigned)(sms / C * C));
            if (err == cudaSuccess) err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
            if (err == cudaSuccess) {
                ctas = clusters > 0 ? clusters * C : -1;  // -1: no cluster of this size fits
                if (rc.n < 32) rc.e[rc.n++] = {dev, ctas};
            }
        }
    }
    if (err != cudaSuccess) return cuda_fail(err, "layernorm_cluster_quantize_amax_kernel setup");
    if (ctas < 0) return FP8Q_ERR_UNSUPPORTED;
    const int64_t batches = (a.rows + batch - 1) / batch;
    const int64_t clusters = batches < (int64_t)(ctas / C) ? batches : (int64_t)(ctas / C);
    cfg.gridDim = dim3((unsigned)(clusters * C));
    cfg.dynamicSmemBytes = kLnBufs * batch * 16u * (uint32_t)hs;
    err = cudaLaunchKernelEx(&cfg, kern, a);
    return err == cudaSuccess ? FP8Q_OK : cuda_fail(err, "layernorm_cluster_quantize_amax_kernel");
}

template <int FMT, bool WRITE_Y>
fp8q_status launch_layernorm(const LnArgs& a, cudaStream_t s) {
    const int hpt = (a.H / 8 + kThreads - 1) / kThreads;  // half-vectors per thread
    if (hpt <= 1) return launch_layernorm_hpt<FMT, WRITE_Y, 1>(a, s);
    if (hpt <= 2) return launch_layernorm_hpt<FMT, WRITE_Y, 2>(a, s);
    const fp8q_status st = launch_layernorm_cluster<FMT, WRITE_Y>(a, s);
    if (st != FP8Q_ERR_UNSUPPORTED) return st;
    // no cluster of that size fits on this device: one CTA per batch of rows
    if (hpt <= 4) return launch_layernorm_hpt<FMT, WRITE_Y, 4>(a, s);
    if (hpt <= 8) return launch_layernorm_hpt<FMT, WRITE_Y, 8>(a, s);
    return launch_layernorm_hpt<FMT, WRITE_Y, 16>(a, s);
}

// Launch a table kernel on the clusters that fit at once (at most one CTA per
// vector pair of its threads, rounded up to whole clusters).
#ifdef FP8Q_TEST_HOOKS  // test-only build: clusters larger than this count as not fitting (0: no limit)
int g_test_gelu_max_cluster = 0;
#endif

// A table kernel needs its thread-block clusters resident at once.  Where no
// cluster of its size fits (a partitioned or shared GPU), this returns
// FP8Q_ERR_UNSUPPORTED without recording a CUDA error, and the caller takes a
// smaller cluster or the direct kernel.
template <typename Kern>
fp8q_status launch_gelu_table(Kern kern, int threads, int unroll, int cluster, uint32_t smem, ResidentCache& cache,
                              const GeluArgs& a, cudaStream_t s, const char* name) {
#ifdef FP8Q_TEST_HOOKS
    if (g_test_gelu_max_cluster > 0 && cluster > g_test_gelu_max_cluster) return FP8Q_ERR_UNSUPPORTED;
#endif
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    int ctas = 0;
    if (err == cudaSuccess) {
        std::lock_guard<std::mutex> lock(cache.mu);
        for (int k = 0; k < cache.n; ++k)
            if (cache.e[k].dev == dev) ctas = cache.e[k].ctas;
        if (ctas == 0) {
            // resident CTAs: the clusters that fit at once, times their size
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            int clusters = 0, sms = 0;
            if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            cfg.gridDim = dim3((unsigned)(sms / cluster * cluster));
            if (err == cudaSuccess) err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
            if (err == cudaSuccess) {
                ctas = clusters > 0 ? clusters * cluster : -1;  // -1: no cluster of this size fits
                if (cache.n < 32) cache.e[cache.n++] = {dev, ctas};
            }
        }
    }
    if (err != cudaSuccess) return cuda_fail(err, name);
    if (ctas < 0) return FP8Q_ERR_UNSUPPORTED;
    const int64_t per_cta = (int64_t)threads * unroll;
    const int64_t need = (a.nvec + per_cta - 1) / per_cta;
    int grid = (int)(need < ctas ? (need > 0 ? need : 1) : ctas);
    grid = (grid + cluster - 1) / cluster * cluster;  // whole clusters
    cfg.gridDim = dim3((unsigned)grid);
    err = cudaLaunchKernelEx(&cfg, kern, a);
    return err == cudaSuccess ? FP8Q_OK : cuda_fail(err, name);
}

// The table kernel with y, its cluster size chosen by the tensor's size; a
// smaller cluster where the first does not fit; FP8Q_ERR_UNSUPPORTED where
// neither does (the caller then takes the direct kernel).
template <int FMT>
fp8q_status launch_gelu_y_table(const GeluArgs& a, cudaStream_t s) {
    static ResidentCache cache, cache_small;
    if (a.n < kGeluYTableSmallBelow) {
        const fp8q_status st = launch_gelu_table(gelu_table_quantize_amax_kernel<FMT, kGeluYTableClusterSmall>,
                                                 kGeluYTableThreads, kGeluYUnroll, kGeluYTableClusterSmall,
                                                 kGeluYTableBytes, cache_small, a, s, "gelu_table_quantize_amax_kernel");
        if (st != FP8Q_ERR_UNSUPPORTED) return st;
    }
    return launch_gelu_table(gelu_table_quantize_amax_kernel<FMT, kGeluYTableCluster>, kGeluYTableThreads,
                             kGeluYUnroll, kGeluYTableCluster, kGeluYTableBytes, cache, a, s,
                             "gelu_table_quantize_amax_kernel");
}

// The code table kernel, likewise.
template <int FMT>
fp8q_status launch_gelu_code_table(const GeluArgs& a, cudaStream_t s) {
    static ResidentCache cache, cache_small;
    if (a.n < kGeluCodeTableSmallBelow) {
        const fp8q_status st = launch_gelu_table(gelu_code_table_kernel<FMT, kGeluCodeTableClusterSmall>,
                                                 kGeluCodeTableThreads, kGeluTableUnroll, kGeluCodeTableClusterSmall,
                                                 kGeluCodeTableBytes, cache_small, a, s, "gelu_code_table_kernel");
        if (st != FP8Q_ERR_UNSUPPORTED) return st;
    }
    return launch_gelu_table(gelu_code_table_kernel<FMT, kGeluCodeTableCluster>, kGeluCodeTableThreads,
                             kGeluTableUnroll, kGeluCodeTableCluster, kGeluCodeTableBytes, cache, a, s,
                             "gelu_code_table_kernel");
}

}  // namespace

// ----------------------------------------------------------------------------
// C ABI

extern "C" {

#ifdef FP8Q_TEST_HOOKS
// Test-only build: GELU table kernels with clusters larger than `max_cluster`
// behave as if their clusters did not fit (0 lifts the limit).
void fp8q_test_set_gelu_max_cluster(int max_cluster) { g_test_gelu_max_cluster = max_cluster; }
// Test-only build: LayerNorm clusters larger than `max_cluster` behave as if
// they did not fit (0 lifts the limit).
void fp8q_test_set_ln_max_cluster(int max_cluster) { g_test_ln_max_cluster = max_cluster; }
#endif

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
    if (sp.mode == kModeVec && n >= (y_bf16 ? kGeluTableMinElemsWithY : kGeluTableMinElems)) {
        fp8q_status st;
        if (fmt == FP8Q_E4M3FN)
            st = y_bf16 ? launch_gelu_y_table<FP8Q_E4M3FN>(a, s) : launch_gelu_code_table<FP8Q_E4M3FN>(a, s);
        else
            st = y_bf16 ? launch_gelu_y_table<FP8Q_E5M2>(a, s) : launch_gelu_code_table<FP8Q_E5M2>(a, s);
        if (st != FP8Q_ERR_UNSUPPORTED) return st;
        // no table kernel's cluster fits on this device: the direct kernel below
    }
    auto kern = fmt == FP8Q_E4M3FN ? (y_bf16 ? gelu_quantize_amax_kernel<FP8Q_E4M3FN, true>
                                             : gelu_quantize_amax_kernel<FP8Q_E4M3FN, false>)
                                    : (y_bf16 ? gelu_quantize_amax_kernel<FP8Q_E5M2, true>
                                             : gelu_quantize_amax_kernel<FP8Q_E5M2, false>);
    return launch_kernel(kern, dim3((unsigned)grid), dim3(kThreads), 0, s, "gelu_quantize_amax_kernel", a);
}

fp8q_status fp8q_layernorm_quantize_amax(const void* x_bf16, void* y_bf16, uint8_t* q, int64_t rows,
                                         int32_t hidden, const float* gamma, const float* beta, float eps,
                                         fp8q_format fmt, const float* scale, float* amax, void* stream) {
    if (!valid_fmt(fmt) || rows < 0 || hidden < 16 || (hidden % 16) != 0) return FP8Q_ERR_INVALID_ARG;
    if (hidden > kLnMaxH) return FP8Q_ERR_UNSUPPORTED;
    if (rows == 0) return FP8Q_OK;
    if (!x_bf16 || !q || !gamma || !beta || !scale || !amax) return FP8Q_ERR_INVALID_ARG;
    if (((uintptr_t)scale & 3u) || ((uintptr_t)amax & 3u)) return FP8Q_ERR_INVALID_ARG;
    if (((uintptr_t)x_bf16 & 15u) || ((uintptr_t)y_bf16 & 15u) || ((uintptr_t)q & 15u) ||
        ((uintptr_t)gamma & 15u) || ((uintptr_t)beta & 15u))
        return FP8Q_ERR_UNSUPPORTED;
    LnArgs a;
    a.x = static_cast<const uint16_t*>(x_bf16);
    a.y = static_cast<uint16_t*>(y_bf16);
    a.q = q;
    a.gamma = gamma;
    a.beta = beta;
    a.scale = scale;
    a.amax = amax;
    a.rows = rows;
    a.H = hidden;
    a.batch = 0;
    a.eps = eps;
    a.slice_half = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fmt == FP8Q_E4M3FN)
        return y_bf16 ? launch_layernorm<FP8Q_E4M3FN, true>(a, s) : launch_layernorm<FP8Q_E4M3FN, false>(a, s);
    return y_bf16 ? launch_layernorm<FP8Q_E5M2, true>(a, s) : launch_layernorm<FP8Q_E5M2, false>(a, s);
}

}  // extern "C"
