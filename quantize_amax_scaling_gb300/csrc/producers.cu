// producers.cu -- the producers fused with quantize + amax:
// GELU (elementwise) and LayerNorm (row-wise).

#include "fp8q_common.cuh"
#include "packed_f32.cuh"

#include <mutex>

namespace {

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
// y = bf16(GELU(h)) depends only on the 16 bits of h.  For large tensors each
// CTA first gets all 65536 values, computed with gelu_pair -- the arithmetic
// of the kernel above, so the same bits -- into shared memory (128 KB); the
// CTAs of a thread-block cluster compute them once between them.  It then
// streams its share of the tensor with one shared-memory lookup per element
// in place of the GELU arithmetic.  One CTA per SM (the table fills most of
// the shared memory), looping over the vectors two at a time, with the next
// two already loading while the current two are converted, so that enough
// loads are in flight.  Building the table costs each cluster about what
// 65536 elements cost the direct kernel, so smaller tensors, and any that
// take the element-by-element path, use the direct kernel.

// threads per CTA: 1024 for the codes alone; 512 when y is stored too (its
// extra registers would spill at 1024)
template <bool WRITE_Y>
__host__ __device__ constexpr int gelu_table_threads() { return WRITE_Y ? 512 : 1024; }
constexpr uint32_t kGeluTableBytes = 65536u * 2u;
// Fewer elements take the direct kernel (measured crossovers on GB300: the
// table wins from about 2^24 elements for the codes alone, 2^26 with y).
constexpr int64_t kGeluTableMinElems = (int64_t)1 << 24;
constexpr int64_t kGeluTableMinElemsWithY = (int64_t)1 << 26;
constexpr int kGeluTableUnroll = 2;
// CTAs of one thread-block cluster (on as many SMs) build their tables
// together: each computes its share of the entries and stores each into the
// shared memory of every CTA of the cluster.  Measured on GB300 (8192x16384):
// clusters of 2 for the codes alone (1024 threads build fast; 72.1 us, 74.3
// without clusters, 74.2 with 4), of 4 with y (512 threads; 112.7 us, 118.5
// without, 117.4 with 2).  Clusters of 8 leave SMs idle (86.4 us codes only).
template <bool WRITE_Y>
__host__ __device__ constexpr int gelu_table_cluster() { return WRITE_Y ? 4 : 2; }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

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

__device__ __forceinline__ uint32_t gelu_lookup_pair(const uint16_t* tab, uint32_t w) {
    return (uint32_t)tab[w & 0xFFFFu] | ((uint32_t)tab[w >> 16] << 16);
}

__device__ __forceinline__ uint4 gelu_lookup4(const uint16_t* tab, const uint4& w) {
    return make_uint4(gelu_lookup_pair(tab, w.x), gelu_lookup_pair(tab, w.y), gelu_lookup_pair(tab, w.z),
                      gelu_lookup_pair(tab, w.w));
}

template <int FMT, bool WRITE_Y>
__global__ void __launch_bounds__(gelu_table_threads<WRITE_Y>(), 1)
    gelu_table_quantize_amax_kernel(const GeluArgs a) {
    constexpr int kGeluTableThreads = gelu_table_threads<WRITE_Y>();
    extern __shared__ __align__(16) uint32_t tab32[];  // word p: the results for inputs 2p and 2p + 1
    __shared__ uint32_t red[kGeluTableThreads / 32];
    {
        constexpr int kGeluTableCluster = gelu_table_cluster<WRITE_Y>();
        constexpr int kShare = 32768 / kGeluTableCluster;  // at least the CTA's thread count
        // No CTA may touch another's shared memory before that CTA is known to
        // be running: arrive on the cluster barrier now, and wait on it just
        // before the first remote store, with the first pair computed meanwhile.
        cluster_arrive_relaxed();
        const uint32_t rank = cluster_ctarank();
        uint32_t dst[kGeluTableCluster];
#pragma unroll
        for (int r = 0; r < kGeluTableCluster; ++r) dst[r] = cluster_map(smem_addr(tab32), (uint32_t)r);
        int p = (int)rank * kShare + threadIdx.x;
        uint32_t y = gelu_pair((uint32_t)(2 * p) | ((uint32_t)(2 * p + 1) << 16));
        cluster_wait();
        for (;;) {
#pragma unroll
            for (int r = 0; r < kGeluTableCluster; ++r) st_cluster_u32(dst[r] + 4u * (uint32_t)p, y);
            p += kGeluTableThreads;
            if (p >= ((int)rank + 1) * kShare) break;
            y = gelu_pair((uint32_t)(2 * p) | ((uint32_t)(2 * p + 1) << 16));
        }
    }
    const QScale c = make_qscale(a.scale);
    cluster_sync_all();  // every CTA's table is complete; no remote store comes after this
    const uint16_t* tab = reinterpret_cast<const uint16_t*>(tab32);
    constexpr int E = GeluGeom::kVecElems;
    const int64_t stride = (int64_t)gridDim.x * kGeluTableThreads;
    uint32_t m2 = 0, ms = 0;
    int64_t v0 = (int64_t)blockIdx.x * kGeluTableThreads + threadIdx.x;
    uint4 wa[kGeluTableUnroll], wb[kGeluTableUnroll];
#pragma unroll
    for (int u = 0; u < kGeluTableUnroll; ++u) {
        const int64_t v = v0 + u * stride;
        if (v < a.nvec) ld_stream_v8(a.h + a.head + v * E, wa[u], wb[u]);
    }
    for (; v0 < a.nvec; v0 += kGeluTableUnroll * stride) {
        uint4 na[kGeluTableUnroll], nb[kGeluTableUnroll];
        const int64_t v1 = v0 + kGeluTableUnroll * stride;
#pragma unroll
        for (int u = 0; u < kGeluTableUnroll; ++u) {
            const int64_t v = v1 + u * stride;
            if (v < a.nvec) ld_stream_v8(a.h + a.head + v * E, na[u], nb[u]);
        }
#pragma unroll
        for (int u = 0; u < kGeluTableUnroll; ++u) {
            const int64_t v = v0 + u * stride;
            if (v < a.nvec) {
                const uint4 ya = gelu_lookup4(tab, wa[u]), yb = gelu_lookup4(tab, wb[u]);
                if (c.fast) gelu_emit<FMT, true, WRITE_Y>(a, c, v, ya, yb, m2);
                else        gelu_emit<FMT, false, WRITE_Y>(a, c, v, ya, yb, m2);
            }
        }
#pragma unroll
        for (int u = 0; u < kGeluTableUnroll; ++u) {
            wa[u] = na[u];
            wb[u] = nb[u];
        }
    }
    if (blockIdx.x == 0) {  // scalar head and tail, each shorter than one vector
        const int64_t tail0 = a.head + a.nvec * E;
        const int64_t nscalar = a.head + (a.n - tail0);
        for (int64_t j = threadIdx.x; j < nscalar; j += kGeluTableThreads) {
            const int64_t i = j < a.head ? j : tail0 + (j - a.head);
            const uint32_t yw = tab[a.h[i]];
            if (WRITE_Y) a.y[i] = (uint16_t)yw;
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
        for (int w = 1; w < kGeluTableThreads / 32; ++w) b = max(b, red[w]);
        atomicMax(reinterpret_cast<int*>(a.amax), (int)b);
    }
}

// ----------------------------------------------------------------------------
// LayerNorm producer fused with quantize + amax
//
// Flax's default LayerNorm in binary32, row by row (H elements, a multiple of
// 16, at most 16384): mean = S / H, var = max(0, Q / H - mean^2) (a NaN kept),
// rstd = 1 / sqrt(var + eps), y = (x - mean) * (rstd * gamma) + beta rounded
// to bf16, then the quantize path on y: FP8 codes of y / scale and
// amax = max |y|.
//
// A row belongs to a group of G = ceil(H / 4096) warps.  Lane l of warp g of
// the group holds the 8-element vectors l + 32 (g + G i), i < KV, of the row
// in registers (KV = H / (256 G), rounded up to a power of two; vectors past
// the row read as +0), so x comes from HBM once and nothing is staged in
// shared memory.  The sums S = sum x and Q = sum x^2 (an exact product inside
// each fma) run in four chains per lane (2 KV elements each), fold pairwise,
// fold across the warp as an xor butterfly (the two lanes of each exchange
// add the same two values, so every lane ends with the same bits), and for
// G > 1 the warp totals are added in warp order after a named barrier of the
// group.  The longest chain of additions is 2 KV + 2 + 5 + (G - 1) <= 42.
// The output step then normalises each pair of elements with the bf16 operand
// taken straight from its word (add.f32.bf16), rstd * gamma and the fused
// multiply-add with beta two lanes at a time, rounds to bf16 and quantizes.
//
// Each CTA takes a contiguous, balanced range of rows, and its groups take
// every (8 / G)-th row of it; a group asks L2 for its next row (one bulk
// prefetch) before it loads the current one, so HBM keeps streaming while the
// group computes.  No thread waits on anything but the group's named barrier
// and one CTA barrier at the end, both in uniform control flow.

constexpr int kLnMaxH = 16384;
constexpr int kLnWarpCols = 4096;  // columns per warp at most (KV <= 16)

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
    float eps;
};

// Streaming stores whose target this kernel never reads back: no memory
// clobber, so the loads of later rows may be scheduled across them.
__device__ __forceinline__ void st_cs_v4(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
}

__device__ __forceinline__ void st_cs_v2(void* p, uint2 v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y));
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Ask L2 to fetch `bytes` (a multiple of 16, 16-byte aligned) starting at p.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
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

// Eight bf16 of y -> eight FP8 codes.
template <int FMT, bool FAST>
__device__ __forceinline__ uint2 ln_quant8(const uint4& y, const QScale& c) {
    if (FAST)
        return make_uint2(quant_pair_x2<FMT>(y.x, c) | (quant_pair_x2<FMT>(y.y, c) << 16),
                          quant_pair_x2<FMT>(y.z, c) | (quant_pair_x2<FMT>(y.w, c) << 16));
    return make_uint2(quant_quad<FMT, false>(y.x, y.y, c), quant_quad<FMT, false>(y.z, y.w, c));
}

__device__ __forceinline__ float max_nan_f32(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

template <int G>
__host__ __device__ constexpr int ln_threads() { return 32 * G * (8 / G); }

// The output of one row: y (optional), |y| into m2, the FP8 codes.
template <int FMT, bool WRITE_Y, int KV, int G, bool FAST>
__device__ __forceinline__ void ln_emit_row(const LnArgs& a, const uint4 (&v)[KV], int64_t row, int gw, int lane,
                                            int nv, float nmean, float rstd, const QScale& c, uint32_t& m2) {
    const float2 rstd2 = splat2(rstd);
#pragma unroll
    for (int i = 0; i < KV; ++i) {
        const int j = lane + 32 * (gw + G * i);
        if (j < nv) {
            const float4 g0 = __ldg(reinterpret_cast<const float4*>(a.gamma) + 2 * j);
            const float4 g1 = __ldg(reinterpret_cast<const float4*>(a.gamma) + 2 * j + 1);
            const float4 b0 = __ldg(reinterpret_cast<const float4*>(a.beta) + 2 * j);
            const float4 b1 = __ldg(reinterpret_cast<const float4*>(a.beta) + 2 * j + 1);
            uint4 yv;
            yv.x = ln_pair(v[i].x, nmean, rstd2, make_float2(g0.x, g0.y), make_float2(b0.x, b0.y));
            yv.y = ln_pair(v[i].y, nmean, rstd2, make_float2(g0.z, g0.w), make_float2(b0.z, b0.w));
            yv.z = ln_pair(v[i].z, nmean, rstd2, make_float2(g1.x, g1.y), make_float2(b1.x, b1.y));
            yv.w = ln_pair(v[i].w, nmean, rstd2, make_float2(g1.z, g1.w), make_float2(b1.z, b1.w));
            const int64_t off = row * a.H + 8 * (int64_t)j;
            if (WRITE_Y) st_cs_v4(a.y + off, yv);
            m2 = bf16x2_absmax(m2, bf16x2_absmax(bf16x2_absmax(yv.x, yv.y), bf16x2_absmax(yv.z, yv.w)));
            st_cs_v2(a.q + off, ln_quant8<FMT, FAST>(yv, c));
        }
    }
}

template <int FMT, bool WRITE_Y, int KV, int G>
__global__ void __launch_bounds__(ln_threads<G>(), 2) layernorm_quantize_amax_kernel(const LnArgs a) {
    constexpr int kGroups = 8 / G;
    constexpr int kWarps = G * kGroups;
    __shared__ float2 part[kGroups][2][G];  // (S, Q) of each warp of a group, by row parity
    __shared__ uint32_t red[kWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = warp / G, gw = warp % G;
    const int nv = a.H >> 3;
    const int64_t r_begin = a.rows * (int64_t)blockIdx.x / gridDim.x;
    const int64_t r_end = a.rows * ((int64_t)blockIdx.x + 1) / gridDim.x;
    const QScale c = make_qscale(a.scale);
    const float Hf = (float)a.H;
    const uint32_t row_bytes = 2u * (uint32_t)a.H;
    uint32_t m2 = 0;
    int parity = 0;
    for (int64_t row = r_begin + grp; row < r_end; row += kGroups, parity ^= 1) {
        if (gw == 0 && lane == 0 && row + kGroups < r_end)
            prefetch_l2_bulk(a.x + (row + kGroups) * a.H, row_bytes);
        const uint16_t* xr = a.x + row * a.H;
        uint4 v[KV];
#pragma unroll
        for (int i = 0; i < KV; ++i) {
            const int j = lane + 32 * (gw + G * i);
            v[i] = j < nv ? ld_stream_v4(xr + 8 * j) : make_uint4(0u, 0u, 0u, 0u);
        }
        float s[4] = {0.0f, 0.0f, 0.0f, 0.0f}, q[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < KV; ++i) {
            acc_bf16<true>(v[i].x, s[0], q[0]);
            acc_bf16<true>(v[i].y, s[1], q[1]);
            acc_bf16<true>(v[i].z, s[2], q[2]);
            acc_bf16<true>(v[i].w, s[3], q[3]);
            acc_bf16<false>(v[i].x, s[0], q[0]);
            acc_bf16<false>(v[i].y, s[1], q[1]);
            acc_bf16<false>(v[i].z, s[2], q[2]);
            acc_bf16<false>(v[i].w, s[3], q[3]);
        }
        float S = __fadd_rn(__fadd_rn(s[0], s[1]), __fadd_rn(s[2], s[3]));
        float Q = __fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3]));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            S = __fadd_rn(S, __shfl_xor_sync(0xFFFFFFFFu, S, o));
            Q = __fadd_rn(Q, __shfl_xor_sync(0xFFFFFFFFu, Q, o));
        }
        if (G > 1) {
            if (lane == 0) part[grp][parity][gw] = make_float2(S, Q);
            named_sync(1 + grp, 32 * G);
            // every warp of the group adds the warp totals in the same order
            float2 t = part[grp][parity][0];
#pragma unroll
            for (int k = 1; k < G; ++k) {
                const float2 u = part[grp][parity][k];
                t.x = __fadd_rn(t.x, u.x);
                t.y = __fadd_rn(t.y, u.y);
            }
            S = t.x;
            Q = t.y;
        }
        const float mean = __fdiv_rn(S, Hf);
        const float var = max_nan_f32(__fsub_rn(__fdiv_rn(Q, Hf), __fmul_rn(mean, mean)), 0.0f);
        const float rstd = __frsqrt_rn(__fadd_rn(var, a.eps));
        if (c.fast) ln_emit_row<FMT, WRITE_Y, KV, G, true>(a, v, row, gw, lane, nv, -mean, rstd, c, m2);
        else        ln_emit_row<FMT, WRITE_Y, KV, G, false>(a, v, row, gw, lane, nv, -mean, rstd, c, m2);
    }
    // CTA-wide max of |y|, one atomic
    uint32_t m = max(abs_bits_lo(m2), m2 & 0x7FFF0000u);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t b = red[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) b = max(b, red[w]);
        atomicMax(reinterpret_cast<int*>(a.amax), (int)b);
    }
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

template <int FMT, bool WRITE_Y, int KV, int G>
fp8q_status launch_layernorm_kv(const LnArgs& a, cudaStream_t s) {
    static ResidentCache cache;
    auto kern = layernorm_quantize_amax_kernel<FMT, WRITE_Y, KV, G>;
    constexpr int threads = ln_threads<G>();
    int dev = 0, ctas = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) {
        std::lock_guard<std::mutex> lock(cache.mu);
        for (int k = 0; k < cache.n; ++k)
            if (cache.e[k].dev == dev) ctas = cache.e[k].ctas;
        if (ctas == 0) {
            int per_sm = 0, sms = 0;
            err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0);
            if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (err == cudaSuccess && per_sm < 1) err = cudaErrorInvalidConfiguration;
            if (err == cudaSuccess) {
                ctas = per_sm * sms;
                if (cache.n < 32) cache.e[cache.n++] = {dev, ctas};
            }
        }
    }
    if (err != cudaSuccess) return cuda_fail(err, "layernorm_quantize_amax_kernel setup");
    // as many CTAs as fit at once, but no more than give each group a row
    const int64_t want = (a.rows + (8 / G) - 1) / (8 / G);
    const int grid = (int)(want < (int64_t)ctas ? want : (int64_t)ctas);
    return launch_kernel(kern, dim3((unsigned)grid), dim3(threads), 0, s, "layernorm_quantize_amax_kernel", a);
}

template <int FMT, bool WRITE_Y>
fp8q_status launch_layernorm(const LnArgs& a, cudaStream_t s) {
    const int G = (a.H + kLnWarpCols - 1) / kLnWarpCols;
    const int kv = (a.H / 8 + 32 * G - 1) / (32 * G);  // vectors per lane
    if (G == 1) {
        if (kv <= 1) return launch_layernorm_kv<FMT, WRITE_Y, 1, 1>(a, s);
        if (kv <= 2) return launch_layernorm_kv<FMT, WRITE_Y, 2, 1>(a, s);
        if (kv <= 4) return launch_layernorm_kv<FMT, WRITE_Y, 4, 1>(a, s);
        if (kv <= 8) return launch_layernorm_kv<FMT, WRITE_Y, 8, 1>(a, s);
        return launch_layernorm_kv<FMT, WRITE_Y, 16, 1>(a, s);
    }
    if (G == 2) return launch_layernorm_kv<FMT, WRITE_Y, 16, 2>(a, s);
    if (G == 3) return launch_layernorm_kv<FMT, WRITE_Y, 16, 3>(a, s);
    return launch_layernorm_kv<FMT, WRITE_Y, 16, 4>(a, s);
}

template <int FMT, bool WRITE_Y>
fp8q_status launch_gelu_table(const GeluArgs& a, cudaStream_t s) {
    static ResidentCache cache;
    constexpr int kGeluTableThreads = gelu_table_threads<WRITE_Y>();
    constexpr int kGeluTableCluster = gelu_table_cluster<WRITE_Y>();
    auto kern = gelu_table_quantize_amax_kernel<FMT, WRITE_Y>;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kGeluTableCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kGeluTableThreads);
    cfg.dynamicSmemBytes = kGeluTableBytes;
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
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGeluTableBytes);
            int clusters = 0, sms = 0;
            if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            cfg.gridDim = dim3((unsigned)(sms / kGeluTableCluster * kGeluTableCluster));
            if (err == cudaSuccess) err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
            if (err == cudaSuccess && clusters < 1) err = cudaErrorInvalidConfiguration;
            if (err == cudaSuccess) {
                ctas = clusters * kGeluTableCluster;
                if (cache.n < 32) cache.e[cache.n++] = {dev, ctas};
            }
        }
    }
    if (err != cudaSuccess) return cuda_fail(err, "gelu_table_quantize_amax_kernel setup");
    const int64_t per_cta = (int64_t)kGeluTableThreads * kGeluTableUnroll;
    const int64_t need = (a.nvec + per_cta - 1) / per_cta;
    int grid = (int)(need < ctas ? (need > 0 ? need : 1) : ctas);
    grid = (grid + kGeluTableCluster - 1) / kGeluTableCluster * kGeluTableCluster;  // whole clusters
    cfg.gridDim = dim3((unsigned)grid);
    err = cudaLaunchKernelEx(&cfg, kern, a);
    return err == cudaSuccess ? FP8Q_OK : cuda_fail(err, "gelu_table_quantize_amax_kernel launch");
}

}  // namespace

// ----------------------------------------------------------------------------
// C ABI

extern "C" {

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
        if (fmt == FP8Q_E4M3FN)
            return y_bf16 ? launch_gelu_table<FP8Q_E4M3FN, true>(a, s) : launch_gelu_table<FP8Q_E4M3FN, false>(a, s);
        return y_bf16 ? launch_gelu_table<FP8Q_E5M2, true>(a, s) : launch_gelu_table<FP8Q_E5M2, false>(a, s);
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
    a.eps = eps;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fmt == FP8Q_E4M3FN)
        return y_bf16 ? launch_layernorm<FP8Q_E4M3FN, true>(a, s) : launch_layernorm<FP8Q_E4M3FN, false>(a, s);
    return y_bf16 ? launch_layernorm<FP8Q_E5M2, true>(a, s) : launch_layernorm<FP8Q_E5M2, false>(a, s);
}

}  // extern "C"
