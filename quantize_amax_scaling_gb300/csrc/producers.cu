// producers.cu -- the producers fused with quantize + amax:
// GELU (elementwise) and LayerNorm (row-wise).

#include "fp8q_common.cuh"

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
// LayerNorm producer fused with quantize + amax
//
// Flax's default LayerNorm in binary32, row by row (H elements, H a multiple
// of 16, at most 16384): mean = S / H, var = max(0, Q / H - mean^2),
// rstd = 1 / sqrt(var + eps), y = (x - mean) * (rstd * gamma) + beta rounded
// to bf16, then the quantize path on y.  S and Q are summed in one fixed
// association that the CPU reference of this library writes out the same way:
// vector v (16 elements) belongs to lane v mod 256, each lane adds its
// elements in index order (s = s + x, q = fma(x, x, q)), warps fold with the
// xor butterfly (offsets 16 .. 1), and the 8 warp totals are added left to
// right.
//
// Persistent grid (as many CTAs as fit on the GPU at once, at most one per
// row); CTA b takes rows b, b + G, b + 2G, ...  Each CTA keeps a ring of
// whole rows in shared memory, filled by cp.async.bulk copies that complete
// on one mbarrier per stage, so up to `stages` rows (64 KB) per CTA are in
// flight while the CTA computes.  A stage is refilled with the row `stages`
// ahead as soon as every thread has copied it into registers (the first
// block-wide reduction's barrier).  With at most 256 vectors per row
// (H <= 4096) each thread always owns the same 16 columns, so it keeps their
// gamma and beta in registers for all its rows.
//
// Every mbarrier wait has a time limit (kWaitLimitNs).  The CTA agrees on the
// outcome at the next barrier; if any thread gave up, the CTA stores the
// pattern 0x7FFFFFFF (a NaN that no bf16 input can produce) into *amax, waits
// (again bounded) for its copies still in flight and returns.

constexpr int kLnMaxVecPerThread = 4;           // H <= 256 * 16 * 4 = 16384
constexpr int kLnMaxStages = 16;
constexpr uint32_t kLnRingBytes = 64u * 1024u;  // shared-memory ring per CTA
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kAmaxTimeoutBits = 0x7FFFFFFF;

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
    int32_t stages;  // ring depth, 2 .. kLnMaxStages, at most kLnRingBytes in all
    float eps;
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
}

// Start a copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global memory into shared memory; its completion flips *bar's phase.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Wait until *bar has completed the phase of the given parity; false if that
// has not happened within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (done) return true;
        if (it == 0) t0 = global_ns();
        else if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Warp part of the fixed-order row sums: the xor butterfly over offsets
// 16 .. 1, for S and Q side by side.  Lane 0 (every lane) ends with the warp's
// totals.
__device__ __forceinline__ float2 warp_sums_fixed_order(float s, float q) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, o));
        q = __fadd_rn(q, __shfl_xor_sync(0xFFFFFFFFu, q, o));
    }
    return make_float2(s, q);
}

// Row statistics from the 8 warp totals (left to right), as (-mean, rstd).
__device__ __forceinline__ float2 ln_stats(const float2* part, int H, float eps) {
    float S = part[0].x, Q = part[0].y;
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) {
        S = __fadd_rn(S, part[w].x);
        Q = __fadd_rn(Q, part[w].y);
    }
    const float Hf = (float)H;
    const float mean = __fdiv_rn(S, Hf);
    float var = __fsub_rn(__fdiv_rn(Q, Hf), __fmul_rn(mean, mean));
    var = var > 0.0f ? var : 0.0f;
    return make_float2(-mean, __frcp_rn(__fsqrt_rn(__fadd_rn(var, eps))));
}

// Two-lane binary32 add and multiply (PTX f32x2, sm_100 and later), each lane
// rounded to nearest even exactly like add.rn.f32 / mul.rn.f32.  A two-lane
// multiply whose result feeds a two-lane add was measured to come out as one
// fused multiply-add (a single rounding) on sm_103a even with the explicit
// rounding mode, so a product that is then added is formed with the scalar
// __fmul_rn / __fadd_rn pair, which is never contracted.
__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Eight bf16 of x (one uint4) -> eight bf16 of y:
// y = ((x + (-mean)) * (rstd * gamma)) + beta, each step rounded on its own
// (x + (-mean) is x - mean); the first two steps two lanes at a time.
__device__ __forceinline__ uint4 ln_normalize8(uint4 w, const float2 (&g)[4], const float2 (&b)[4],
                                               float2 nmean, float2 rstd) {
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t out[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 x = make_float2(__uint_as_float(in[k] << 16), __uint_as_float(in[k] & 0xFFFF0000u));
        const float2 d = add2_rn(x, nmean);
        const float2 m = mul2_rn(rstd, g[k]);
        out[k] = cvt_bf16x2(__fadd_rn(__fmul_rn(d.x, m.x), b[k].x), __fadd_rn(__fmul_rn(d.y, m.y), b[k].y));
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// quant_pair (fast path) with the first product taken two lanes at a time.
template <int FMT>
__device__ __forceinline__ uint32_t quant_pair_x2(uint32_t w, const QScale& c, float2 r2) {
    w = bf16x2_clamp(w, c.t2);
    const float2 x = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    const float2 y0 = mul2_rn(x, r2);
    const float e0 = __fmaf_rn(y0.x, c.s, -x.x);
    const float e1 = __fmaf_rn(y0.y, c.s, -x.y);
    return cvt_fp8x2<FMT>(__fmaf_rn(-e0, c.r, y0.x), __fmaf_rn(-e1, c.r, y0.y));
}

template <int FMT, bool FAST>
__device__ __forceinline__ uint4 ln_quant16(const uint4& ya, const uint4& yb, const QScale& c, float2 r2) {
    if (FAST)
        return make_uint4(quant_pair_x2<FMT>(ya.x, c, r2) | (quant_pair_x2<FMT>(ya.y, c, r2) << 16),
                          quant_pair_x2<FMT>(ya.z, c, r2) | (quant_pair_x2<FMT>(ya.w, c, r2) << 16),
                          quant_pair_x2<FMT>(yb.x, c, r2) | (quant_pair_x2<FMT>(yb.y, c, r2) << 16),
                          quant_pair_x2<FMT>(yb.z, c, r2) | (quant_pair_x2<FMT>(yb.w, c, r2) << 16));
    return make_uint4(quant_quad<FMT, false>(ya.x, ya.y, c), quant_quad<FMT, false>(ya.z, ya.w, c),
                      quant_quad<FMT, false>(yb.x, yb.y, c), quant_quad<FMT, false>(yb.z, yb.w, c));
}

__device__ __forceinline__ void load4f2(const float* p, float2 (&d)[4]) {
    const float4 u = __ldg(reinterpret_cast<const float4*>(p));
    const float4 v = __ldg(reinterpret_cast<const float4*>(p) + 1);
    d[0] = make_float2(u.x, u.y);
    d[1] = make_float2(u.z, u.w);
    d[2] = make_float2(v.x, v.y);
    d[3] = make_float2(v.z, v.w);
}

template <int FMT, bool WRITE_Y, int VPT>
__global__ void __launch_bounds__(kThreads) layernorm_quantize_amax_kernel(const LnArgs a) {
    extern __shared__ __align__(128) uint8_t ring[];  // a.stages rows of 2H bytes
    __shared__ uint64_t bar[kLnMaxStages];
    __shared__ float2 part[kThreads / 32];  // per-warp (S, Q)
    __shared__ float2 stats;                // (-mean, rstd) of the current row
    __shared__ uint32_t red[kThreads / 32];
    constexpr bool kGammaInRegs = (VPT == 1);
    const int nv = a.H / 16;
    const uint32_t row_bytes = 2u * (uint32_t)a.H;
    const int64_t G = gridDim.x;
    const int64_t n_mine = (a.rows - 1 - blockIdx.x) / G + 1;  // the launch keeps G <= rows
    const int stages = a.stages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&bar[s]);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int s = 0; s < stages && s < n_mine; ++s)
            bulk_load(ring + (size_t)s * row_bytes, a.x + (blockIdx.x + s * G) * a.H, row_bytes, &bar[s]);
    }
    const QScale c = make_qscale(a.scale);
    const float2 r2 = make_float2(c.r, c.r);
    float2 gr[kGammaInRegs ? 2 : 1][4], br[kGammaInRegs ? 2 : 1][4];
    if (kGammaInRegs && (int)threadIdx.x < nv) {
        load4f2(a.gamma + 16 * threadIdx.x, gr[0]);
        load4f2(a.gamma + 16 * threadIdx.x + 8, gr[kGammaInRegs ? 1 : 0]);
        load4f2(a.beta + 16 * threadIdx.x, br[0]);
        load4f2(a.beta + 16 * threadIdx.x + 8, br[kGammaInRegs ? 1 : 0]);
    }
    __syncthreads();  // barriers initialised before anyone waits on them

    uint32_t m2 = 0;
    bool ok = true;
    int st = 0;
    uint32_t parity = 0;
    int64_t i = 0;
    for (; i < n_mine; ++i) {
        const int64_t row = blockIdx.x + i * G;
        const bool arrived = mbar_wait(&bar[st], parity);
        const uint8_t* srow = ring + (size_t)st * row_bytes;
        uint4 wa[VPT], wb[VPT];
        float s = 0.0f, q = 0.0f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = threadIdx.x + k * kThreads;
            if (v < nv) {
                wa[k] = *reinterpret_cast<const uint4*>(srow + 32 * v);
                wb[k] = *reinterpret_cast<const uint4*>(srow + 32 * v + 16);
                const uint32_t w8[8] = {wa[k].x, wa[k].y, wa[k].z, wa[k].w, wb[k].x, wb[k].y, wb[k].z, wb[k].w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float x0 = __uint_as_float(w8[e] << 16);
                    const float x1 = __uint_as_float(w8[e] & 0xFFFF0000u);
                    s = __fadd_rn(s, x0);
                    q = __fmaf_rn(x0, x0, q);
                    s = __fadd_rn(s, x1);
                    q = __fmaf_rn(x1, x1, q);
                }
            }
        }
        const float2 wsum = warp_sums_fixed_order(s, q);
        if (lane == 0) part[warp] = wsum;
        ok = __syncthreads_and(arrived) != 0;  // every thread also holds its part of the row now
        if (!ok) break;                        // uniform
        if (warp == 0) {
            if (lane == 0 && i + stages < n_mine)  // refill the stage just read
                bulk_load(ring + (size_t)st * row_bytes, a.x + (row + stages * G) * a.H, row_bytes, &bar[st]);
            const float2 t = ln_stats(part, a.H, a.eps);
            if (lane == 0) stats = t;
        }
        __syncthreads();
        const float2 sv = stats;
        const float2 nmean = make_float2(sv.x, sv.x), rstd = make_float2(sv.y, sv.y);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = threadIdx.x + k * kThreads;
            if (v < nv) {
                float2 g0[4], g1[4], b0[4], b1[4];
                if (kGammaInRegs) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        g0[e] = gr[0][e]; g1[e] = gr[kGammaInRegs ? 1 : 0][e];
                        b0[e] = br[0][e]; b1[e] = br[kGammaInRegs ? 1 : 0][e];
                    }
                } else {
                    load4f2(a.gamma + 16 * v, g0);
                    load4f2(a.gamma + 16 * v + 8, g1);
                    load4f2(a.beta + 16 * v, b0);
                    load4f2(a.beta + 16 * v + 8, b1);
                }
                const uint4 ya = ln_normalize8(wa[k], g0, b0, nmean, rstd);
                const uint4 yb = ln_normalize8(wb[k], g1, b1, nmean, rstd);
                const int64_t off = row * a.H + 16 * v;
                if (WRITE_Y) {
                    st_v4(a.y + off, ya);
                    st_v4(a.y + off + 8, yb);
                }
                m2 = bf16x2_absmax(m2, bf16x2_absmax(bf16x2_absmax(bf16x2_absmax(ya.x, ya.y),
                                                                   bf16x2_absmax(ya.z, ya.w)),
                                                     bf16x2_absmax(bf16x2_absmax(yb.x, yb.y),
                                                                   bf16x2_absmax(yb.z, yb.w))));
                const uint4 o = c.fast ? ln_quant16<FMT, true>(ya, yb, c, r2) : ln_quant16<FMT, false>(ya, yb, c, r2);
                st_v4(a.q + off, o);
            }
        }
        if (++st == stages) {
            st = 0;
            parity ^= 1u;
        }
    }
    if (!ok) {
        // A copy did not arrive in time: mark the result, then wait (bounded)
        // for the copies this CTA still has in flight before leaving.
        if (threadIdx.x == 0) {
            atomicMax(reinterpret_cast<int*>(a.amax), kAmaxTimeoutBits);
            for (int64_t j = i; j < n_mine && j < i + stages; ++j) {
                const int64_t d = j - i + st;
                mbar_wait(&bar[d % stages], parity ^ (uint32_t)((d / stages) & 1));
            }
        }
        return;
    }
    flush_amax(m2, 0u, a.amax, red);
}

// Resident CTAs of one kernel instantiation at a given dynamic shared-memory
// size, per device (the persistent LayerNorm grid).  The first use on a device
// also raises the kernel's dynamic shared-memory limit to kLnRingBytes.
struct ResidentCache {
    std::mutex mu;
    struct Entry {
        int dev;
        uint32_t smem;
        int ctas;
    } e[32];
    int n = 0;
};

template <class K>
cudaError_t resident_ctas(K kern, uint32_t smem, ResidentCache& cache, int* ctas) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(cache.mu);
    for (int k = 0; k < cache.n; ++k) {
        if (cache.e[k].dev == dev && cache.e[k].smem == smem) {
            *ctas = cache.e[k].ctas;
            return cudaSuccess;
        }
    }
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLnRingBytes);
    if (err != cudaSuccess) return err;
    int per_sm = 0, sms = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    *ctas = per_sm * sms;
    if (cache.n < 32) cache.e[cache.n++] = {dev, smem, *ctas};
    return cudaSuccess;
}

template <int FMT, bool WRITE_Y, int VPT>
fp8q_status launch_layernorm_vpt(LnArgs a, cudaStream_t s) {
    static ResidentCache cache;
    auto kern = layernorm_quantize_amax_kernel<FMT, WRITE_Y, VPT>;
    const uint32_t row_bytes = 2u * (uint32_t)a.H;
    int stages = (int)(kLnRingBytes / row_bytes);
    stages = stages < 2 ? 2 : (stages > kLnMaxStages ? kLnMaxStages : stages);
    a.stages = stages;
    const uint32_t smem = (uint32_t)stages * row_bytes;
    int ctas = 0;
    const cudaError_t err = resident_ctas(kern, smem, cache, &ctas);
    if (err != cudaSuccess) return cuda_fail(err, "layernorm_quantize_amax_kernel setup");
    const int64_t grid = a.rows < (int64_t)ctas ? a.rows : (int64_t)ctas;
    kern<<<(unsigned)grid, kThreads, smem, s>>>(a);
    return after_launch("layernorm_quantize_amax_kernel");
}

template <int FMT, bool WRITE_Y>
fp8q_status launch_layernorm(const LnArgs& a, cudaStream_t s) {
    const int vpt = (a.H / 16 + kThreads - 1) / kThreads;
    if (vpt <= 1) return launch_layernorm_vpt<FMT, WRITE_Y, 1>(a, s);
    if (vpt <= 2) return launch_layernorm_vpt<FMT, WRITE_Y, 2>(a, s);
    return launch_layernorm_vpt<FMT, WRITE_Y, 4>(a, s);
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
    if (fmt == FP8Q_E4M3FN) {
        if (y_bf16) gelu_quantize_amax_kernel<FP8Q_E4M3FN, true><<<grid, kThreads, 0, s>>>(a);
        else        gelu_quantize_amax_kernel<FP8Q_E4M3FN, false><<<grid, kThreads, 0, s>>>(a);
    } else {
        if (y_bf16) gelu_quantize_amax_kernel<FP8Q_E5M2, true><<<grid, kThreads, 0, s>>>(a);
        else        gelu_quantize_amax_kernel<FP8Q_E5M2, false><<<grid, kThreads, 0, s>>>(a);
    }
    return after_launch("gelu_quantize_amax_kernel");
}

fp8q_status fp8q_layernorm_quantize_amax(const void* x_bf16, void* y_bf16, uint8_t* q, int64_t rows,
                                         int32_t hidden, const float* gamma, const float* beta, float eps,
                                         fp8q_format fmt, const float* scale, float* amax, void* stream) {
    if (!valid_fmt(fmt) || rows < 0 || hidden < 16 || (hidden % 16) != 0) return FP8Q_ERR_INVALID_ARG;
    if (hidden > 16 * kThreads * kLnMaxVecPerThread) return FP8Q_ERR_UNSUPPORTED;
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
    a.stages = 0;
    a.eps = eps;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fmt == FP8Q_E4M3FN)
        return y_bf16 ? launch_layernorm<FP8Q_E4M3FN, true>(a, s) : launch_layernorm<FP8Q_E4M3FN, false>(a, s);
    return y_bf16 ? launch_layernorm<FP8Q_E5M2, true>(a, s) : launch_layernorm<FP8Q_E5M2, false>(a, s);
}

}  // extern "C"
