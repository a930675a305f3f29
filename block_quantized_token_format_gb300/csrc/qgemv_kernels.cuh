// Dequant-GEMV kernels for sm_103a: y[t][o] = sum_i dequant(W)[o][i] * x[t][i], ntok <= 4.
//
// The operator is the multi-token gemv of the Track 2 Audit & Optimization
// Report (M5 Metal kernels), section 1 item 1: every lane keeps fp32
// accumulators for its rows and all ntok activation rows, and the cost is one
// pass over the weight bytes ("Where the time goes on an M2 Max", format
// table: effective bandwidth = weight bytes / time).  The Metal tiles on those
// pages were made for Apple GPUs; this is a GB300 design:
//
//  * Persistent grid (a few CTAs per SM).  Each CTA stages x once, in fp32,
//    in shared memory with an XOR swizzle that makes the per-lane 16-column
//    reads conflict-free, so x never costs HBM traffic after the first read.
//  * Every row is streamed exactly once with 16-byte (8-bit, BF16) or 8-byte
//    (4-bit) non-allocating loads; a lane owns 16-weight chunks lane, lane+32,
//    ... of the row.  A warp walks RPW rows at once (x is read from shared
//    memory once per chunk and reused for the RPW rows) and keeps DEPTH chunk
//    sets in flight in registers, in one flat pipeline that runs across
//    row-group boundaries so the loads never drain between groups.
//  * Dequantization in registers without I2F: a code is placed in the
//    mantissa of 2^23 (byte permute or mask) and the offset is removed with
//    an exact packed FADD (two codes per add.rn.f32x2).  Block scales are
//    applied once per 16-weight chunk.
//  * FP32 math in packed pairs: per (row, token) two partial sums, even and
//    odd columns, advanced by fma.rn.f32x2 (two columns per instruction) and
//    added once per chunk.  On GB300 the packed FMA does not raise the FP32
//    rate, but it halves the instructions issued for the multiply-adds.
//    4-bit codes at nibble position 4m of a half-word come out as q*16^m; x is
//    stored pre-multiplied by 16^-m (exact), so the products are q*x exactly.
//  * The affine bias term b*sum(x) uses per-chunk sums of x computed once per
//    CTA; the per-chunk fp32 order is fixed.
//  * Reduction: per lane, chunks in increasing order; across the warp, a
//    transposed butterfly (reduce-scatter by halving, then xor steps).  The
//    order depends only on (fmt, n_in), never on ntok, RPW or the grid, so a
//    token's outputs are bitwise identical for every ntok (the opus-mtp-turbo
//    Track 1 report, item 3, relies on exactly this property).
//  * The fused argmax (perf(speculative): cut the MTP drafter's per-step
//    cost, Phase 2 item 2a) keeps a running (max, lowest index) per lane,
//    reduces it per CTA into the workspace, and the last CTA to take a ticket
//    reduces the partials.  Nothing ever waits on another CTA.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "qg_layout.h"

namespace qg {

constexpr int kMaxGrid = 4096;            // upper bound on CTAs of any launch (workspace sizing)
constexpr unsigned kFull = 0xFFFFFFFFu;

struct ArgmaxPartial { float v; int i; };

struct KernelArgs {
    const uint8_t* W;          // device layout, rows of `stride` bytes
    const float* x;            // [ntok][n_in]
    float* y;                  // [ntok][n_out], may be null for argmax-only
    int* argmax;               // [ntok] (argmax kernels)
    ArgmaxPartial* partials;   // [gridDim.x][ntok] (argmax kernels)
    unsigned int* ticket;      // zero on entry, left zero on exit (argmax kernels)
    long long stride;
    int n_out;
    int n_in;
    int pf;                    // L2 bulk-prefetch distance in row groups of this warp (0 = off)
};

// ------------------------------------------------------------------------------ loads

__device__ __forceinline__ uint4 ld_stream16(const uint8_t* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ld_stream8(const uint8_t* p) {
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_u16(const uint8_t* p) {
    unsigned short r;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_u32(const uint8_t* p) {
    uint32_t r;
    asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

// One bulk copy of [p, p + bytes) from HBM into L2 (no registers, no shared memory).
// p and bytes must be multiples of 16.
__device__ __forceinline__ void prefetch_l2(const uint8_t* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float h2f(uint32_t bits) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
}

// ------------------------------------------------------------------------------ formats
// Raw: what one lane loads for one 16-weight chunk of one row.
// load(row, n_in, c): chunk c of the row.   dec(raw, i, f): columns 4i..4i+3 as floats.

template <int FMT> struct Fmt;

template <> struct Fmt<QG_Q8_0> {
    static constexpr bool kFour = false;
    struct Raw { uint4 q; uint32_t d; };
    static __device__ __forceinline__ Raw load(const uint8_t* row, int n_in, int c) {
        Raw r;
        r.q = ld_stream16(row + 16 * c);
        r.d = ld_u16(row + n_in + 2 * (c >> 1));
        return r;
    }
    // bytes hold q + 128; 2^23 + (q + 128) - (2^23 + 128) = q, exact.
    static __device__ __forceinline__ void dec(const Raw& r, int i, float2& lo, float2& hi) {
        const uint32_t w = i == 0 ? r.q.x : i == 1 ? r.q.y : i == 2 ? r.q.z : r.q.w;
        const float2 m = make_float2(-8388736.0f, -8388736.0f);
        lo = __fadd2_rn(make_float2(__int_as_float(__byte_perm(w, 0x4B000000u, 0x7440)),
                                    __int_as_float(__byte_perm(w, 0x4B000000u, 0x7441))), m);
        hi = __fadd2_rn(make_float2(__int_as_float(__byte_perm(w, 0x4B000000u, 0x7442)),
                                    __int_as_float(__byte_perm(w, 0x4B000000u, 0x7443))), m);
    }
};

// Nibble m (bits 4m..4m+3) of a half-word h as the float 2^23 + q*16^m.
__device__ __forceinline__ float nib(uint32_t h, uint32_t mask) {
    return __int_as_float((h & mask) | 0x4B000000u);
}

template <> struct Fmt<QG_Q4_0> {
    static constexpr bool kFour = true;
    struct Raw { uint2 q; uint32_t d; };
    static __device__ __forceinline__ Raw load(const uint8_t* row, int n_in, int c) {
        Raw r;
        r.q = ld_stream8(row + 8 * c);
        r.d = ld_u16(row + n_in / 2 + 2 * (c >> 1));
        return r;
    }
    // (2^23 + q*16^m) - (2^23 + 8*16^m) = (q - 8) * 16^m, exact.
    static __device__ __forceinline__ void dec(const Raw& r, int i, float2& lo, float2& hi) {
        const uint32_t w = (i >> 1) ? r.q.y : r.q.x;
        const uint32_t h = (i & 1) ? (w >> 16) : w;
        lo = __fadd2_rn(make_float2(nib(h, 0x000Fu), nib(h, 0x00F0u)), make_float2(-8388616.0f, -8388736.0f));
        hi = __fadd2_rn(make_float2(nib(h, 0x0F00u), nib(h, 0xF000u)), make_float2(-8390656.0f, -8421376.0f));
    }
};

template <> struct Fmt<QG_AFFINE4_G64> {
    static constexpr bool kFour = true;
    struct Raw { uint2 q; uint32_t sb; };
    static __device__ __forceinline__ Raw load(const uint8_t* row, int n_in, int c) {
        Raw r;
        r.q = ld_stream8(row + 8 * c);
        r.sb = ld_u32(row + n_in / 2 + 4 * (c >> 2));
        return r;
    }
    // (2^23 + q*16^m) - 2^23 = q * 16^m, exact.
    static __device__ __forceinline__ void dec(const Raw& r, int i, float2& lo, float2& hi) {
        const uint32_t w = (i >> 1) ? r.q.y : r.q.x;
        const uint32_t h = (i & 1) ? (w >> 16) : w;
        const float2 m = make_float2(-8388608.0f, -8388608.0f);
        lo = __fadd2_rn(make_float2(nib(h, 0x000Fu), nib(h, 0x00F0u)), m);
        hi = __fadd2_rn(make_float2(nib(h, 0x0F00u), nib(h, 0xF000u)), m);
    }
};

template <> struct Fmt<QG_BF16> {
    static constexpr bool kFour = false;
    struct Raw { uint4 a; uint4 b; };
    static __device__ __forceinline__ Raw load(const uint8_t* row, int, int c) {
        Raw r;
        r.a = ld_stream16(row + 32 * c);
        r.b = ld_stream16(row + 32 * c + 16);
        return r;
    }
    static __device__ __forceinline__ void dec(const Raw& r, int i, float2& lo, float2& hi) {
        const uint32_t w0 = i == 0 ? r.a.x : i == 1 ? r.a.z : i == 2 ? r.b.x : r.b.z;
        const uint32_t w1 = i == 0 ? r.a.y : i == 1 ? r.a.w : i == 2 ? r.b.y : r.b.w;
        lo = make_float2(__int_as_float(w0 << 16), __int_as_float(w0 & 0xFFFF0000u));
        hi = make_float2(__int_as_float(w1 << 16), __int_as_float(w1 & 0xFFFF0000u));
    }
};

// ------------------------------------------------------------------------------ helpers

// Physical float4 slot of logical slot g within one token's staged x row.
__device__ __forceinline__ int xswz(int g) { return g ^ ((g >> 3) & 3); }

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

template <int V> struct Pow2Up { static constexpr int value = V <= 1 ? 1 : V <= 2 ? 2 : V <= 4 ? 4 : V <= 8 ? 8 : 16; };
template <int V> struct Log2 { static constexpr int value = V <= 1 ? 0 : 1 + Log2<V / 2>::value; };
template <> struct Log2<1> { static constexpr int value = 0; };

// ------------------------------------------------------------------------------ kernel

template <int FMT, int NTOK, int RPW, int DEPTH, bool ARGMAX>
__global__ void __launch_bounds__(256, 2) qgemv_kernel(const KernelArgs a) {
    using F = Fmt<FMT>;
    using Raw = typename F::Raw;
    constexpr int V = RPW * NTOK;                   // outputs per row group
    constexpr int VP = Pow2Up<V>::value;
    constexpr int LG = Log2<VP>::value;
    constexpr int SPAN = 32 / VP;                   // lanes sharing one reduced value

    extern __shared__ float4 smem[];
    const int n_in = a.n_in;
    const int n4 = n_in >> 2;
    const int nchunks = n_in >> 4;
    const int kmax = (nchunks + 31) >> 5;
    float4* xs = smem;                                          // [NTOK][n4], swizzled
    float* cs = reinterpret_cast<float*>(smem + NTOK * n4);     // affine: [NTOK][nchunks]

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int gw = blockIdx.x * nwarps + warp;
    const int GW = gridDim.x * nwarps;
    const int ngroups = (a.n_out + RPW - 1) / RPW;
    const int sw = (lane >> 1) & 3;

    // ---- load-side pipeline state (runs DEPTH chunk-steps ahead of compute)
    Raw buf[DEPTH][RPW];
    int gl = gw, kl = 0;
    const uint8_t* lrow[RPW];
    auto set_load_rows = [&](int g) {
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            long long row = (long long)g * RPW + r;
            if (row >= a.n_out) row = a.n_out - 1;      // tail group: re-read the last row, result dropped
            lrow[r] = a.W + row * a.stride;
        }
    };
    // Rows of group g lie in [g*RPW, g*RPW + RPW) and are contiguous in memory, so one
    // bulk prefetch brings the whole group into L2 ahead of the register loads.
    auto prefetch_group = [&](int g) {
        if (lane == 0 && g < ngroups) {
            const long long r0 = (long long)g * RPW;
            const long long r1 = r0 + RPW < a.n_out ? r0 + RPW : a.n_out;
            prefetch_l2(a.W + r0 * a.stride, uint32_t((r1 - r0) * a.stride));
        }
    };
    auto load_step = [&](Raw (&b)[RPW]) {
        if (gl < ngroups) {
            const int c = lane + 32 * kl;
            if (c < nchunks) {
#pragma unroll
                for (int r = 0; r < RPW; ++r) b[r] = F::load(lrow[r], n_in, c);
            }
        }
        if (++kl == kmax) {
            kl = 0;
            gl += GW;
            set_load_rows(gl);
            if (a.pf > 0) prefetch_group(gl + a.pf * GW);
        }
    };

    set_load_rows(gl);
    for (int j = 0; j <= a.pf && a.pf > 0; ++j) prefetch_group(gw + j * GW);
#pragma unroll
    for (int u = 0; u < DEPTH; ++u) load_step(buf[u]);

    // ---- stage x (overlaps the first weight loads)
    {
        const float4* x4 = reinterpret_cast<const float4*>(a.x);
        for (int i = threadIdx.x; i < NTOK * n4; i += blockDim.x) {
            const int t = i / n4;
            const int g = i - t * n4;
            float4 v = __ldg(x4 + i);
            if constexpr (F::kFour) {   // column j is used as q*16^(j%4): store x * 16^-(j%4)
                v.y *= 0.0625f;
                v.z *= 0.00390625f;
                v.w *= 0.000244140625f;
            }
            xs[t * n4 + xswz(g)] = v;
        }
        if constexpr (FMT == QG_AFFINE4_G64) {
            for (int i = threadIdx.x; i < NTOK * nchunks; i += blockDim.x) {
                const int t = i / nchunks;
                const int c = i - t * nchunks;
                const float4* src = x4 + t * n4 + 4 * c;
                float s = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 v = __ldg(src + q);
                    s = __fadd_rn(s, v.x); s = __fadd_rn(s, v.y); s = __fadd_rn(s, v.z); s = __fadd_rn(s, v.w);
                }
                cs[i] = s;
            }
        }
    }
    __syncthreads();

    float best_v = -INFINITY;
    int best_i = 0x7FFFFFFF;

    // Per (row, token): within a chunk, a pair of fp32 partial sums (even and odd
    // columns) advanced with packed fma.rn.f32x2, two columns per instruction; the
    // pair is added and scaled once per chunk into one fp32 accumulator.  BF16 has
    // no scale and keeps the pair across the whole row.
    constexpr bool kPairAcc = (FMT == QG_BF16);
    float acc[RPW][NTOK];
    float2 acc2[kPairAcc ? RPW : 1][kPairAcc ? NTOK : 1];
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int t = 0; t < NTOK; ++t) acc[r][t] = 0.f;
#pragma unroll
    for (int r = 0; r < (kPairAcc ? RPW : 1); ++r)
#pragma unroll
        for (int t = 0; t < (kPairAcc ? NTOK : 1); ++t) acc2[r][t] = make_float2(0.f, 0.f);

    int gc = gw, kc = 0;
    while (gc < ngroups) {
#pragma unroll
        for (int u = 0; u < DEPTH; ++u) {
            if (gc < ngroups) {
                const int c = lane + 32 * kc;
                if (c < nchunks) {
                    // ---- one 16-weight chunk of RPW rows against NTOK tokens
                    const float4* xr = xs + 4 * c;
                    float2 p[kPairAcc ? 1 : RPW][kPairAcc ? 1 : NTOK];
#pragma unroll
                    for (int r = 0; r < (kPairAcc ? 1 : RPW); ++r)
#pragma unroll
                        for (int t = 0; t < (kPairAcc ? 1 : NTOK); ++t) p[r][t] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float4 xv[NTOK];
#pragma unroll
                        for (int t = 0; t < NTOK; ++t) xv[t] = xr[t * n4 + (i ^ sw)];
#pragma unroll
                        for (int r = 0; r < RPW; ++r) {
                            float2 wlo, whi;
                            F::dec(buf[u][r], i, wlo, whi);
#pragma unroll
                            for (int t = 0; t < NTOK; ++t) {
                                float2& pp = [&]() -> float2& {
                                    if constexpr (kPairAcc) return acc2[r][t]; else return p[r][t];
                                }();
                                pp = __ffma2_rn(wlo, make_float2(xv[t].x, xv[t].y), pp);
                                pp = __ffma2_rn(whi, make_float2(xv[t].z, xv[t].w), pp);
                            }
                        }
                    }
                    if constexpr (FMT == QG_Q8_0 || FMT == QG_Q4_0) {
#pragma unroll
                        for (int r = 0; r < RPW; ++r) {
                            const float d = h2f(buf[u][r].d);
#pragma unroll
                            for (int t = 0; t < NTOK; ++t)
                                acc[r][t] = __fmaf_rn(d, __fadd_rn(p[r][t].x, p[r][t].y), acc[r][t]);
                        }
                    } else if constexpr (FMT == QG_AFFINE4_G64) {
                        float csv[NTOK];
#pragma unroll
                        for (int t = 0; t < NTOK; ++t) csv[t] = cs[t * nchunks + c];
#pragma unroll
                        for (int r = 0; r < RPW; ++r) {
                            const uint32_t sb = buf[u][r].sb;
                            const float sc = h2f(sb & 0xFFFFu), b = h2f(sb >> 16);
#pragma unroll
                            for (int t = 0; t < NTOK; ++t)
                                acc[r][t] = __fmaf_rn(sc, __fadd_rn(p[r][t].x, p[r][t].y), __fmaf_rn(b, csv[t], acc[r][t]));
                        }
                    }
                }
                load_step(buf[u]);
                if (++kc == kmax) {
                    // ---- finish the row group: transposed warp reduction
                    float v[VP];
#pragma unroll
                    for (int j = 0; j < VP; ++j) {
                        if constexpr (kPairAcc)
                            v[j] = j < V ? __fadd_rn(acc2[j / NTOK][j % NTOK].x, acc2[j / NTOK][j % NTOK].y) : 0.f;
                        else
                            v[j] = j < V ? acc[j / NTOK][j % NTOK] : 0.f;
                    }
#pragma unroll
                    for (int s = 0; s < LG; ++s) {
                        const int h = VP >> (s + 1);
                        const int mask = 16 >> s;
                        const bool upper = (lane & mask) != 0;
#pragma unroll
                        for (int j = 0; j < h; ++j) {
                            const float send = upper ? v[j] : v[j + h];
                            const float keep = upper ? v[j + h] : v[j];
                            v[j] = keep + __shfl_xor_sync(kFull, send, mask);
                        }
                    }
#pragma unroll
                    for (int mask = 16 >> LG; mask >= 1; mask >>= 1) v[0] += __shfl_xor_sync(kFull, v[0], mask);
                    const int vi = lane / SPAN;                       // value index this lane holds
                    if (vi < V && (lane % SPAN) == 0) {
                        const int r = vi / NTOK, t = vi - r * NTOK;
                        const long long row = (long long)gc * RPW + r;
                        if (row < a.n_out) {
                            if (!ARGMAX || a.y) a.y[(long long)t * a.n_out + row] = v[0];
                            if (ARGMAX && better(v[0], int(row), best_v, best_i)) { best_v = v[0]; best_i = int(row); }
                        }
                    }
#pragma unroll
                    for (int r = 0; r < RPW; ++r)
#pragma unroll
                        for (int t = 0; t < NTOK; ++t) acc[r][t] = 0.f;
#pragma unroll
                    for (int r = 0; r < (kPairAcc ? RPW : 1); ++r)
#pragma unroll
                        for (int t = 0; t < (kPairAcc ? NTOK : 1); ++t) acc2[r][t] = make_float2(0.f, 0.f);
                    kc = 0;
                    gc += GW;
                }
            }
        }
    }

    if constexpr (ARGMAX) {
        // ---- per-token argmax: warp -> CTA partial -> last CTA reduces all partials
        __shared__ ArgmaxPartial wbest[16][kMaxNtok];
        __shared__ bool last_cta;
        const int vi = lane / SPAN;
        const int my_t = (vi < V && (lane % SPAN) == 0) ? vi % NTOK : -1;
#pragma unroll
        for (int t = 0; t < NTOK; ++t) {
            float bv = (my_t == t) ? best_v : -INFINITY;
            int bi = (my_t == t) ? best_i : 0x7FFFFFFF;
#pragma unroll
            for (int mask = 16; mask >= 1; mask >>= 1) {
                const float ov = __shfl_xor_sync(kFull, bv, mask);
                const int oi = __shfl_xor_sync(kFull, bi, mask);
                if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
            }
            if (lane == 0) wbest[warp][t] = {bv, bi};
        }
        __syncthreads();
        if (threadIdx.x < NTOK) {
            const int t = threadIdx.x;
            ArgmaxPartial b = wbest[0][t];
            for (int w = 1; w < nwarps; ++w)
                if (better(wbest[w][t].v, wbest[w][t].i, b.v, b.i)) b = wbest[w][t];
            a.partials[blockIdx.x * NTOK + t] = b;
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) last_cta = (atomicAdd(a.ticket, 1u) == gridDim.x - 1);
        __syncthreads();
        if (last_cta) {
            __threadfence();
            for (int t = warp; t < NTOK; t += nwarps) {
                float bv = -INFINITY;
                int bi = 0x7FFFFFFF;
                for (int b = lane; b < (int)gridDim.x; b += 32) {
                    const float pv = __ldcg(&a.partials[b * NTOK + t].v);
                    const int pi = __ldcg(&a.partials[b * NTOK + t].i);
                    if (better(pv, pi, bv, bi)) { bv = pv; bi = pi; }
                }
#pragma unroll
                for (int mask = 16; mask >= 1; mask >>= 1) {
                    const float ov = __shfl_xor_sync(kFull, bv, mask);
                    const int oi = __shfl_xor_sync(kFull, bi, mask);
                    if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
                }
                if (lane == 0) a.argmax[t] = (bi == 0x7FFFFFFF) ? -1 : bi;
            }
            if (threadIdx.x == 0) *a.ticket = 0u;   // ready for the next call on this workspace
        }
    }
}

// Shared memory bytes of one CTA.
inline size_t smem_bytes(int fmt, int ntok, int n_in) {
    size_t b = size_t(ntok) * size_t(n_in) * 4;
    if (fmt == QG_AFFINE4_G64) b += size_t(ntok) * size_t(n_in / 16) * 4;
    return b;
}

// Lookup of an instantiated kernel (defined in the per-format instantiation units).
const void* kernel_lookup(int fmt, int ntok, int rpw, int depth, bool argmax);

}  // namespace qg
