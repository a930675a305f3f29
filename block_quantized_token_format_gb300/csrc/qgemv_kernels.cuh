// Dequant-GEMV kernels for sm_103a: y[t][o] = sum_i dequant(W)[o][i] * x[t][i], ntok <= 4.
//
// The operator is the multi-token gemv of the Track 2 Audit & Optimization
// Report (M5 Metal kernels), section 1 item 1: every lane keeps fp32
// accumulators for its rows and all ntok activation rows, and the cost is one
// pass over the weight bytes ("Where the time goes on an M2 Max", format
// table: effective bandwidth = weight bytes / time).  The Metal tiles on those
// pages were made for Apple GPUs; this is a GB300 design:
//
//  * Persistent grid (a few CTAs per SM).  Each CTA stages x once in shared
//    memory (16-bit integers for the integer chunk dot, fp32 for BF16), chunk by
//    chunk with an odd chunk stride that makes the lanes' loads conflict-free,
//    so x never costs HBM traffic after the first read.
//  * Weights move HBM -> shared memory by TMA tensor copies
//    (cp.async.bulk.tensor.2d, completion counted on an mbarrier), never
//    through registers: each warp owns a ring of `depth` stages, a stage holds
//    one 512-byte code step (plus its scales) of each of the warp's RPW rows,
//    fetched as ONE box of RPW rows x one step (the tensor map views the packed
//    matrix as [n_out][row stride / 8] 8-byte elements), so one thread issues
//    one copy per step whatever RPW is.  Rows past n_out and the bytes past a
//    short last step are outside the tensor and arrive as zeros without being
//    read.  The bytes in flight per SM are set by shared memory, not by
//    registers, and every weight byte is read exactly once.  One flat pipeline
//    runs across row-group boundaries, so the copies never drain between groups.
//  * Q8_0, Q4_0, Q5_0 and affine 4-bit: integer chunk dots.  x is staged per
//    chunk (32 columns, 16 for Q8_0) and token as 16-bit integers
//    X = rn(x * 2^(15-k)) capped at 32767, with 2^(k-1) <= max|x| < 2^k (error
//    <= 2^-14 of the chunk's largest |x|, 2^-15 where the cap does not act);
//    codes become bytes (Q8_0's stored
//    q + 128 as they are; a nibble word's even codes by one mask, its odd codes
//    by one shift and mask, Q5_0's fifth bits merged from the chunk's record),
//    and dp2a (16-bit x 8-bit pairs into int32, exact) takes two products per
//    instruction.  Per chunk one I2F and one FMA with scale * 2^(k-15).  On
//    GB300 this issues about half the instructions of a magic-float decode
//    with packed FP32 FMAs, whose issue cost bound the quantized formats at
//    ntok 3-4 (measured: a register-only model of the 4-bit ntok-4 inner loop
//    reaches 27 weights/clk/SM against 18 with packed FP32).
//  * BF16: codes widened to fp32 by shifts and masks.
//  * BF16 math in packed pairs: per (row, token) a pair of partial sums (even
//    and odd columns) advanced by fma.rn.f32x2.  On GB300 the packed FMA does
//    not raise the FP32 rate, but it halves the instructions issued.
//  * The affine bias term b*sum(x) uses per-chunk fp32 sums of x computed once
//    per CTA in a fixed order.
//  * Reduction: per lane, chunks in increasing order; across the warp, a
//    transposed butterfly (reduce-scatter by halving, then xor steps); where a
//    row's steps are split over a team of warps, the segments' sums in segment
//    order.  The order depends only on (fmt, n_out, n_in), never on ntok, the
//    tile or the grid, so a token's outputs are bitwise identical for every ntok
//    (the opus-mtp-turbo Track 1 report, item 3, relies on exactly this property).
//  * The fused argmax (perf(speculative): cut the MTP drafter's per-step
//    cost, Phase 2 item 2a) keeps a running (max, lowest index) per lane,
//    reduces it per CTA into the workspace, and the last CTA to take a ticket
//    reduces the partials.  No CTA ever waits on another CTA.
//  * Every mbarrier wait is bounded: after `wait_limit` polls it sets bit 0 of
//    the device status word, stops issuing copies, drains (again bounded) the
//    copies it already issued, and the kernel runs to its normal exit.
#pragma once

#include <cuda.h>            // CUtensorMap (type only; the library does not link the driver API)
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "qg_layout.h"

namespace qg {

constexpr int kMaxGrid = 4096;            // upper bound on CTAs of any launch (workspace sizing)
constexpr int kMaxWarps = 16;             // warps per CTA (launch bound 512 threads)
constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr uint32_t kWaitLimit = 1u << 22; // mbarrier polls before a wait is declared failed
constexpr unsigned kStatusWaitTimeout = 1u;
constexpr unsigned kStatusBadRowId = 2u;    // a row gather met an id outside the head

struct ArgmaxPartial { float v; int i; };

struct KernelArgs {
    CUtensorMap wmap;          // the packed weights as a 2-D tensor [n_out][stride / 8] of 8-byte
                               // elements, box = one full step x RPW rows, zero fill outside
    const float* x;            // [ntok][n_in]
    float* y;                  // [ntok][n_out], may be null for argmax-only
    int* argmax;               // [ntok] (argmax kernels)
    const int32_t* row_ids;    // optional [n_out]: the argmax is written as row_ids[winning row]
                               // (a draft head gathered from a full head: back to full ids)
    ArgmaxPartial* partials;   // [gridDim.x][ntok] (argmax kernels)
    unsigned int* ticket;      // zero on entry, left zero on exit (argmax kernels)
    unsigned int* status;      // device status word (bit 0: a bounded wait gave up)
    int n_out;
    int n_in;
    int depth;                 // ring stages per warp
    int pre;                   // stages each warp requests before the wait (1..depth), the
                               // rest once x is staged
    int split;                 // warps per team: a row group's steps are split into this many
                               // segments, one per team warp (1 = no split)
    int seg_len;               // steps per segment (the last one may be shorter)
    uint32_t wait_limit;       // polls per mbarrier wait before giving up
    uint32_t drain_limit;      // polls per wait while draining after giving up
    uint32_t test_extra_tx;    // test hook: bytes added to the first expected transaction of
                               // every warp, so that wait can never complete (0 = off)
    uint32_t stage_tx;         // bytes one box delivers: RPW x full step (zero fill included)
    unsigned long long* phase; // profiling: this launch's slot of per-CTA phase stamps, or null
};

// ------------------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ unsigned int sm_id() {
    unsigned int v;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(v));
    return v;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait: false if the phase did not complete within `limit` polls.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Tensor copy of the box at element coordinates (x, y) of the 2-D tensor map at
// `map` (a kernel parameter) into this CTA's shared memory, completion counted
// on `bar`.  x * 8 bytes is a multiple of 16 (x is a multiple of a step's
// element count, and steps are multiples of 16 bytes).
// The weights are read once per call: the copy carries an L2 evict-first policy so
// that the stream does not push x, y and other recently written data out of L2.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, int x, int y, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy) : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
    return r;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
    unsigned short r;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(r) : "r"(a));
    return r;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t r;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(a));
    return r;
}

__device__ __forceinline__ float h2f(uint32_t bits) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
}

// A pair of fp32 values in one 64-bit register pair, as the packed f32x2
// instructions take them.  Keeping pairs as 64-bit PTX values lets ptxas build
// each pair in place (no register moves to assemble operands).
typedef unsigned long long f2_t;
__device__ __forceinline__ f2_t f2_pack(uint32_t lo, uint32_t hi) {
    f2_t d;
    asm("mov.b64 %0, {%1,%2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}
__device__ __forceinline__ f2_t f2_fma(f2_t a, f2_t b, f2_t c) {
    f2_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// lo + hi of a pair, in that order.
__device__ __forceinline__ float f2_sum(f2_t a) {
    float x, y;
    asm("mov.b64 {%0,%1}, %2;" : "=f"(x), "=f"(y) : "l"(a));
    return __fadd_rn(x, y);
}
// Two consecutive pairs (four floats) from shared memory.
__device__ __forceinline__ void lds_f2x2(uint32_t a, f2_t& p0, f2_t& p1) {
    asm volatile("ld.shared.v2.b64 {%0,%1}, [%2];" : "=l"(p0), "=l"(p1) : "r"(a));
}

// ------------------------------------------------------------------------------ formats
// A lane's chunk is 16 bytes of codes.  kW: weights per chunk; kW / 4 float4
// slots of x per chunk.  dec(q, i, lo, hi): columns 4i..4i+3 of the chunk as
// two pairs.  The scale word of chunk j of a step sits scale_off(j) bytes after
// the step's codes; scale(addr) loads it.

template <int FMT> struct Fmt;

template <> struct Fmt<QG_Q8_0> {
    static constexpr int kW = 16;
    static constexpr int kStepScale = 32;
    static __device__ __forceinline__ uint32_t scale_off(int j) { return 2u * uint32_t(j >> 1); }
    static __device__ __forceinline__ uint32_t scale(uint32_t a) { return lds16(a); }
};

// Q4_0 and the affine format run the integer chunk dot (step_idp); their traits give the
// chunk width and where the scales sit.
template <> struct Fmt<QG_Q4_0> {
    static constexpr int kW = 32;
    static constexpr int kStepScale = 64;
    static __device__ __forceinline__ uint32_t scale_off(int j) { return 2u * uint32_t(j); }
    static __device__ __forceinline__ uint32_t scale(uint32_t a) { return lds16(a); }
};

template <> struct Fmt<QG_AFFINE4_G64> {
    static constexpr int kW = 32;
    static constexpr int kStepScale = 64;
    static __device__ __forceinline__ uint32_t scale_off(int j) { return 4u * uint32_t(j >> 1); }
    static __device__ __forceinline__ uint32_t scale(uint32_t a) { return lds32(a); }
};

template <> struct Fmt<QG_BF16> {
    static constexpr int kW = 8;
    static constexpr int kStepScale = 0;
    static __device__ __forceinline__ uint32_t scale_off(int) { return 0u; }
    static __device__ __forceinline__ uint32_t scale(uint32_t) { return 0u; }
    static __device__ __forceinline__ void dec(const uint4& q, int i, f2_t& lo, f2_t& hi) {
        const uint32_t w0 = i == 0 ? q.x : q.z;
        const uint32_t w1 = i == 0 ? q.y : q.w;
        lo = f2_pack(w0 << 16, w0 & 0xFFFF0000u);
        hi = f2_pack(w1 << 16, w1 & 0xFFFF0000u);
    }
};

// Q5_0: the Q4_0 nibbles plus a fifth bit per element.  A chunk's scale record (6 bytes at
// 6j after the step's codes) holds its fifth bits (uint32, element e at bit 8b + g with
// g = 2 (e / 8) + e % 2 and b = (e % 8) / 2) and then its fp16 d.
template <> struct Fmt<QG_Q5_0> {
    static constexpr int kW = 32;
    static constexpr int kStepScale = 192;
    static __device__ __forceinline__ uint32_t scale_off(int j) { return 6u * uint32_t(j); }
    static __device__ __forceinline__ uint32_t scale(uint32_t a) { return lds16(a + 4); }
    static __device__ __forceinline__ uint32_t high(uint32_t a) { return lds16(a) | (lds16(a + 2) << 16); }
};

// Formats that run the integer chunk dot (x staged as 16-bit integers).
__host__ __device__ constexpr bool idp_format(int fmt) {
    return fmt == QG_Q8_0 || fmt == QG_Q4_0 || fmt == QG_AFFINE4_G64 || fmt == QG_Q5_0;
}
template <int FMT> struct IsIdp { static constexpr bool value = idp_format(FMT); };

// 16-byte slots of staged x per chunk and token: the chunk's columns as fp32 (BF16, 8
// columns), or as 16-bit integers for the integer dot (Q8_0 16, the 4- and 5-bit
// formats 32 columns).
__host__ __device__ constexpr int x_slots(int fmt) {
    return fmt == QG_Q8_0 ? 2 : idp_format(fmt) ? 4 : 2;
}
// Pad slots after a chunk's staged x.  Integer dot: slot 0 holds per token the chunk's
// scale 2^(k-15), slot 1 per token the starting sum that removes the code offset
// (Q8_0 -128 * sum(X), Q4_0 -8 * sum(X), Q5_0 -16 * sum(X), int32) or the affine
// bias's sum(x) (fp32); slot 2 pads the stride to an odd count.  BF16: one slot
// (unused but for the odd stride).
__host__ __device__ constexpr int x_pad_slots(int fmt) { return idp_format(fmt) ? 3 : 1; }

// ------------------------------------------------------------------------------ helpers

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

template <int V> struct Pow2Up {
    static_assert(V >= 1 && V <= 32, "a warp reduces at most 32 outputs per row group");
    static constexpr int value = V <= 1 ? 1 : V <= 2 ? 2 : V <= 4 ? 4 : V <= 8 ? 8 : V <= 16 ? 16 : 32;
};
template <int V> struct Log2 { static constexpr int value = V <= 1 ? 0 : 1 + Log2<V / 2>::value; };
template <> struct Log2<1> { static constexpr int value = 0; };

// Shared memory layout of one CTA (bytes): staged x, the warps' mbarriers, the
// warps' rings.  x is stored chunk by chunk: for lane-chunk c, the NTOK*S float4
// slots of its columns (token-major), then the pad slots (x_pad_slots).  The chunk
// stride of NTOK*S + pad slots is odd, so the 8 lanes of a 128-byte shared-memory
// phase hit 8 distinct 16-byte bank groups, and every load offset is a
// compile-time constant.
struct SmemPlan {
    int x_bytes, bar_off, tbar_off, xch_off, ring_off, total;
};

// One ring stage: RPW rows of one full step, rounded up to 128 bytes (tensor
// copies land on 128-byte boundaries).
__host__ __device__ constexpr int full_step(int fmt) {
    return int(kStepCodeBytes) + (fmt == QG_Q8_0 ? 32 : fmt == QG_BF16 ? 0 : fmt == QG_Q5_0 ? 192 : 64);
}
__host__ __device__ constexpr int stage_bytes(int fmt, int rpw) { return (rpw * full_step(fmt) + 127) / 128 * 128; }

// With a split of P > 1, each team of P warps also has four mbarriers (full and
// empty, two parities) and an exchange area of 2 x (P - 1) x 32 floats for the
// reduced values of its segments.
__host__ __device__ inline SmemPlan smem_plan(int fmt, int ntok, int n_in, int rpw, int depth, int warps,
                                              int split) {
    SmemPlan p;
    const int slots = x_slots(fmt);
    const int teams = split > 1 ? warps / split : 0;
    // x holds whole steps of chunks (32 per step), zero past n_in.
    const int codes = fmt == QG_Q8_0 ? n_in : fmt == QG_BF16 ? 2 * n_in : n_in / 2;
    p.x_bytes = (codes + 511) / 512 * 32 * (ntok * slots + x_pad_slots(fmt)) * 16;
    p.bar_off = (p.x_bytes + 15) / 16 * 16;
    p.tbar_off = p.bar_off + warps * depth * 8;
    p.xch_off = p.tbar_off + teams * 32;
    p.ring_off = (p.xch_off + teams * 2 * (split - 1) * 32 * 4 + 127) / 128 * 128;
    // + 128: the kernel rounds the ring's shared-memory ADDRESS up to 128 bytes
    // (the dynamic shared memory base itself may be less aligned).
    p.total = p.ring_off + warps * depth * stage_bytes(fmt, rpw) + 128;
    return p;
}

// ------------------------------------------------------------------------------ kernel pieces
// Shared by the mat-vec kernel and the expert-grouped kernel.

// max(a, b) that returns NaN when either input is NaN (fmaxf would return the other).
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// The rounding of one (chunk, token) pair of x for the integer chunk dot: with
// m = max|v| over the chunk's W values and 2^(k-1) <= m < 2^k, y[i] = 1.5 * 2^23 + X_i
// where X_i = rn(v_i * 2^(15-k)) capped at 32767 (formed exactly by one FMA: the integer
// sits in the low bits of the sum, round to nearest even; a value within 2^-16 m of 2^k
// rounds to 2^15, which int16 cannot hold), so -2^15 <= X_i < 2^15 and
// |v_i - X_i 2^(k-15)| <= 2^(k-15) <= 2^-14 m (half that where the cap does not act).
// down = 2^(k-15) (0 for a chunk with m < 2^-112, staged as zero; NaN where a value is
// not finite), sx = the fp32 sum of v in column order, sX = the sum of X (exact; y lies
// in [2^23, 2^24), so its bits are 0x4B400000 + X and the integer sum of the bits gives
// it).  NAN_MAX: m by a NaN-propagating max, so one test of m finds a NaN or an
// infinity; otherwise (the affine format) a test per value — the two give the same
// results, but with the NaN max the affine LM-head kernel at ntok 4 was allocated 116
// registers instead of 122 and ran 3.6% slower (same-box A/B), while the other formats'
// small launches ran 0.5-1.8% faster.
template <int W, bool NAN_MAX>
__device__ __forceinline__ void round_chunk(const float (&v)[W], float (&y)[W], float& down, float& sx,
                                            uint32_t& sX) {
    float m = 0.f;
    sx = 0.f;
    bool finite = true;
#pragma unroll
    for (int i = 0; i < W; ++i) {
        if constexpr (NAN_MAX) {
            m = fmax_nan(m, fabsf(v[i]));
        } else {
            m = fmaxf(m, fabsf(v[i]));
            finite = finite && (fabsf(v[i]) <= 3.402823466e38f);
        }
        sx = __fadd_rn(sx, v[i]);
    }
    if constexpr (NAN_MAX) finite = m <= 3.402823466e38f;
    const int e = int(__float_as_uint(m) >> 23);           // m in [2^(e-127), 2^(e-126))
    const bool live_chunk = e >= 15;
    // 2^(15-k) = 2^(141-e) and 2^(k-15) = 2^(e-141), k = e - 126, as float bits
    const float up = live_chunk ? __uint_as_float(uint32_t(268 - e) << 23) : 0.f;
    down = live_chunk ? __uint_as_float(uint32_t(e - 14) << 23) : 0.f;
    if (!finite) down = __uint_as_float(0x7FC00000u);
    uint32_t bits = 0u;
#pragma unroll
    for (int i = 0; i < W; ++i) {
        y[i] = fminf(__fmaf_rn(v[i], up, 12582912.0f), 12615679.0f);   // 1.5 * 2^23 + X, X <= 32767
        bits += __float_as_uint(y[i]);
    }
    sX = bits - uint32_t(W) * 0x4B400000u;                 // modulo 2^32: the exact sum of X
}

// Stage x rows[0..live-1] (each n_in fp32, 16-byte aligned) into the chunk-interleaved
// layout for NTOK tokens at `smem` (see SmemPlan), zero past n_in up to whole steps;
// the slots of tokens live..NTOK-1 are left as they are.  Each thread issues all its
// loads of a batch before its first store, so staging costs about one L2 round trip,
// not one per float4; token and chunk indices come from the loop structure and shifts
// (S is a power of two), not from divisions.  Ends without a barrier: the caller
// synchronizes the CTA before the staged x is read.
template <int FMT, int NTOK, bool NC = true>
__device__ __forceinline__ void stage_x(unsigned char* smem, const float4* const (&rows)[NTOK], int n_in, int spr,
                                        int live = NTOK) {
    // NC: x is read-only for the kernel's lifetime (non-coherent loads); otherwise x
    // was written earlier in this kernel by other CTAs (L2 loads).
    auto ld = [](const float4* p) { if constexpr (NC) return __ldg(p); else return __ldcg(p); };
    constexpr int S = x_slots(FMT);
    constexpr int kCS = NTOK * S + x_pad_slots(FMT);
    float4* xs = reinterpret_cast<float4*>(smem);
    const int n4 = n_in >> 2;
    const int nchunks = n_in / Fmt<FMT>::kW;
    const int nt = int(blockDim.x);
    if constexpr (IsIdp<FMT>::value) {
        // One (chunk, token) pair per thread and pass: the chunk's values (32 columns, 16
        // for Q8_0) are loaded at once and rounded to 16-bit integers X (round_chunk).  X
        // is stored as the 16-bit pairs dp2a takes: per word of 8 nibble codes (x0|x2,
        // x4|x6, x1|x3, x5|x7) against its even and odd codes, per word of 4 byte codes
        // (x0|x1, x2|x3).  A chunk with m < 2^-112 is staged as zero (an absolute error
        // below 2^-112); one with a NaN or an infinity gets a NaN scale.
        constexpr int W = Fmt<FMT>::kW;                         // columns per chunk: 16 or 32
        uint32_t* xu = reinterpret_cast<uint32_t*>(smem);
        const int npairs = live * nchunks;
        // The (chunk, token) pair's row of x and its first float4.
        auto src_of = [&](int idx, int& t, int& c) {
            t = int(idx >= nchunks) + int(idx >= 2 * nchunks) + int(idx >= 3 * nchunks);
            c = idx - t * nchunks;
            const float4* rt = rows[0];
#pragma unroll
            for (int u = 1; u < NTOK; ++u) rt = (t == u) ? rows[u] : rt;
            return rt + (W / 4) * c;
        };
        // Round, pack and store one pair's values.
        auto put = [&](const float (&v)[W], int t, int c) {
            float y[W];
            float down, sx;
            uint32_t sX;
            round_chunk<W, FMT != QG_AFFINE4_G64>(v, y, down, sx, sX);
            uint32_t* dst = xu + (c * kCS + t * S) * 4;
            if constexpr (FMT == QG_Q8_0) {
                // byte codes: the pairs in column order, (x0|x1, x2|x3) per word of 4 codes
#pragma unroll
                for (int j = 0; j < W / 2; ++j)
                    dst[j] = __byte_perm(__float_as_uint(y[2 * j]), __float_as_uint(y[2 * j + 1]), 0x5410);
            } else {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float* yw = y + 8 * w;
                    dst[4 * w + 0] = __byte_perm(__float_as_uint(yw[0]), __float_as_uint(yw[2]), 0x5410);
                    dst[4 * w + 1] = __byte_perm(__float_as_uint(yw[4]), __float_as_uint(yw[6]), 0x5410);
                    dst[4 * w + 2] = __byte_perm(__float_as_uint(yw[1]), __float_as_uint(yw[3]), 0x5410);
                    dst[4 * w + 3] = __byte_perm(__float_as_uint(yw[5]), __float_as_uint(yw[7]), 0x5410);
                }
            }
            uint32_t* pad = xu + (c * kCS + NTOK * S) * 4;
            pad[t] = __float_as_uint(down);
            if constexpr (FMT == QG_Q8_0) pad[4 + t] = sX * uint32_t(-128);
            else if constexpr (FMT == QG_Q4_0) pad[4 + t] = sX * uint32_t(-8);
            else if constexpr (FMT == QG_Q5_0) pad[4 + t] = sX * uint32_t(-16);
            else pad[4 + t] = __float_as_uint(sx);
        };
        // Two pairs per thread and pass, both pairs' loads issued before either is
        // rounded (one L2 round trip where a CTA has up to twice as many pairs as threads).
        for (int i0 = threadIdx.x; i0 < npairs; i0 += 2 * nt) {
            const int i1 = i0 + nt;
            int t0, c0, t1 = 0, c1 = 0;
            const float4* s0 = src_of(i0, t0, c0);
            const float4* s1 = i1 < npairs ? src_of(i1, t1, c1) : s0;
            float v0[W], v1[W];
#pragma unroll
            for (int q = 0; q < W / 4; ++q) {
                const float4 f = ld(s0 + q);
                v0[4 * q] = f.x; v0[4 * q + 1] = f.y; v0[4 * q + 2] = f.z; v0[4 * q + 3] = f.w;
            }
#pragma unroll
            for (int q = 0; q < W / 4; ++q) {
                const float4 f = ld(s1 + q);
                v1[4 * q] = f.x; v1[4 * q + 1] = f.y; v1[4 * q + 2] = f.z; v1[4 * q + 3] = f.w;
            }
            put(v0, t0, c0);
            if (i1 < npairs) put(v1, t1, c1);
        }
        for (int i = nchunks * kCS + int(threadIdx.x); i < spr * 32 * kCS; i += int(blockDim.x))
            xs[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    constexpr int kXG = NTOK >= 8 ? 1 : 8 / NTOK;   // float4 columns per thread and batch
    for (int g0 = threadIdx.x; g0 < n4; g0 += kXG * nt) {
        float4 v[kXG][NTOK];
#pragma unroll
        for (int j = 0; j < kXG; ++j) {
            const int g = g0 + j * nt;
#pragma unroll
            for (int t = 0; t < NTOK; ++t)
                if (g < n4 && t < live) v[j][t] = ld(rows[t] + g);
        }
#pragma unroll
        for (int j = 0; j < kXG; ++j) {
            const int g = g0 + j * nt;
            if (g < n4) {
                float4* dst = xs + (g / S) * kCS + (g % S);
#pragma unroll
                for (int t = 0; t < NTOK; ++t) {
                    if (t >= live) break;
                    dst[t * S] = v[j][t];
                }
            }
        }
    }
    // Chunks past n_in (the lanes past a row's short last step) read as zero.
    for (int i = nchunks * kCS + int(threadIdx.x); i < spr * 32 * kCS; i += int(blockDim.x))
        xs[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// A lane's accumulators for one row group: per (row, token) one fp32 sum of scaled
// chunk sums, or (BF16, no scales) a pair of partial sums over the whole row.
// A lane's accumulators for one row group: per (row, token) one fp32 sum of scaled
// chunk sums, or (BF16, no scales) a pair of partial sums over the whole row.
template <int FMT, int NTOK, int RPW> struct Acc {
    static constexpr bool kPair = (FMT == QG_BF16);
    float s[RPW][NTOK];
    f2_t p[kPair ? RPW : 1][kPair ? NTOK : 1];
    __device__ __forceinline__ void clear() {
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int t = 0; t < NTOK; ++t) s[r][t] = 0.f;
#pragma unroll
        for (int r = 0; r < (kPair ? RPW : 1); ++r)
#pragma unroll
            for (int t = 0; t < (kPair ? NTOK : 1); ++t) p[r][t] = 0ull;
    }
    // The lane's sum for output j = r * NTOK + t (j < RPW * NTOK).
    __device__ __forceinline__ float value(int j) const {
        if constexpr (kPair) return f2_sum(p[j / NTOK][j % NTOK]);
        else return s[j / NTOK][j % NTOK];
    }
};

// One ring stage into the accumulators: the lane's 16-byte code chunk of each of the
// RPW rows (at `codes` + r * full step), the chunk's scale word (at `scales` + r * full
// step), the lane's staged x chunk at `xr` (a layout for XT >= NTOK tokens; tokens
// 0..NTOK-1 are used).  Within the chunk a pair of partial sums (even / odd columns)
// per (row, token) is advanced by packed FMAs, then added and scaled once.
template <int FMT, int NTOK, int RPW, int XT>
__device__ __forceinline__ void step_fp(Acc<FMT, NTOK, RPW>& A, uint32_t xr, uint32_t codes, uint32_t scales) {
    using F = Fmt<FMT>;
    constexpr int S = x_slots(FMT);
    constexpr int kFullStep = int(kStepCodeBytes) + F::kStepScale;
    constexpr bool kPairAcc = Acc<FMT, NTOK, RPW>::kPair;
    uint4 qv[RPW];
    uint32_t sv[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        qv[r] = lds128(codes + r * kFullStep);
        sv[r] = F::scale(scales + r * kFullStep);
    }
    f2_t p[kPairAcc ? 1 : RPW][kPairAcc ? 1 : NTOK];
#pragma unroll
    for (int r = 0; r < (kPairAcc ? 1 : RPW); ++r)
#pragma unroll
        for (int t = 0; t < (kPairAcc ? 1 : NTOK); ++t) p[r][t] = 0ull;
#pragma unroll
    for (int i = 0; i < S; ++i) {
        f2_t x01[NTOK], x23[NTOK];
#pragma unroll
        for (int t = 0; t < NTOK; ++t) lds_f2x2(xr + 16u * uint32_t(t * S + i), x01[t], x23[t]);
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            f2_t wlo, whi;
            F::dec(qv[r], i, wlo, whi);
#pragma unroll
            for (int t = 0; t < NTOK; ++t) {
                f2_t& pp = [&]() -> f2_t& {
                    if constexpr (kPairAcc) return A.p[r][t]; else return p[r][t];
                }();
                pp = f2_fma(wlo, x01[t], pp);
                pp = f2_fma(whi, x23[t], pp);
            }
        }
    }
}

// Integer chunk dot (Q8_0, Q4_0, Q5_0, affine).  Q4_0 / Q5_0 / affine: the lane's
// 16-byte chunk of each of the RPW rows is 4 words of 8 codes; a word gives its even
// codes as 4 bytes (w & 0x0F0F0F0F) and its odd codes (w >> 4 & 0x0F0F0F0F), Q5_0 ORs
// in each group's fifth bits (the record word shifted by 4 - g, masked to bit 4 of
// each byte), and per token four dp2a add the 8 products of the word's staged 16-bit x
// pairs into an int32 (exact).  Q8_0: the chunk is 16 byte codes q + 128, taken by
// dp2a as they are.  The sums start at -128 / -8 / -16 * sum(X) (Q8_0 / Q4_0 / Q5_0),
// which removes the code offset exactly; the chunk then adds (I2F(sum) * 2^(k-15)) * d,
// and the affine format also b * sum(x).  (|sum| <= 2^24 for the 4- and 5-bit formats,
// so the I2F is exact; a Q8_0 chunk sum can reach 2^26 and then rounds to 24 bits.)
// The order of additions is fixed per lane and chunk.
__device__ __forceinline__ int dp2a_lo(uint32_t x, uint32_t q, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(x), "r"(q), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t x, uint32_t q, int c) {
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(x), "r"(q), "r"(c));
    return d;
}

template <int FMT, int NTOK, int RPW, int XT>
__device__ __forceinline__ void step_idp(Acc<FMT, NTOK, RPW>& A, uint32_t xr, uint32_t codes, uint32_t scales) {
    using F = Fmt<FMT>;
    constexpr int S = x_slots(FMT);
    constexpr int kFullStep = int(kStepCodeBytes) + F::kStepScale;
    uint4 qv[RPW];
    uint32_t sv[RPW];
    uint32_t hv[FMT == QG_Q5_0 ? RPW : 1];         // Q5_0: the chunk's fifth bits
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        qv[r] = lds128(codes + r * kFullStep);
        sv[r] = F::scale(scales + r * kFullStep);
        if constexpr (FMT == QG_Q5_0) hv[r] = F::high(scales + r * kFullStep);
    }
    const uint4 pk = lds128(xr + 16u * uint32_t(XT * S));         // 2^(k-15) per token
    const uint4 pb = lds128(xr + 16u * uint32_t(XT * S + 1));     // Q4_0: -8 sum(X); affine: sum(x)
    const uint32_t pkv[4] = {pk.x, pk.y, pk.z, pk.w};
    const uint32_t pbv[4] = {pb.x, pb.y, pb.z, pb.w};
    int acc[RPW][NTOK];
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int t = 0; t < NTOK; ++t) acc[r][t] = FMT == QG_AFFINE4_G64 ? 0 : int(pbv[t]);
    if constexpr (FMT == QG_Q8_0) {
        // 16 byte codes (q + 128) per row: slot j of staged x holds the pairs of words
        // 2j and 2j + 1; dp2a.lo takes a word's bytes 0-1, dp2a.hi its bytes 2-3.
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            uint4 xv[NTOK];
#pragma unroll
            for (int t = 0; t < NTOK; ++t) xv[t] = lds128(xr + 16u * uint32_t(t * S + j));
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const uint32_t w0 = j == 0 ? qv[r].x : qv[r].z, w1 = j == 0 ? qv[r].y : qv[r].w;
#pragma unroll
                for (int t = 0; t < NTOK; ++t) {
                    int a = acc[r][t];
                    a = dp2a_lo(xv[t].x, w0, a);
                    a = dp2a_hi(xv[t].y, w0, a);
                    a = dp2a_lo(xv[t].z, w1, a);
                    a = dp2a_hi(xv[t].w, w1, a);
                    acc[r][t] = a;
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < (FMT == QG_Q8_0 ? 0 : 4); ++j) {
        uint4 xv[NTOK];
#pragma unroll
        for (int t = 0; t < NTOK; ++t) xv[t] = lds128(xr + 16u * uint32_t(t * S + j));
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const uint32_t w = j == 0 ? qv[r].x : j == 1 ? qv[r].y : j == 2 ? qv[r].z : qv[r].w;
            uint32_t ev = w & 0x0F0F0F0Fu, od = (w >> 4) & 0x0F0F0F0Fu;
            if constexpr (FMT == QG_Q5_0) {
                // fifth bits of the word's even (group 2j) and odd (group 2j + 1) codes
                // to bit 4 of their bytes
                const int ge = 2 * j, go = 2 * j + 1;
                const uint32_t he = ge <= 4 ? hv[r] << (4 - ge) : hv[r] >> (ge - 4);
                const uint32_t ho = go <= 4 ? hv[r] << (4 - go) : hv[r] >> (go - 4);
                ev |= he & 0x10101010u;
                od |= ho & 0x10101010u;
            }
#pragma unroll
            for (int t = 0; t < NTOK; ++t) {
                int a = acc[r][t];
                a = dp2a_lo(xv[t].x, ev, a);
                a = dp2a_hi(xv[t].y, ev, a);
                a = dp2a_lo(xv[t].z, od, a);
                a = dp2a_hi(xv[t].w, od, a);
                acc[r][t] = a;
            }
        }
    }
    // Per token: (affine) A += b * sum(x); then A += (I2F(sum) * 2^(k-15)) * scale (the
    // product with the power of two is exact).
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const float sc = FMT == QG_AFFINE4_G64 ? h2f(sv[r] & 0xFFFFu) : h2f(sv[r]);
        if constexpr (FMT == QG_AFFINE4_G64) {
            const float b = h2f(sv[r] >> 16);
#pragma unroll
            for (int t = 0; t < NTOK; ++t) A.s[r][t] = __fmaf_rn(b, __uint_as_float(pbv[t]), A.s[r][t]);
        }
#pragma unroll
        for (int t = 0; t < NTOK; ++t)
            A.s[r][t] = __fmaf_rn(__fmul_rn(__int2float_rn(acc[r][t]), __uint_as_float(pkv[t])), sc, A.s[r][t]);
    }
}

// One ring stage into the accumulators: the integer chunk dot for the quantized formats,
// packed FP32 FMAs for BF16.
template <int FMT, int NTOK, int RPW, int XT = NTOK>
__device__ __forceinline__ void step_fma(Acc<FMT, NTOK, RPW>& A, uint32_t xr, uint32_t codes, uint32_t scales) {
    if constexpr (IsIdp<FMT>::value) step_idp<FMT, NTOK, RPW, XT>(A, xr, codes, scales);
    else step_fp<FMT, NTOK, RPW, XT>(A, xr, codes, scales);
}

// Transposed warp reduction of the V = RPW * NTOK lane sums (reduce-scatter by
// halving, then xor steps): lane l returns the full sum of output l / (32 / VP).
// The order depends only on V's power-of-two size, never on the data.
template <int FMT, int NTOK, int RPW>
__device__ __forceinline__ float warp_reduce(const Acc<FMT, NTOK, RPW>& A, int lane) {
    constexpr int V = RPW * NTOK;
    constexpr int VP = Pow2Up<V>::value;
    constexpr int LG = Log2<VP>::value;
    float v[VP];
#pragma unroll
    for (int j = 0; j < VP; ++j) v[j] = j < V ? A.value(j) : 0.f;
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
    return v[0];
}

// ------------------------------------------------------------------------------ kernel

// Threads per CTA a kernel allows: 512 (16 warps), or 384 (12 warps) where a warp
// keeps more than 20 outputs per row group (8 rows at ntok 3, 6 rows at ntok 4), so
// that each thread may hold up to 168 registers instead of 128 and the extra rows'
// accumulators do not spill.  Kernels that fit in 128 keep 16 warps.
template <int FMT, int NTOK, int RPW> struct MaxThreads {
    static constexpr int value = RPW * NTOK > 20 ? 384 : 512;
};

template <int FMT, int NTOK, int RPW, bool ARGMAX, bool SPLIT>
__global__ void __launch_bounds__(MaxThreads<FMT, NTOK, RPW>::value, 1) qgemv_kernel(const __grid_constant__ KernelArgs a) {
    using F = Fmt<FMT>;
    constexpr int S = F::kW / 4;                    // x float4 slots per chunk
    constexpr int V = RPW * NTOK;                   // outputs per row group
    constexpr int VP = Pow2Up<V>::value;
    static_assert(VP >= V && VP <= 32, "butterfly width");
    constexpr int SPAN = 32 / VP;                   // lanes sharing one reduced value
    constexpr int kFullStep = int(kStepCodeBytes) + F::kStepScale;
    constexpr int kStage = stage_bytes(FMT, RPW);   // ring stage: RPW rows of one step
    constexpr int kBoxX = kFullStep / 8;            // 8-byte tensor elements per step
    static_assert(kFullStep == full_step(FMT) && kFullStep % 16 == 0, "step size");

    extern __shared__ __align__(128) unsigned char smem[];
    const int n_in = a.n_in;
    const int n4 = n_in >> 2;
    const int codes = FMT == QG_Q8_0 ? n_in : FMT == QG_BF16 ? 2 * n_in : n_in / 2;
    const int spr = (codes + 511) >> 9;             // steps per row
    const int last_codes = codes - 512 * (spr - 1);
    const int depth = a.depth;
    const uint32_t limit = a.wait_limit;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    // Split: the warps form teams of P; warp `seg` of a team streams steps
    // [seg * L, min(spr, (seg + 1) * L)) of every row of the team's groups, and the
    // team adds the segments' reduced values in segment order.  P depends only on
    // (fmt, n_out, n_in), so the arithmetic never depends on ntok or the tile.
    // (SPLIT = false: the kernel for P = 1, without the team exchange's registers.)
    const int P = SPLIT ? a.split : 1, L = SPLIT ? a.seg_len : spr;
    const int team = warp / P, seg = warp - team * P, nteams = nwarps / P;
    const int k0 = seg * L;
    const int k1 = (k0 + L < spr) ? k0 + L : spr;
    // Row groups go round-robin over the CTAs first (group g -> CTA g mod grid), so
    // every SM gets an equal share (within one group) even when the groups do not
    // fill the teams evenly; team m of CTA b takes groups b + grid * (m + nteams * k).
    const int gw = blockIdx.x + gridDim.x * team;
    const int GW = gridDim.x * nteams;
    const int ngroups = (a.n_out + RPW - 1) / RPW;

    constexpr int kCS = NTOK * x_slots(FMT) + x_pad_slots(FMT);   // 16-byte slots per chunk of staged x
    const SmemPlan plan = smem_plan(FMT, NTOK, n_in, RPW, depth, nwarps, P);
    const uint32_t xs_base = smem_addr(smem);
    const uint32_t bars = smem_addr(smem + plan.bar_off) + warp * depth * 8;
    const uint32_t ring = ((smem_addr(smem + plan.ring_off) + 127u) & ~127u) + uint32_t(warp * depth * kStage);
    const uint32_t tbar = smem_addr(smem + plan.tbar_off) + uint32_t(team * 32);   // full[2], empty[2]
    float* xch = reinterpret_cast<float*>(smem + plan.xch_off) + team * 2 * (P - 1) * 32;

    // ---- issue side of the warp's ring: runs `depth` steps ahead of the compute side
    int gi = gw, ki = k0, si = 0;                  // group, step in row, stage
    const uint64_t wpolicy = l2_evict_first_policy();
    uint32_t issued = 0;
    bool failed = false;
    // Lane 0 announces the stage's bytes on its mbarrier and starts one tensor
    // copy of the box (RPW rows x one step).  A box always completes in full:
    // rows past n_out and the bytes past a short last step arrive as zeros.
    // (gi * RPW < n_out <= 2^31 - 1 for every issued group, so it fits an int.)
    auto issue = [&]() {
        if (gi < ngroups && !failed) {
            if (lane == 0) {
                const uint32_t bar = bars + si * 8;
                mbar_arrive_expect_tx(bar, a.stage_tx + (issued == 0 ? a.test_extra_tx : 0u));
                tma_load_2d(ring + uint32_t(si * kStage), &a.wmap, ki * kBoxX, gi * RPW, bar, wpolicy);
            }
            ++issued;
        }
        if (++ki == k1) { ki = k0; gi += GW; }
        if (++si == depth) si = 0;
    };

    // Profiling stamps (thread 0, only when a phase slot is given): the SM clock at
    // each phase (none inside the step loop; nothing stays live in registers).
    auto stamp = [&](int k) {
        if (a.phase && threadIdx.x == 0) a.phase[size_t(blockIdx.x) * QG_PHASE_WORDS + k] = uint32_t(clock());
    };
    stamp(6);
    if (a.phase && threadIdx.x == 0) {
        a.phase[size_t(blockIdx.x) * QG_PHASE_WORDS] = global_ns();
        a.phase[size_t(blockIdx.x) * QG_PHASE_WORDS + 2] = sm_id();
    }

    // Programmatic dependent launch: let the next kernel in the stream start its
    // own weight copies as soon as SMs free up (a no-op without that launch mode).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (lane == 0)   // the weight tensor map is read by this warp's first copy below
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&a.wmap)) : "memory");

    if (lane == 0) {
        for (int s = 0; s < depth; ++s) mbar_init(bars + s * 8, 1);
        if (SPLIT && P > 1 && seg == 0) {   // the team's exchange barriers; first used after __syncthreads
            mbar_init(tbar, uint32_t(P - 1));
            mbar_init(tbar + 8, uint32_t(P - 1));
            mbar_init(tbar + 16, 1);
            mbar_init(tbar + 24, 1);
        }
    }
    mbar_fence_init();
    __syncwarp();
    // The first copies read only W, which no earlier kernel writes (the caller's
    // promise when it enables the early start), so they go before the wait.  Only the
    // first `pre` stages do: the rest of the ring is requested once x is staged, so that
    // the loads of x after the wait do not queue behind the whole initial burst of
    // weights (measured on GB300: 1.5-5% faster on 7-33 MB projections at ntok 2-4 with
    // pre = 1; the tile table keeps the whole ring where that was ahead).
    for (int s = 0; s < a.pre; ++s) issue();
    stamp(3);
    // (profiling only) when warp 0's first stages land, seen before the wait below
    if (a.phase && threadIdx.x == 0)
        for (uint32_t s = 0; s < issued && s < 7u; ++s)
            if (mbar_wait(bars + s * 8, 0u, limit)) stamp(9 + int(s));

    // Everything below may depend on the previous kernel in the stream (x, y, the
    // argmax workspace): wait for it to complete (a no-op without the early start).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    stamp(4);

    // ---- stage x (overlaps the first copies)
    {
        const float4* x4 = reinterpret_cast<const float4*>(a.x);
        const float4* rows[NTOK];
#pragma unroll
        for (int t = 0; t < NTOK; ++t) rows[t] = x4 + t * n4;
        stage_x<FMT, NTOK>(smem, rows, n_in, spr);
    }
    __syncthreads();
    stamp(5);
    for (int s = a.pre; s < depth; ++s) issue();

    float best_v = -INFINITY;
    int best_i = 0x7FFFFFFF;
    const uint32_t x_lane = xs_base + uint32_t(lane) * (kCS * 16);          // chunk `lane` of step 0
    const uint32_t code_lane = ring + 16u * uint32_t(lane);
    const uint32_t scale_lane = ring + F::scale_off(lane);

    Acc<FMT, NTOK, RPW> acc;
    acc.clear();

    int gc = gw, sc = 0;
    uint32_t consumed = 0, phase = 0, jg = 0;       // jg: row groups this warp has finished
    for (; gc < ngroups; gc += GW) {
      for (int kc = k0; kc < k1; ++kc) {
        // The decision to give up is warp-uniform: every lane leaves together.
        if (!__all_sync(kFull, mbar_wait(bars + sc * 8, phase, limit))) {
            failed = true;
            break;
        }
        ++consumed;
        // In a row's short last step the lanes past its codes read zero-filled or
        // scale bytes with a zero scale, against zero-padded x: they add exact zeros.
        const int codes_k = (kc == spr - 1) ? last_codes : 512;
        {
            const uint32_t stage = uint32_t(sc) * uint32_t(kStage);
            step_fma<FMT, NTOK, RPW>(acc, x_lane + uint32_t(kc) * (32u * kCS * 16u), code_lane + stage,
                                     scale_lane + stage + uint32_t(codes_k));
        }
        __syncwarp();          // every lane has read this stage before it is refilled
        issue();
        if (++sc == depth) { sc = 0; phase ^= 1u; }
      }
      if (failed) break;
        {
            // ---- finish the row group: transposed warp reduction
            float v0 = warp_reduce<FMT, NTOK, RPW>(acc, lane);
            const int vi = lane / SPAN;                       // value index this lane holds
            const bool holder = vi < V && (lane % SPAN) == 0;
            if (SPLIT && P > 1) {
                // Team exchange (double-buffered by group parity, bounded waits):
                // segments 1..P-1 publish their values, segment 0 adds them in order.
                const int par = int(jg & 1u);
                const uint32_t use = jg >> 1;
                float* slot = xch + par * (P - 1) * 32;
                if (seg > 0) {
                    if (jg >= 2 && !__all_sync(kFull, mbar_wait(tbar + 16 + 8 * par, (use - 1) & 1u, limit))) {
                        failed = true;
                        break;
                    }
                    if (holder) slot[(seg - 1) * 32 + vi] = v0;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tbar + 8 * par);
                } else {
                    if (!__all_sync(kFull, mbar_wait(tbar + 8 * par, use & 1u, limit))) {
                        failed = true;
                        break;
                    }
                    if (holder)
                        for (int q = 0; q < P - 1; ++q) v0 += slot[q * 32 + vi];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tbar + 16 + 8 * par);
                }
                ++jg;
            }
            if (holder && seg == 0) {
                const int r = vi / NTOK, t = vi - r * NTOK;
                const long long row = (long long)gc * RPW + r;
                if (row < a.n_out) {
                    if (!ARGMAX || a.y) a.y[(long long)t * a.n_out + row] = v0;
                    if (ARGMAX && better(v0, int(row), best_v, best_i)) { best_v = v0; best_i = int(row); }
                }
            }
            acc.clear();
        }
    }

    if (failed) {
        // Report, then drain (bounded) every copy this warp issued but did not consume,
        // so no TMA copy is still writing this CTA's shared memory when it exits.
        if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
        for (uint32_t f = consumed; f < issued; ++f) {
            mbar_wait(bars + sc * 8, phase, a.drain_limit);
            if (++sc == depth) { sc = 0; phase ^= 1u; }
        }
    }
    stamp(7);

    if constexpr (ARGMAX) {
        // ---- per-token argmax: warp -> CTA partial -> last CTA reduces all partials
        __shared__ ArgmaxPartial wbest[kMaxWarps][kMaxNtok];
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
                if (lane == 0) a.argmax[t] = (bi == 0x7FFFFFFF) ? -1 : (a.row_ids ? a.row_ids[bi] : bi);
            }
            if (threadIdx.x == 0) *a.ticket = 0u;   // ready for the next call on this workspace
        }
    }
    if (a.phase) {             // uniform over the CTA
        __syncthreads();
        stamp(8);
        if (threadIdx.x == 0) a.phase[size_t(blockIdx.x) * QG_PHASE_WORDS + 1] = global_ns();
    }
}

// Lookup of an instantiated kernel (defined in the per-format instantiation units).
const void* kernel_lookup(int fmt, int ntok, int rpw, bool argmax, bool split);

}  // namespace qg
