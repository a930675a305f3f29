// Expert-grouped multi-token mat-vec for sm_103a (routed experts at ntok <= 4).
//
// The operator of the Track 2 Audit & Optimization Report (M5 Metal kernels),
// section 1 item 2: a plan groups a step's (token, expert) pairs by expert, and
// the gate/up and down projections run every group with its own token count
// ne = 1..4, reading each active expert's weights from memory once.  Here the
// experts' matrices are stacked ([n_experts * n_out][n_in], expert e = rows
// e * n_out ..), one tensor map covers the stack, and the plan sits in device
// memory, written by the plan kernel (or the caller), so no host round trip
// separates routing from the projections.
//
// GB300 design, on the pieces of the plain mat-vec kernel (stage_x, step_fma,
// warp_reduce): a persistent grid whose CTAs are dealt to groups (one each, the
// rest in proportion to a weight base + the group's token count, since a group's
// compute grows with its tokens; see assign_groups); a CTA stages the x rows of its
// group's ne tokens once and its warps stream the expert's row blocks round-robin
// through their TMA rings.  ne is a run-time value: the kernel switches to a body
// compiled for each ne, so a one-token group costs what a one-token mat-vec costs.
// The first copies of a group need only the expert id and go out before x is
// staged.  With more groups than CTAs, a CTA takes groups b, b + C, ... one after
// the other, restaging x between them.  The same pieces also make the whole layer
// (plan, gate/up with its activation, down) one persistent launch
// (qgemv_expert_layer_kernel, below).
//
// Optionally a launch also prefetches into L2 the same experts' rows of the NEXT
// projection's stack (the down projection while gate/up runs): the 129 MB L2
// holds a step's active experts, so the next launch's first copies hit L2 instead
// of waiting for HBM, and HBM keeps streaming across the launch boundary.  The
// prefetch is spread over the group's CTAs: one SM's bulk-copy engine alone
// would issue it far too slowly.
//
// The addition order of an output depends only on (fmt, n_in): it is the order of
// the plain mat-vec without a split, whatever ne, the group, the tile or the grid.
#pragma once

#include "qgemv_kernels.cuh"

namespace qg {

constexpr unsigned kStatusBadPlan = 4u;   // a plan entry or a routed expert id out of range
constexpr unsigned kExpertsXBySlot = QG_EXPERTS_X_BY_SLOT;
constexpr unsigned kExpertsPlanReady = QG_EXPERTS_PLAN_READY;
constexpr unsigned kExpertsSwiglu = QG_EXPERTS_SWIGLU;
constexpr int kMaxPlanPairs = 1024;      // (token, choice) pairs one plan can hold

// Offsets (in int32 entries) of the plan's arrays for n_slots = ntok * topk slots.
__host__ __device__ constexpr int plan_group_start(int) { return 1; }           // n_slots + 1 entries
__host__ __device__ constexpr int plan_group_expert(int G) { return 2 + G; }    // n_slots entries
__host__ __device__ constexpr int plan_slot_pair(int G) { return 2 + 2 * G; }
__host__ __device__ constexpr int plan_slot_token(int G) { return 2 + 3 * G; }
__host__ __device__ constexpr int plan_pair_slot(int G) { return 2 + 4 * G; }
__host__ __device__ constexpr int plan_ints(int G) { return 2 + 5 * G; }

// The expert kernel's shared memory: the mat-vec layout for kMaxNtok tokens (x,
// barriers, rings), then the plan's group arrays and slot tokens, 2 + 3G ints.
__host__ __device__ constexpr int plan_smem_off(int plan_total) { return (plan_total + 15) / 16 * 16; }
__host__ __device__ constexpr int plan_smem_bytes(int G) { return (2 + 3 * G) * 4; }

struct ExpertArgs {
    CUtensorMap wmap;          // the stacked experts' packed rows as [n_experts * n_out][stride / 8]
                               // 8-byte elements, box = one full step x RPW rows, zero fill outside
    const float* x;            // [n_x][n_in]
    float* y;                  // [n_slots][n_out]
    const int32_t* plan;       // the plan (offsets above)
    unsigned int* status;      // device status word
    int n_experts;
    int n_out;
    int n_in;
    int n_slots;
    int n_x;                   // rows of x
    unsigned flags;            // kExpertsXBySlot: slot s reads x[s] (else x[slot_token[s]]);
                               // kExpertsPlanReady: the plan is complete when the launch begins
    int depth;
    uint32_t wait_limit, drain_limit, stage_tx;
    uint32_t test_extra_tx;    // test hook: bytes added to every warp's first expected transaction
    const unsigned char* next_w;   // optional: a second stack of the same experts whose active
                                   // experts this launch prefetches into L2 (nullptr = none)
    long long next_bytes;          // bytes per expert of that stack (a multiple of 16)
    int group_base;                // CTA shares: weight base + ne per group (0 = equal)
};

constexpr int kL2PrefetchPiece = 32768;   // bytes per L2 prefetch instruction

// Bulk prefetch of [p, p + bytes) into L2 (p 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
                 : "memory");
}

// One warp's ring over the groups a CTA serves: the issue cursor (row block, step,
// stage) runs `depth` steps ahead of the consume cursor (stage, phase).  All
// copies of a group are consumed before the next group's first copy is issued, so
// the issue stage of a new group starts at the consume stage.
template <int RPW, int kStage, int kBoxX>
struct ExpertRing {
    uint32_t bars, ring;
    uint64_t policy;
    int depth, spr, nblk;
    int sc = 0;
    uint32_t phase = 0, issued = 0, consumed = 0;
    bool failed = false;
    int gi = 0, ki = 0, si = 0, gstride = 1, ebase = 0;

    __device__ __forceinline__ void start_group(int first_block, int stride, int expert_row0) {
        gi = first_block;
        ki = 0;
        si = sc;
        gstride = stride;
        ebase = expert_row0;
    }
    // Lane 0 announces the stage's bytes and starts one tensor copy of the box
    // (RPW rows x one step); rows past the stack arrive as zeros.
    __device__ __forceinline__ void issue(const CUtensorMap* map, uint32_t tx, uint32_t extra, int lane) {
        if (gi < nblk && !failed) {
            if (lane == 0) {
                const uint32_t bar = bars + si * 8;
                mbar_arrive_expect_tx(bar, tx + (issued == 0 ? extra : 0u));
                tma_load_2d(ring + uint32_t(si * kStage), map, ki * kBoxX, ebase + gi * RPW, bar, policy);
            }
            ++issued;
        }
        if (++ki == spr) { ki = 0; gi += gstride; }
        if (++si == depth) si = 0;
    }
};

// One group of NE tokens (x staged in the layout for XT >= NE tokens): stream this
// warp's row blocks of the expert and write y[s0 + t][row].
template <int FMT, int RPW, int NE, int XT, class Ring>
__device__ __forceinline__ void expert_group(const ExpertArgs& a, Ring& R, unsigned char* smem, int s0,
                                             int first_block, int lane) {
    using F = Fmt<FMT>;
    constexpr int S = F::kW / 4;
    constexpr int kCS = XT * x_slots(FMT) + x_pad_slots(FMT);
    constexpr int V = RPW * NE;
    constexpr int SPAN = 32 / Pow2Up<V>::value;
    constexpr int kStage = stage_bytes(FMT, RPW);
    const int n_in = a.n_in, n_out = a.n_out;
    const int codes = FMT == QG_Q8_0 ? n_in : FMT == QG_BF16 ? 2 * n_in : n_in / 2;
    const int last_codes = codes - 512 * (R.spr - 1);
    const uint32_t x_lane = smem_addr(smem) + uint32_t(lane) * (kCS * 16);
    const uint32_t code_lane = R.ring + 16u * uint32_t(lane);
    const uint32_t scale_lane = R.ring + F::scale_off(lane);
    Acc<FMT, NE, RPW> acc;
    acc.clear();
    for (int gc = first_block; gc < R.nblk; gc += R.gstride) {
        for (int kc = 0; kc < R.spr; ++kc) {
            if (!__all_sync(kFull, mbar_wait(R.bars + R.sc * 8, R.phase, a.wait_limit))) {
                R.failed = true;
                break;
            }
            ++R.consumed;
            const int codes_k = (kc == R.spr - 1) ? last_codes : 512;
            const uint32_t stage = uint32_t(R.sc) * uint32_t(kStage);
            step_fma<FMT, NE, RPW, XT>(acc, x_lane + uint32_t(kc) * (32u * kCS * 16u), code_lane + stage,
                                   scale_lane + stage + uint32_t(codes_k));
            __syncwarp();                        // every lane has read this stage before it is refilled
            R.issue(&a.wmap, a.stage_tx, a.test_extra_tx, lane);
            if (++R.sc == R.depth) { R.sc = 0; R.phase ^= 1u; }
        }
        if (R.failed) break;
        const float v0 = warp_reduce<FMT, NE, RPW>(acc, lane);
        const int vi = lane / SPAN;
        bool stored = false;
        if constexpr (RPW % 2 == 0) {
            if (a.flags & kExpertsSwiglu) {
                // Rows 2j (gate) and 2j + 1 (up) of a block sit NE values apart: the
                // gate's lane takes the up value and writes silu(gate) * up.
                const float up = __shfl_down_sync(kFull, v0, NE * SPAN);
                if (vi < V && (lane % SPAN) == 0) {
                    const int r = vi / NE, t = vi - r * NE;
                    const int row = gc * RPW + r;
                    if ((r & 1) == 0 && row < n_out)
                        a.y[(long long)(s0 + t) * (n_out >> 1) + (row >> 1)] = v0 / (1.0f + expf(-v0)) * up;
                }
                stored = true;
            }
        }
        if (!stored && vi < V && (lane % SPAN) == 0) {
            const int r = vi / NE, t = vi - r * NE;
            const int row = gc * RPW + r;
            if (row < n_out) a.y[(long long)(s0 + t) * n_out + row] = v0;
        }
        acc.clear();
    }
}

// Group g of the plan in shared memory: its first slot, token count, expert and x
// rows; false if any entry is out of range.  Every thread reads the same words, so
// the result is CTA-uniform.
__device__ __forceinline__ bool decode_group(const ExpertArgs& a, const int* ps, int G, int g, int& s0, int& ne,
                                             int& e, int (&xrow)[kMaxNtok]) {
    s0 = ps[plan_group_start(G) + g];
    const int s1 = ps[plan_group_start(G) + g + 1];
    e = ps[plan_group_expert(G) + g];
    ne = s1 - s0;
    bool ok = s0 >= 0 && s1 <= G && ne >= 1 && ne <= kMaxNtok && e >= 0 && e < a.n_experts;
#pragma unroll
    for (int k = 0; k < kMaxNtok; ++k) {
        xrow[k] = 0;
        if (ok && k < ne) {
            xrow[k] = (a.flags & kExpertsXBySlot) ? s0 + k : ps[2 + 2 * G + s0 + k];
            ok = ok && xrow[k] >= 0 && xrow[k] < a.n_x;
        }
    }
    return ok;
}

// The group's CTAs split expert e's bytes of the next stack; the warps of a CTA split
// its share in pieces (lane 0 issues).  The copies land in L2 while this and the next
// launch run, so the next projection starts on cached weights.
__device__ __forceinline__ void prefetch_next(const ExpertArgs& a, int e, int ci, int cn, int warp, int nwarps) {
    const long long B = a.next_bytes;
    const long long per = ((B + cn - 1) / cn + 15) / 16 * 16;
    const long long lo = (long long)ci * per;
    const long long hi = lo + per < B ? lo + per : B;
    const unsigned char* base = a.next_w + (long long)e * B;
    for (long long off = lo + (long long)warp * kL2PrefetchPiece; off < hi; off += (long long)nwarps * kL2PrefetchPiece)
        l2_prefetch(base + off, uint32_t(hi - off < kL2PrefetchPiece ? hi - off : kL2PrefetchPiece));
}

// Threads per CTA: 16 warps up to 2 rows per warp; 12 warps (168 registers a thread)
// at 4 rows, whose four-token body does not fit in 128 registers beside the group
// loop's state.
template <int RPW> struct ExpertThreads { static constexpr int value = RPW >= 4 ? 384 : 512; };

// CTAs over groups.  With n_groups <= C every group gets one CTA and the other
// C - n_groups CTAs are dealt in proportion to the groups' weights base + ne (a group
// costs its expert's bytes, the same for all, plus compute per token; base <= 0:
// equal shares, CTA b serving group floor(b * n_groups / C)).  With more groups than
// CTAs, CTA b takes whole groups b, b + C, ...  `ps` is the plan in shared memory.
// Every thread of the CTA calls it (the weighted path has a barrier).
__device__ __forceinline__ void assign_groups(const int* ps, int G, int ng, int C, int b, int base, int& g,
                                              int& gstep, int& ci, int& cn) {
    if (ng > C) {
        g = b;
        ci = 0;
        cn = 1;
        gstep = C;
        return;
    }
    const int d = ng > 0 ? ng : 1;
    gstep = d;
    // Equal shares when the weights are equal: no weighting asked for, or every group
    // one token (ng == G, e.g. ntok 1).
    if (base <= 0 || ng == 0 || ng == G) {
        g = int((long long)b * ng / C);
        const int b0 = int(((long long)g * C + d - 1) / d);
        const int b1 = int(((long long)(g + 1) * C + d - 1) / d);
        ci = b - b0;
        cn = b1 - b0;
        return;
    }
    // The first warp computes the shares with a scan over the groups' weights (one
    // CTA's group is the one whose CTA range holds b); the others wait at the barrier.
    auto weight = [&](int h) {
        int ne = ps[plan_group_start(0) + h + 1] - ps[plan_group_start(0) + h];
        ne = ne < 0 ? 0 : ne > kMaxNtok ? kMaxNtok : ne;
        return (long long)(base + ne);
    };
    __shared__ int s_assign[3];
    if (threadIdx.x < 32) {
        const int lane = int(threadIdx.x);
        long long W = 0;
        for (int h = lane; h < ng; h += 32) W += weight(h);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) W += __shfl_xor_sync(kFull, W, m);
        const long long extra = C - ng;
        long long carry = 0;
        for (int h0 = 0; h0 < ng; h0 += 32) {
            const int h = h0 + lane;
            const long long w = h < ng ? weight(h) : 0;
            long long inc = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long n = __shfl_up_sync(kFull, inc, o);
                if (lane >= o) inc += n;
            }
            if (h < ng) {
                const int st = h + int((extra * (carry + inc - w) + W - 1) / W);   // first CTA of group h
                const int nx = h + 1 + int((extra * (carry + inc) + W - 1) / W);   // first CTA of group h + 1
                if (b >= st && b < nx) {
                    s_assign[0] = h;
                    s_assign[1] = st;
                    s_assign[2] = nx;
                }
            }
            carry += __shfl_sync(kFull, inc, 31);
        }
    }
    __syncthreads();
    g = s_assign[0];
    ci = b - s_assign[1];
    cn = s_assign[2] - s_assign[1];
}

// A group's first copies (and its prefetch of the next stack): they need only the
// expert id.  (e * n_out + n_out <= 2^31 - 1, checked at launch.)
template <class Ring>
__device__ __forceinline__ void issue_group(const ExpertArgs& a, Ring& R, int e, int ci, int cn, int warp, int nwarps,
                                            int lane) {
    R.start_group(ci + cn * warp, cn * nwarps, e * a.n_out);
    for (int s = 0; s < R.depth; ++s) R.issue(&a.wmap, a.stage_tx, a.test_extra_tx, lane);
    if (a.next_w != nullptr && lane == 0) prefetch_next(a, e, ci, cn, warp, nwarps);
}

// Every group this CTA serves for one projection: stage the group's x rows once,
// then its warps stream their row blocks (the bodies for ne = 1..4).  `g_issued`:
// the group whose first copies are already out (-1: none).  COHERENT_X: x was
// written earlier in this kernel.
template <int FMT, int RPW, bool COHERENT_X, class Ring>
__device__ __forceinline__ void serve_groups(const ExpertArgs& a, Ring& R, unsigned char* smem, const int* ps, int G,
                                             int ng, int g, int gstep, int ci, int cn, int g_issued, int warp,
                                             int nwarps, int lane) {
    const int first = ci + cn * warp;
    for (; g < ng; g += gstep) {
        int s0, ne, e, xrow[kMaxNtok];
        if (!decode_group(a, ps, G, g, s0, ne, e, xrow)) {
            if (threadIdx.x == 0) atomicOr(a.status, kStatusBadPlan);
            continue;
        }
        if (g != g_issued) issue_group(a, R, e, ci, cn, warp, nwarps, lane);
        __syncthreads();                         // no warp still reads the previous group's x
        {
            // One staging path for every ne (the layout for kMaxNtok tokens; slots of
            // tokens >= ne are never read).
            const float4* x4 = reinterpret_cast<const float4*>(a.x);
            const float4* rows[kMaxNtok];
#pragma unroll
            for (int k = 0; k < kMaxNtok; ++k) rows[k] = x4 + (long long)xrow[k] * (a.n_in >> 2);
            stage_x<FMT, kMaxNtok, !COHERENT_X>(smem, rows, a.n_in, R.spr, ne);
        }
        __syncthreads();
        if (R.failed) continue;
        switch (ne) {
            case 1: expert_group<FMT, RPW, 1, kMaxNtok>(a, R, smem, s0, first, lane); break;
            case 2: expert_group<FMT, RPW, 2, kMaxNtok>(a, R, smem, s0, first, lane); break;
            case 3: expert_group<FMT, RPW, 3, kMaxNtok>(a, R, smem, s0, first, lane); break;
            default: expert_group<FMT, RPW, 4, kMaxNtok>(a, R, smem, s0, first, lane); break;
        }
    }
}

// After a failed wait: report, then drain (bounded) the copies issued but not consumed.
template <class Ring>
__device__ __forceinline__ void drain_ring(const ExpertArgs& a, Ring& R, int lane) {
    if (!R.failed) return;
    if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
    for (uint32_t f = R.consumed; f < R.issued; ++f) {
        mbar_wait(R.bars + R.sc * 8, R.phase, a.drain_limit);
        if (++R.sc == R.depth) { R.sc = 0; R.phase ^= 1u; }
    }
}

template <int FMT, int RPW>
__global__ void __launch_bounds__(ExpertThreads<RPW>::value, 1) qgemv_experts_kernel(const __grid_constant__ ExpertArgs a) {
    using F = Fmt<FMT>;
    constexpr int kFullStep = int(kStepCodeBytes) + F::kStepScale;
    constexpr int kStage = stage_bytes(FMT, RPW);
    constexpr int kBoxX = kFullStep / 8;
    static_assert(kFullStep == full_step(FMT) && kFullStep % 16 == 0, "step size");

    extern __shared__ __align__(128) unsigned char smem[];
    const int n_in = a.n_in;
    const int codes = FMT == QG_Q8_0 ? n_in : FMT == QG_BF16 ? 2 * n_in : n_in / 2;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;

    const SmemPlan sp = smem_plan(FMT, kMaxNtok, n_in, RPW, a.depth, nwarps, 1);
    ExpertRing<RPW, kStage, kBoxX> R;
    R.depth = a.depth;
    R.spr = (codes + 511) >> 9;
    R.nblk = (a.n_out + RPW - 1) / RPW;
    R.bars = smem_addr(smem + sp.bar_off) + warp * R.depth * 8;
    R.ring = ((smem_addr(smem + sp.ring_off) + 127u) & ~127u) + uint32_t(warp * R.depth * kStage);
    R.policy = l2_evict_first_policy();

    if (lane == 0) {
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&a.wmap)) : "memory");
        for (int s = 0; s < R.depth; ++s) mbar_init(R.bars + s * 8, 1);
    }
    mbar_fence_init();
    __syncwarp();
    // x (and, unless the caller says it is complete, the plan) may come from the
    // previous kernel in the stream.  Dependents may begin only once this launch's own
    // dependencies are complete: a later launch that reads the plan before its wait
    // (kExpertsPlanReady) then finds it complete.
    const bool plan_ready = (a.flags & kExpertsPlanReady) != 0;
    if (!plan_ready) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }

    // The plan's group arrays and slot tokens into shared memory with one round of
    // independent loads (every group's entries then cost no further global latency):
    // ps[0 .. 2 + 2G) = n_groups, group_start, group_expert; ps[2 + 2G ..) = slot_token.
    const int G = a.n_slots;
    int* ps = reinterpret_cast<int*>(smem + plan_smem_off(sp.total));
    {
        const int n_head = 2 + 2 * G, n_all = 2 + 3 * G;
        for (int i0 = threadIdx.x; i0 < n_all; i0 += 8 * blockDim.x) {
            int v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = i0 + j * int(blockDim.x);
                if (i < n_all) v[j] = __ldg(a.plan + (i < n_head ? i : i + G));   // skip slot_pair
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = i0 + j * int(blockDim.x);
                if (i < n_all) ps[i] = v[j];
            }
        }
    }
    __syncthreads();
    int ng = ps[0];
    if (ng < 0 || ng > G) {
        if (threadIdx.x == 0) atomicOr(a.status, kStatusBadPlan);
        ng = 0;
    }
    int g, gstep, ci, cn;
    assign_groups(ps, G, ng, int(gridDim.x), int(blockIdx.x), a.group_base, g, gstep, ci, cn);

    // The first group's weight copies need only the plan: they go out before the
    // wait for the previous kernel when the plan is known to be complete.
    int g_issued = -1;
    if (g < ng) {
        int s0, ne, e, xrow[kMaxNtok];
        if (decode_group(a, ps, G, g, s0, ne, e, xrow)) {
            issue_group(a, R, e, ci, cn, warp, nwarps, lane);
            g_issued = g;
        }
    }
    if (plan_ready) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    serve_groups<FMT, RPW, false>(a, R, smem, ps, G, ng, g, gstep, ci, cn, g_issued, warp, nwarps, lane);
    drain_ring(a, R, lane);
}

// ------------------------------------------------------------------------------ the plan

// The plan of n routed pairs, built by one CTA: a pair's slot is the number of pairs
// with a smaller expert id, or the same id and a smaller index (a stable sort by
// expert); a slot starts a group when its pair is its expert's 0th, 4th, 8th, ...
// Writes the compact shared-memory form ps (2 + 3n ints: n_groups, group_start[n + 1],
// group_expert[n], slot_token[n]) and, if gplan is not null, the full plan in the
// header's layout.  scratch: 3n + 1 ints.  Returns false (n_groups = 0) when an id is
// outside [0, n_experts).  Every thread of the CTA must call it.
__device__ __forceinline__ bool plan_build(const int32_t* ids, int n, int topk, int n_experts, int* scratch, int* ps,
                                           int32_t* gplan) {
    const int G = n, tid = int(threadIdx.x), bd = int(blockDim.x);
    int* e_s = scratch;
    int* start_s = scratch + n;
    int* pair_s = scratch + 2 * n;
    int* count_s = scratch + 3 * n;
    bool bad = false;
    for (int i = tid; i < n; i += bd) {
        const int e = __ldg(ids + i);
        bad = bad || e < 0 || e >= n_experts;
        e_s[i] = e;
    }
    if (tid == 0) *count_s = 0;
    if (__syncthreads_or(bad)) {
        if (tid == 0) {
            ps[0] = 0;
            if (gplan) gplan[0] = 0;
        }
        __syncthreads();
        return false;
    }
    for (int i = tid; i < n; i += bd) {
        const int e = e_s[i];
        int r = 0, w = 0;
        for (int j = 0; j < n; ++j) {
            const int f = e_s[j];
            r += (f < e) || (f == e && j < i);
            w += (f == e && j < i);
        }
        pair_s[r] = i;
        start_s[r] = (w % kMaxNtok) == 0;
        ps[2 + 2 * G + r] = i / topk;
        if (gplan) {
            gplan[plan_slot_pair(G) + r] = i;
            gplan[plan_slot_token(G) + r] = i / topk;
            gplan[plan_pair_slot(G) + i] = r;
        }
    }
    __syncthreads();
    int mine = 0;
    for (int s = tid; s < n; s += bd) {
        if (!start_s[s]) continue;
        int g = 0;
        for (int q = 0; q < s; ++q) g += start_s[q];
        const int e = e_s[pair_s[s]];
        ps[plan_group_start(G) + g] = s;
        ps[plan_group_expert(G) + g] = e;
        if (gplan) {
            gplan[plan_group_start(G) + g] = s;
            gplan[plan_group_expert(G) + g] = e;
        }
        ++mine;
    }
    // One shared atomic per warp (a per-thread atomic on one word serialises).
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) mine += __shfl_xor_sync(kFull, mine, m);
    if ((tid & 31) == 0 && mine) atomicAdd(count_s, mine);
    __syncthreads();
    const int ng = *count_s;
    for (int g = ng + tid; g <= G; g += bd) {
        ps[plan_group_start(G) + g] = G;
        if (g < G) ps[plan_group_expert(G) + g] = -1;
        if (gplan) {
            gplan[plan_group_start(G) + g] = G;
            if (g < G) gplan[plan_group_expert(G) + g] = -1;
        }
    }
    if (tid == 0) {
        ps[0] = ng;
        if (gplan) gplan[0] = ng;
    }
    __syncthreads();
    return true;
}

// Shared memory of the plan's compact form plus its scratch, for n pairs.
__host__ __device__ constexpr int plan_build_bytes(int n) { return (2 + 3 * n) * 4 + (3 * n + 1) * 4; }

// ------------------------------------------------------------------------------ one layer

// The routed-expert layer in one persistent launch: every CTA builds the plan from
// the routing ids in shared memory (CTA 0 also writes it out), serves its groups of
// the gate/up projection (writing silu(gate) * up and prefetching the same experts'
// down rows into L2), issues the first copies of its down rows, and serves the same
// groups of the down projection.  A group's down rows read only that group's
// activation rows, which only that group's CTAs write: so the CTAs of a group meet
// at a barrier of their own (a counter per group), and a group that finishes its
// gate/up early goes on without waiting for the slowest group.  (With more groups
// than CTAs a group has one CTA and needs no barrier.)  The grid is sized to be
// resident at once; every wait is bounded.
struct LayerArgs {
    ExpertArgs gu;               // gate/up: x = token rows, y = activation [n_slots][d_ff], SWIGLU
    ExpertArgs dn;               // down: x = the activation (by slot), y = [n_slots][d_model]
    const int32_t* ids;          // [ntok][topk] routed experts
    int topk;
    int32_t* plan_out;           // the plan in the header's layout (written by CTA 0)
    unsigned int* barrier;       // [0] departures, [1 + g] arrivals of group g; zero between launches
    uint32_t barrier_limit;      // polls of the arrival counter before the barrier gives up
};

template <int FMT, int RPW>
__global__ void __launch_bounds__(ExpertThreads<RPW>::value, 1) qgemv_expert_layer_kernel(const __grid_constant__ LayerArgs L) {
    using F = Fmt<FMT>;
    constexpr int kFullStep = int(kStepCodeBytes) + F::kStepScale;
    constexpr int kStage = stage_bytes(FMT, RPW);
    constexpr int kBoxX = kFullStep / 8;
    static_assert(kFullStep == full_step(FMT) && kFullStep % 16 == 0, "step size");

    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int max_in = L.gu.n_in > L.dn.n_in ? L.gu.n_in : L.dn.n_in;
    auto spr_of = [](int n_in) {
        const int codes = FMT == QG_Q8_0 ? n_in : FMT == QG_BF16 ? 2 * n_in : n_in / 2;
        return (codes + 511) >> 9;
    };

    const SmemPlan sp = smem_plan(FMT, kMaxNtok, max_in, RPW, L.gu.depth, nwarps, 1);
    ExpertRing<RPW, kStage, kBoxX> R;
    R.depth = L.gu.depth;
    R.bars = smem_addr(smem + sp.bar_off) + warp * R.depth * 8;
    R.ring = ((smem_addr(smem + sp.ring_off) + 127u) & ~127u) + uint32_t(warp * R.depth * kStage);
    R.policy = l2_evict_first_policy();
    if (lane == 0) {
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&L.gu.wmap)) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&L.dn.wmap)) : "memory");
        for (int s = 0; s < R.depth; ++s) mbar_init(R.bars + s * 8, 1);
    }
    mbar_fence_init();
    __syncwarp();
    // The routing ids and x come from earlier kernels, and the outputs may still be
    // read by them.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int G = L.gu.n_slots;
    int* ps = reinterpret_cast<int*>(smem + plan_smem_off(sp.total));
    int* scratch = ps + 2 + 3 * G;
    if (!plan_build(L.ids, G, L.topk, L.gu.n_experts, scratch, ps, blockIdx.x == 0 ? L.plan_out : nullptr)) {
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(L.gu.status, kStatusBadPlan);
    }
    const int ng = ps[0];
    int g, gstep, ci, cn;
    assign_groups(ps, G, ng, int(gridDim.x), int(blockIdx.x), L.gu.group_base, g, gstep, ci, cn);
    const int g0 = g;

    // ---- gate/up (+ activation, + L2 prefetch of the down rows)
    R.spr = spr_of(L.gu.n_in);
    R.nblk = (L.gu.n_out + RPW - 1) / RPW;
    serve_groups<FMT, RPW, false>(L.gu, R, smem, ps, G, ng, g, gstep, ci, cn, -1, warp, nwarps, lane);

    // ---- the first down copies need only the plan: out before the barrier
    R.spr = spr_of(L.dn.n_in);
    R.nblk = (L.dn.n_out + RPW - 1) / RPW;
    int g_issued = -1;
    if (g0 < ng) {
        int s0, ne, e, xrow[kMaxNtok];
        if (decode_group(L.dn, ps, G, g0, s0, ne, e, xrow)) {
            issue_group(L.dn, R, e, ci, cn, warp, nwarps, lane);
            g_issued = g0;
        }
    }

    // ---- group barrier (bounded): the group's activation rows are all written
    __shared__ int passed;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        bool ok = true;
        if (g0 < ng && ng <= int(gridDim.x)) {
            unsigned* cnt = L.barrier + 1 + g0;
            atomicAdd(cnt, 1u);
            ok = false;
            for (uint32_t it = 0; it < L.barrier_limit; ++it) {
                unsigned v;
                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
                if (v >= unsigned(cn)) { ok = true; break; }
                __nanosleep(32);
            }
            __threadfence();
        }
        if (!ok) atomicOr(L.gu.status, kStatusWaitTimeout);
        passed = ok ? 1 : 0;
    }
    __syncthreads();
    if (!passed) R.failed = true;

    // ---- down
    serve_groups<FMT, RPW, true>(L.dn, R, smem, ps, G, ng, g0, gstep, ci, cn, g_issued, warp, nwarps, lane);
    drain_ring(L.dn, R, lane);

    // ---- the last CTA out resets the counters for the next launch
    __shared__ bool last;
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(L.barrier, 1u) == gridDim.x - 1;
    __syncthreads();
    if (last) {
        for (int i = threadIdx.x; i <= G; i += blockDim.x) L.barrier[i] = 0u;   // [0] and the G groups
        __threadfence();
    }
}

// Lookup of an instantiated expert kernel (qgemv_experts.cu).
const void* expert_kernel_lookup(int fmt, int rpw);
const void* expert_layer_kernel_lookup(int fmt, int rpw);

}  // namespace qg
