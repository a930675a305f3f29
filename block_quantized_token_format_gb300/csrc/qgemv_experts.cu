// Instantiations of the expert-grouped mat-vec kernel (every format, 1, 2 and 4 rows
// per warp; each kernel holds the bodies for ne = 1..4) and of the one-launch layer.
#include <algorithm>
#include <cstdio>
#include <initializer_list>
#include <mutex>

#include "qgemv_experts.cuh"
#include "qgemv_host.h"
#include "tile_select.h"

namespace qg {

const void* expert_kernel_lookup(int fmt, int rpw) {
#define QG_X(F)                                                            \
    if (fmt == F) {                                                        \
        if (rpw == 1) return (const void*)&qgemv_experts_kernel<F, 1>;     \
        if (rpw == 2) return (const void*)&qgemv_experts_kernel<F, 2>;     \
        if (rpw == 4) return (const void*)&qgemv_experts_kernel<F, 4>;     \
        return nullptr;                                                    \
    }
    QG_X(QG_Q8_0) QG_X(QG_Q4_0) QG_X(QG_AFFINE4_G64) QG_X(QG_BF16) QG_X(QG_Q5_0)
#undef QG_X
    return nullptr;
}

// The one-launch layer: gate/up pairs need an even number of rows per warp.
const void* expert_layer_kernel_lookup(int fmt, int rpw) {
#define QG_L(F)                                                                \
    if (fmt == F) {                                                            \
        if (rpw == 2) return (const void*)&qgemv_expert_layer_kernel<F, 2>;    \
        if (rpw == 4) return (const void*)&qgemv_expert_layer_kernel<F, 4>;    \
        return nullptr;                                                        \
    }
    QG_L(QG_Q8_0) QG_L(QG_Q4_0) QG_L(QG_AFFINE4_G64) QG_L(QG_BF16) QG_L(QG_Q5_0)
#undef QG_L
    return nullptr;
}

}  // namespace qg

// ------------------------------------------------------------------ host side (C ABI)
namespace qg {
namespace {

// The plan of a step's routed pairs (one CTA, one thread per pair; at most 1024
// pairs, so every quadratic loop is short).  The same plan as plan_build, written
// for this one-thread-per-pair launch: measured ~0.5 µs faster per call than
// plan_build's general (strided, shared-memory) form, and the plan call sits on the
// layer's critical path.  Slot of pair i = the number of pairs
// with a smaller expert id, or the same id and a smaller i (a stable sort by
// expert); the slot starts a group when the pair is its expert's 0th, 4th, 8th, ...
__global__ void __launch_bounds__(kMaxPlanPairs) expert_plan_kernel(const int32_t* __restrict__ ids, int n, int topk,
                                                                    int n_experts, int32_t* __restrict__ plan,
                                                                    unsigned int* status) {
    __shared__ int e_s[kMaxPlanPairs];
    __shared__ int start_s[kMaxPlanPairs];
    __shared__ int slot_e[kMaxPlanPairs];
    // Let the projections that follow start their prologue; the ids may come from
    // the previous kernel.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int i = int(threadIdx.x);
    const int G = n;
    int e = -1;
    if (i < n) e = __ldg(ids + i);
    const bool bad_here = i < n && (e < 0 || e >= n_experts);
    if (i < n) e_s[i] = e;
    if (__syncthreads_or(bad_here)) {
        if (i == 0) {
            plan[0] = 0;
            atomicOr(status, kStatusBadPlan);
        }
        return;
    }
    if (i < n) {
        int r = 0, w = 0;
        for (int j = 0; j < n; ++j) {
            const int f = e_s[j];
            r += (f < e) || (f == e && j < i);
            w += (f == e && j < i);
        }
        plan[plan_slot_pair(G) + r] = i;
        plan[plan_slot_token(G) + r] = i / topk;
        plan[plan_pair_slot(G) + i] = r;
        start_s[r] = (w % kMaxNtok) == 0;
        slot_e[r] = e;
    }
    __syncthreads();
    const int ng = __syncthreads_count(i < n && start_s[i]);
    if (i < n && start_s[i]) {
        int g = 0;
        for (int q = 0; q < i; ++q) g += start_s[q];
        plan[plan_group_start(G) + g] = i;
        plan[plan_group_expert(G) + g] = slot_e[i];
    }
    for (int g = ng + i; g <= G; g += int(blockDim.x)) {
        plan[plan_group_start(G) + g] = G;
        if (g < G) plan[plan_group_expert(G) + g] = -1;
    }
    if (i == 0) plan[0] = ng;
}

qg_status plan_experts(int fmt, int64_t n_out, int64_t n_in, Plan* plan) {
    int dev = 0, sms = 0, optin = 0;
    unsigned int* status = nullptr;
    qg_status st = device_info(&dev, &sms, &optin, &status);
    if (st != QG_OK) return st;
    Tile t = apply_override(select_expert_tile(fmt, n_out, n_in), current_override());
    if (!rpw_ok(t.rpw) || !depth_ok(t.depth) || t.warps < 1 || t.warps > kMaxWarps || t.ctas < 1) return QG_EINVAL;
    t.split = 1;
    t.rpw = t.rpw >= 4 ? 4 : t.rpw >= 2 ? 2 : 1;           // the instantiated rows per warp
    const void* fn = expert_kernel_lookup(fmt, t.rpw);
    auto cap_warps = [&]() {
        const int mw = fn ? max_threads(fn) / 32 : 0;
        if (mw < 1) return false;
        if (t.warps > mw) t.warps = mw;
        return true;
    };
    if (!cap_warps()) return QG_EUNSUPPORTED;
    // Sized for the largest plan (1024 slots); a launch allocates what its plan needs.
    auto total = [&](int depth, int warps) {
        return size_t(plan_smem_off(smem_plan(fmt, kMaxNtok, int(n_in), t.rpw, depth, warps, 1).total));
    };
    auto fits = [&]() {
        return total(t.depth, t.warps) + plan_smem_bytes(kMaxPlanPairs) + kStaticSmemReserve <= size_t(optin);
    };
    while (!fits() && t.depth > 2) --t.depth;
    while (!fits() && t.warps > 1) --t.warps;
    while (!fits() && t.rpw > 1) {
        t.rpw /= 2;
        fn = expert_kernel_lookup(fmt, t.rpw);
        if (!cap_warps()) return QG_EUNSUPPORTED;
    }
    const size_t smem = total(t.depth, t.warps);
    if (!fits()) return QG_EUNSUPPORTED;
    const int threads = 32 * t.warps;
    const int occ = blocks_per_sm(fn, dev, optin, threads, smem + plan_smem_bytes(kMaxPlanPairs));
    if (occ < 1) return QG_EUNSUPPORTED;
    int64_t grid = int64_t(sms) * std::min(t.ctas, occ);
    if (grid > kMaxGrid) grid = kMaxGrid;
    plan->fn = fn;
    plan->tile = t;
    plan->tile.ctas = std::min(t.ctas, occ);
    plan->tile.pre = t.depth;    // the expert kernels request a group's whole ring at once
    plan->grid = int(grid);
    plan->threads = threads;
    plan->smem = smem;
    plan->status = status;
    plan->seg_len = 0;
    return QG_OK;
}

// Expert plans cached per thread like the mat-vec's (key: device, shape, override).
struct PlanKey {
    int dev, fmt; int64_t n_out, n_in; uint64_t gen;
    bool operator==(const PlanKey& o) const {
        return dev == o.dev && fmt == o.fmt && n_out == o.n_out && n_in == o.n_in && gen == o.gen;
    }
};

qg_status plan_experts_cached(int fmt, int64_t n_out, int64_t n_in, Plan* plan) {
    constexpr int kSlots = 16;
    struct Slot { bool used = false; PlanKey key; Plan plan; };
    thread_local Slot cache[kSlots];
    read_env_override();
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return QG_ECUDA; }
    const PlanKey key{dev, fmt, n_out, n_in, override_generation()};
    const uint64_t h = (uint64_t(n_out) * 0x9E3779B97F4A7C15ull) ^ (uint64_t(n_in) * 0xC2B2AE3D27D4EB4Full) ^
                       uint64_t(fmt * 31 + dev * 131);
    Slot& sl = cache[(h ^ (h >> 29)) % kSlots];
    if (sl.used && sl.key == key) { *plan = sl.plan; return QG_OK; }
    const qg_status st = plan_experts(fmt, n_out, n_in, plan);
    if (st == QG_OK) { sl.used = true; sl.key = key; sl.plan = *plan; }
    return st;
}

qg_status launch_experts(const Plan& p, const ExpertArgs& args, void* stream) {
    ExpertArgs a = args;
    void* params[] = {&a};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(p.threads);
    cfg.dynamicSmemBytes = p.smem + plan_smem_bytes(a.n_slots);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    if (launch_flags() & QG_LAUNCH_EARLY_START) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if (cudaLaunchKernelExC(&cfg, p.fn, params) != cudaSuccess) { cudaGetLastError(); return QG_ECUDA; }
    return QG_OK;
}

}  // namespace
}  // namespace qg

using namespace qg;

extern "C" {

size_t qg_expert_plan_ints(int64_t n_pairs) {
    if (n_pairs < 1 || n_pairs > kMaxPlanPairs) return 0;
    return size_t(plan_ints(int(n_pairs)));
}

qg_status qg_expert_plan(const int32_t* ids, int ntok, int topk, int n_experts, int32_t* plan, void* stream) {
    if (!ids || !plan || ntok < 1 || topk < 1 || n_experts < 1) return QG_EINVAL;
    if (int64_t(ntok) * topk > kMaxPlanPairs) return QG_EINVAL;
    if (!aligned(ids, 4) || !aligned(plan, 4)) return QG_EALIGN;
    int dev = 0, sms = 0, optin = 0;
    unsigned int* status = nullptr;
    qg_status st = device_info(&dev, &sms, &optin, &status);
    if (st != QG_OK) return st;
    const int n = ntok * topk;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3((n + 31) / 32 * 32);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    if (launch_flags() & QG_LAUNCH_EARLY_START) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if (cudaLaunchKernelEx(&cfg, expert_plan_kernel, ids, n, topk, n_experts, plan, status) != cudaSuccess) {
        cudaGetLastError();
        return QG_ECUDA;
    }
    return QG_OK;
}

qg_status qgemv_experts(qg_fmt fmt, const void* W, int64_t n_experts, int64_t n_out, int64_t n_in, const float* x,
                        int64_t n_x, unsigned int flags, const int32_t* plan, int64_t n_slots, float* y,
                        const void* W_next, int64_t next_n_out, int64_t next_n_in, void* stream) {
    if (n_experts < 1 || n_out < 1 || n_experts > ((int64_t(1) << 31) - 1) / n_out) return QG_EINVAL;
    if (!shape_valid(fmt, n_experts * n_out, n_in)) return QG_EINVAL;
    if (n_slots < 1 || n_slots > kMaxPlanPairs || n_x < 1 || n_x > (int64_t(1) << 31) - 1) return QG_EINVAL;
    if (flags & ~(QG_EXPERTS_X_BY_SLOT | QG_EXPERTS_PLAN_READY | QG_EXPERTS_SWIGLU)) return QG_EINVAL;
    if ((flags & QG_EXPERTS_SWIGLU) && (n_out % 2) != 0) return QG_EINVAL;
    if ((flags & QG_EXPERTS_X_BY_SLOT) && n_x < n_slots) return QG_EINVAL;
    if (!W || !x || !plan || !y) return QG_EINVAL;
    if (W_next) {
        if (next_n_out < 1 || n_experts > ((int64_t(1) << 31) - 1) / next_n_out) return QG_EINVAL;
        if (!shape_valid(fmt, n_experts * next_n_out, next_n_in)) return QG_EINVAL;
    }
    if (!aligned(W, 16) || !aligned(x, 16) || !aligned(plan, 4) || !aligned(y, 4) || !aligned(W_next, 16))
        return QG_EALIGN;
    Plan p;
    qg_status st = plan_experts_cached(fmt, n_out, n_in, &p);
    if (st != QG_OK) return st;
    if ((flags & QG_EXPERTS_SWIGLU) && (p.tile.rpw % 2) != 0) return QG_EUNSUPPORTED;   // gate/up pairs per block
    ExpertArgs a{};
    st = encode_weight_map(&a.wmap, fmt, W, n_experts * n_out, n_in, p.tile.rpw);
    if (st != QG_OK) return st;
    a.x = x;
    a.y = y;
    a.plan = plan;
    a.status = p.status;
    a.n_experts = int(n_experts);
    a.n_out = int(n_out);
    a.n_in = int(n_in);
    a.n_slots = int(n_slots);
    a.n_x = int(n_x);
    a.flags = flags;
    a.depth = p.tile.depth;
    a.wait_limit = wait_limit();
    a.drain_limit = std::max<uint32_t>(a.wait_limit, 1u << 16);
    a.test_extra_tx = test_extra_tx();
    a.stage_tx = uint32_t(p.tile.rpw * full_step_bytes(fmt));
    a.next_w = static_cast<const unsigned char*>(W_next);
    a.next_bytes = W_next ? (long long)(next_n_out * row_stride(fmt, next_n_in)) : 0;
    a.group_base = p.tile.gw;
    return launch_experts(p, a, stream);
}

size_t qgemv_expert_layer_workspace_bytes(void) { return size_t(1 + kMaxPlanPairs) * 4 + 12; }   // 4112

qg_status qgemv_expert_layer(qg_fmt fmt, const void* W_gate_up, const void* W_down, int64_t n_experts, int64_t d_model,
                             int64_t d_ff, const float* x, int ntok, const int32_t* ids, int topk, int32_t* plan,
                             float* act, float* y, void* workspace, size_t workspace_bytes, void* stream) {
    const int64_t kMaxRows = (int64_t(1) << 31) - 1;
    if (n_experts < 1 || d_model < 1 || d_ff < 1) return QG_EINVAL;
    if (n_experts > kMaxRows / (2 * d_ff) || n_experts > kMaxRows / d_model) return QG_EINVAL;
    if (!shape_valid(fmt, n_experts * 2 * d_ff, d_model) || !shape_valid(fmt, n_experts * d_model, d_ff))
        return QG_EINVAL;
    if (ntok < 1 || topk < 1 || int64_t(ntok) * topk > kMaxPlanPairs) return QG_EINVAL;
    if (!W_gate_up || !W_down || !x || !ids || !plan || !act || !y) return QG_EINVAL;
    if (!aligned(W_gate_up, 16) || !aligned(W_down, 16) || !aligned(x, 16) || !aligned(act, 16) || !aligned(y, 4) ||
        !aligned(plan, 4) || !aligned(ids, 4))
        return QG_EALIGN;
    if (!workspace || workspace_bytes < qgemv_expert_layer_workspace_bytes()) return QG_EWORKSPACE;
    if (!aligned(workspace, 16)) return QG_EALIGN;
    int dev = 0, sms = 0, optin = 0;
    unsigned int* status = nullptr;
    qg_status st = device_info(&dev, &sms, &optin, &status);
    if (st != QG_OK) return st;
    const int G = ntok * topk;
    const int max_in = int(std::max(d_model, d_ff));
    Tile t = apply_override(select_expert_tile(fmt, 2 * d_ff, d_model), current_override());
    if (!depth_ok(t.depth) || t.warps < 1 || t.warps > kMaxWarps || t.ctas < 1) return QG_EINVAL;
    t.split = 1;
    t.rpw = t.rpw >= 4 ? 4 : 2;                                 // gate/up pairs: an even row count
    const void* fn = expert_layer_kernel_lookup(fmt, t.rpw);
    if (!fn) return QG_EUNSUPPORTED;
    t.warps = std::min(t.warps, max_threads(fn) / 32);
    auto total = [&](int depth, int warps) {
        return size_t(plan_smem_off(smem_plan(fmt, kMaxNtok, max_in, t.rpw, depth, warps, 1).total)) +
               size_t(plan_build_bytes(G));
    };
    while (total(t.depth, t.warps) + kStaticSmemReserve > size_t(optin) && t.depth > 2) --t.depth;
    while (total(t.depth, t.warps) + kStaticSmemReserve > size_t(optin) && t.warps > 1) --t.warps;
    const size_t smem = total(t.depth, t.warps);
    if (t.warps < 1 || smem + kStaticSmemReserve > size_t(optin)) return QG_EUNSUPPORTED;
    const int threads = 32 * t.warps;
    const int occ = blocks_per_sm(fn, dev, optin, threads, smem);
    if (occ < 1) return QG_EUNSUPPORTED;
    // Every CTA must be resident at once (they meet at the grid barrier).
    const int grid = int(std::min<int64_t>(int64_t(sms) * std::min(t.ctas, occ), kMaxGrid));

    LayerArgs L{};
    st = encode_weight_map(&L.gu.wmap, fmt, W_gate_up, n_experts * 2 * d_ff, d_model, t.rpw);
    if (st != QG_OK) return st;
    st = encode_weight_map(&L.dn.wmap, fmt, W_down, n_experts * d_model, d_ff, t.rpw);
    if (st != QG_OK) return st;
    const uint32_t wl = wait_limit();
    for (ExpertArgs* a : {&L.gu, &L.dn}) {
        a->group_base = t.gw;
        a->status = status;
        a->n_experts = int(n_experts);
        a->n_slots = G;
        a->depth = t.depth;
        a->wait_limit = wl;
        a->drain_limit = std::max<uint32_t>(wl, 1u << 16);
        a->test_extra_tx = test_extra_tx();
        a->stage_tx = uint32_t(t.rpw * full_step_bytes(fmt));
    }
    L.gu.x = x;
    L.gu.y = act;
    L.gu.n_out = int(2 * d_ff);
    L.gu.n_in = int(d_model);
    L.gu.n_x = ntok;
    L.gu.flags = QG_EXPERTS_SWIGLU;
    L.gu.next_w = static_cast<const unsigned char*>(W_down);
    L.gu.next_bytes = (long long)(d_model * row_stride(fmt, d_ff));
    L.dn.x = act;
    L.dn.y = y;
    L.dn.n_out = int(d_model);
    L.dn.n_in = int(d_ff);
    L.dn.n_x = G;
    L.dn.flags = QG_EXPERTS_X_BY_SLOT;
    L.ids = ids;
    L.topk = topk;
    L.plan_out = plan;
    L.barrier = static_cast<unsigned int*>(workspace);
    L.barrier_limit = std::max<uint32_t>(wl, 1u << 16) / 4u;   // ~1 s of polls by default

    void* params[] = {&L};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    // A cooperative launch: the driver starts the grid only when every CTA can be
    // resident at once, so the CTAs that meet at the barriers never wait on a CTA that
    // other work keeps off the GPU (the bounded waits stay as a guard).  Early start is
    // added when enabled; if the driver refuses the two together, the layer launches
    // cooperatively without it.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (launch_flags() & QG_LAUNCH_EARLY_START) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, params);
    if (e != cudaSuccess && cfg.numAttrs == 2) {
        cudaGetLastError();
        cfg.numAttrs = 1;
        e = cudaLaunchKernelExC(&cfg, fn, params);
    }
    if (e != cudaSuccess) { cudaGetLastError(); return QG_ECUDA; }
    return QG_OK;
}

qg_status qg_describe_expert_tile(qg_fmt fmt, int64_t n_out, int64_t n_in, char* buf, size_t len) {
    if (!buf || len == 0) return QG_EINVAL;
    if (!shape_valid(fmt, n_out, n_in)) return QG_EINVAL;
    Plan p;
    qg_status st = plan_experts(fmt, n_out, n_in, &p);
    if (st != QG_OK) return st;
    std::snprintf(buf, len, "%s,gw=%d,grid=%d", tile_to_string(p.tile).c_str(), p.tile.gw, p.grid);
    return QG_OK;
}

}  // extern "C"

