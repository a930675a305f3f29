// C ABI entry points of the mat-vec: validation, tile selection, launch, and the host
// helpers the expert calls (qgemv_experts.cu) share.  The operation and every argument
// rule are documented in include/qgemv.h.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "qgemv_kernels.cuh"
#include "qgemv_host.h"
#include "tile_select.h"

namespace qg {

const void* kernel_lookup_fmt0(int, int, bool, bool);
const void* kernel_lookup_fmt1(int, int, bool, bool);
const void* kernel_lookup_fmt2(int, int, bool, bool);
const void* kernel_lookup_fmt3(int, int, bool, bool);
const void* kernel_lookup_fmt4(int, int, bool, bool);

const void* kernel_lookup(int fmt, int ntok, int rpw, bool argmax, bool split) {
    switch (fmt) {
        case 0: return kernel_lookup_fmt0(ntok, rpw, argmax, split);
        case 1: return kernel_lookup_fmt1(ntok, rpw, argmax, split);
        case 2: return kernel_lookup_fmt2(ntok, rpw, argmax, split);
        case 3: return kernel_lookup_fmt3(ntok, rpw, argmax, split);
        case 4: return kernel_lookup_fmt4(ntok, rpw, argmax, split);
        default: return nullptr;
    }
}

// Device status word: kernels OR bits into it (kStatusWaitTimeout when a bounded
// mbarrier wait gave up); read and cleared by qg_device_status.
__device__ unsigned int g_device_status;

namespace {
constexpr int kMaxDevices = 64;

// Per-device constants, read once.
struct DevInfo {
    std::atomic<int> sms{0};
    std::atomic<int> smem_optin{0};
    std::atomic<unsigned int*> status{nullptr};
};
DevInfo g_dev[kMaxDevices];

// Test hook values (qg_set_wait_limit).
std::atomic<uint32_t> g_wait_limit{kWaitLimit};
std::atomic<uint32_t> g_test_extra_tx{0};

// Profiling hook (qg_set_phase_record): the buffer, its slot count, the launch counter.
std::mutex g_phase_mu;
unsigned long long* g_phase_buf = nullptr;
int64_t g_phase_slots = 0, g_phase_next = 0;

// Tile override: QGEMV_TILE at first use, or qg_set_tile_override.
std::mutex g_override_mu;
std::atomic<uint64_t> g_override_gen{1};   // bumped whenever the override changes (plan cache key)
TileOverride g_override;
std::once_flag g_env_once;

}  // namespace

void read_env_override() {
    std::call_once(g_env_once, [] {
        const char* e = std::getenv("QGEMV_TILE");
        TileOverride o;
        if (e && parse_tile_spec(e, &o)) {
            std::lock_guard<std::mutex> lk(g_override_mu);
            g_override = o;
        }
    });
}

TileOverride current_override() {
    read_env_override();
    std::lock_guard<std::mutex> lk(g_override_mu);
    return g_override;
}

// ---- host helpers shared with the expert calls (declared in qgemv_host.h)

uint64_t override_generation() { return g_override_gen.load(std::memory_order_acquire); }
uint32_t wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }
uint32_t test_extra_tx() { return g_test_extra_tx.load(std::memory_order_relaxed); }

namespace {
// Occupancy, cached per (kernel, device, threads, smem bytes).  The first use of a
// kernel on a device raises its dynamic shared memory limit to the device maximum.
std::mutex g_occ_mu;
std::map<std::tuple<const void*, int, size_t, int>, int> g_occ;
std::map<std::pair<const void*, int>, bool> g_configured;
}  // namespace

qg_status device_info(int* dev, int* sms, int* smem_optin, unsigned int** status) {
    if (cudaGetDevice(dev) != cudaSuccess) { cudaGetLastError(); return QG_ECUDA; }
    if (*dev < 0 || *dev >= kMaxDevices) return QG_EUNSUPPORTED;
    DevInfo& d = g_dev[*dev];
    int s = d.sms.load(std::memory_order_acquire);
    int m = d.smem_optin.load(std::memory_order_acquire);
    unsigned int* st = d.status.load(std::memory_order_acquire);
    if (s == 0 || m == 0 || st == nullptr) {
        void* addr = nullptr;
        if (cudaDeviceGetAttribute(&s, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&m, cudaDevAttrMaxSharedMemoryPerBlockOptin, *dev) != cudaSuccess ||
            cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) {
            cudaGetLastError();
            return QG_ECUDA;
        }
        st = static_cast<unsigned int*>(addr);
        d.sms.store(s, std::memory_order_release);
        d.smem_optin.store(m, std::memory_order_release);
        d.status.store(st, std::memory_order_release);
    }
    *sms = s;
    *smem_optin = m;
    if (status) *status = st;
    return QG_OK;
}

// Blocks of `fn` resident per SM with `threads` threads and `smem` dynamic bytes (0 on error).
int blocks_per_sm(const void* fn, int dev, int optin, int threads, size_t smem) {
    auto key = std::make_tuple(fn, dev, smem, threads);
    std::lock_guard<std::mutex> lk(g_occ_mu);
    auto it = g_occ.find(key);
    if (it != g_occ.end()) return it->second;
    auto ck = std::make_pair(fn, dev);
    if (!g_configured[ck]) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess ||
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - int(fa.sharedSizeBytes)) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        g_configured[ck] = true;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    g_occ[key] = n;
    return n;
}

// Threads per block a kernel allows (its launch bound), cached per kernel.
int max_threads(const void* fn) {
    static std::mutex mu;
    static std::map<const void*, int> cache;
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(fn);
    if (it != cache.end()) return it->second;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) { cudaGetLastError(); return 0; }
    cache[fn] = fa.maxThreadsPerBlock;
    return fa.maxThreadsPerBlock;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

namespace {

// Everything up to the launch.  Checks that need no CUDA call come first.
qg_status plan_launch(int fmt, int64_t n_out, int64_t n_in, int ntok, bool argmax, Plan* plan) {
    int dev = 0, sms = 0, optin = 0;
    unsigned int* status = nullptr;
    qg_status st = device_info(&dev, &sms, &optin, &status);
    if (st != QG_OK) return st;
    Tile t = apply_override(select_tile(fmt, n_out, n_in, ntok), current_override());
    if (!rpw_ok(t.rpw) || !depth_ok(t.depth) || t.warps < 1 || t.warps > kMaxWarps || t.ctas < 1 ||
        t.split < 0 || t.split > kMaxSplit)
        return QG_EINVAL;
    // Split: the shape's default unless overridden, at most one segment per step;
    // segments of L steps (the last may be shorter), none empty.  The warps of a CTA
    // are a whole number of teams.
    // The split is lowered until one team fits in shared memory in the worst case
    // (ntok 4, one row per warp, a 2-stage ring), so it is the same for every ntok.
    const int spr = int(steps_per_row(fmt, n_in));
    int P = t.split > 0 ? t.split : select_split(fmt, n_out, n_in);
    if (P > spr) P = spr;
    while (P > 1 && size_t(smem_plan(fmt, kMaxNtok, int(n_in), 1, 2, P, P).total) + kStaticSmemReserve >
                        size_t(optin))
        --P;
    const int L = (spr + P - 1) / P;
    P = (spr + L - 1) / L;
    t.split = P;
    if (t.warps < P) t.warps = P;
    t.warps -= t.warps % P;
    const void* fn = kernel_lookup(fmt, ntok, t.rpw, argmax, P > 1);
    if (!fn) return QG_EUNSUPPORTED;
    // The kernel's thread limit (12 warps where a warp keeps more than 16 outputs).
    auto cap_warps = [&]() {
        const int mw = max_threads(fn) / 32;
        if (mw < 1) return false;
        if (t.warps > mw) t.warps = mw - mw % P;
        return t.warps >= P;
    };
    if (!cap_warps()) return QG_EUNSUPPORTED;
    // Shrink the ring, then the warps (whole teams), then the rows per warp (to the
    // next smaller instantiated value) until the CTA fits in shared memory; x alone
    // must fit.
    auto total = [&](int depth, int warps) {
        return size_t(smem_plan(fmt, ntok, int(n_in), t.rpw, depth, warps, P).total);
    };
    auto fits = [&]() { return total(t.depth, t.warps) + kStaticSmemReserve <= size_t(optin); };
    while (!fits() && t.depth > 2) --t.depth;
    while (!fits() && t.warps > P) t.warps -= P;
    while (!fits() && t.rpw > 1) {
        int r = t.rpw - 1;
        while (r > 1 && !kernel_lookup(fmt, ntok, r, argmax, P > 1)) --r;
        t.rpw = r;
        fn = kernel_lookup(fmt, ntok, t.rpw, argmax, P > 1);
        if (!fn || !cap_warps()) return QG_EUNSUPPORTED;
    }
    const size_t smem = total(t.depth, t.warps);
    if (smem + kStaticSmemReserve > size_t(optin)) return QG_EUNSUPPORTED;
    const int threads = 32 * t.warps;
    const int occ = blocks_per_sm(fn, dev, optin, threads, smem);
    if (occ < 1) return QG_EUNSUPPORTED;
    // Groups are dealt to CTAs round-robin: every CTA up to one per group has work.
    const int64_t ngroups = (n_out + t.rpw - 1) / t.rpw;
    int64_t grid = int64_t(sms) * std::min(t.ctas, occ);
    if (ngroups < grid) grid = ngroups;
    if (grid > kMaxGrid) grid = kMaxGrid;
    if (grid < 1) grid = 1;
    plan->fn = fn;
    plan->tile = t;
    plan->tile.ctas = std::min(t.ctas, occ);
    plan->tile.pre = t.pre <= 0 ? 1 : std::min(t.pre, t.depth);
    plan->grid = int(grid);
    plan->threads = threads;
    plan->smem = smem;
    plan->status = status;
    plan->seg_len = L;
    return QG_OK;
}

// Plans cached per thread (a call's plan depends on the device, the shape, ntok,
// argmax and the override; the override's generation is part of the key), so a
// repeated call skips tile selection and the occupancy lookup.
struct PlanKey {
    int dev, fmt, ntok; int64_t n_out, n_in; bool argmax; uint64_t gen;
    bool operator==(const PlanKey& o) const {
        return dev == o.dev && fmt == o.fmt && ntok == o.ntok && n_out == o.n_out && n_in == o.n_in &&
               argmax == o.argmax && gen == o.gen;
    }
};

qg_status plan_launch_cached(int fmt, int64_t n_out, int64_t n_in, int ntok, bool argmax, Plan* plan) {
    constexpr int kSlots = 64;
    struct Slot { bool used = false; PlanKey key; Plan plan; };
    thread_local Slot cache[kSlots];
    read_env_override();
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return QG_ECUDA; }
    const PlanKey key{dev, fmt, ntok, n_out, n_in, argmax, g_override_gen.load(std::memory_order_acquire)};
    const uint64_t h = (uint64_t(n_out) * 0x9E3779B97F4A7C15ull) ^ (uint64_t(n_in) * 0xC2B2AE3D27D4EB4Full) ^
                       uint64_t(fmt * 31 + ntok * 7 + (argmax ? 3 : 0) + dev * 131);
    Slot& sl = cache[(h ^ (h >> 29)) % kSlots];
    if (sl.used && sl.key == key) { *plan = sl.plan; return QG_OK; }
    const qg_status st = plan_launch(fmt, n_out, n_in, ntok, argmax, plan);
    if (st == QG_OK) { sl.used = true; sl.key = key; sl.plan = *plan; }
    return st;
}

}  // namespace

// cuTensorMapEncodeTiled, fetched from the driver through the runtime once
// (the library links only the runtime).  Encoding is a host-only computation.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return EncodeTiledFn(nullptr);
        }
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// The packed matrix as a 2-D tensor of 8-byte elements: dim 0 = one row
// (row stride / 8 elements), dim 1 = the n_out rows; one box = one full step of
// rpw rows, so the box's rows land in shared memory one full step apart.
// Elements outside the tensor (rows >= n_out, bytes past a row's short last
// step, or past a row shorter than one step) are not read and arrive as zeros.
// Maps are cached per thread (32 slots) and reused when the same matrix and box come again.
qg_status encode_weight_map(CUtensorMap* map, int fmt, const void* W, int64_t n_out, int64_t n_in, int rpw) {
    struct Key {
        const void* W; int64_t n_out, n_in; int fmt, rpw;
        bool operator==(const Key& o) const {
            return W == o.W && n_out == o.n_out && n_in == o.n_in && fmt == o.fmt && rpw == o.rpw;
        }
    };
    constexpr int kSlots = 32;
    struct Slot { Key key{nullptr, 0, 0, -1, 0}; CUtensorMap map; };
    thread_local Slot cache[kSlots];
    const Key k{W, n_out, n_in, fmt, rpw};
    const uint64_t h = (reinterpret_cast<uintptr_t>(W) >> 8) * 0x9E3779B97F4A7C15ull ^
                       uint64_t(n_out) * 0xC2B2AE3D27D4EB4Full ^ uint64_t(n_in * 13 + fmt * 7 + rpw);
    Slot& sl = cache[(h ^ (h >> 31)) % kSlots];
    if (sl.key == k) { *map = sl.map; return QG_OK; }
    const EncodeTiledFn enc = encode_tiled();
    if (!enc) return QG_ECUDA;
    const int64_t stride = row_stride(fmt, n_in);
    const cuuint64_t dims[2] = {cuuint64_t(stride / 8), cuuint64_t(n_out)};
    const cuuint64_t strides[1] = {cuuint64_t(stride)};
    const cuuint32_t box[2] = {cuuint32_t(full_step_bytes(fmt) / 8), cuuint32_t(rpw)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(W), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return QG_ECUDA;
    sl.key = k;
    sl.map = *map;
    return QG_OK;
}

namespace {

qg_status fill_common(KernelArgs& a, const Plan& p, int fmt, const void* W, int64_t n_out, int64_t n_in,
                      const float* x, float* y) {
    const qg_status st = encode_weight_map(&a.wmap, fmt, W, n_out, n_in, p.tile.rpw);
    if (st != QG_OK) return st;
    a.x = x;
    a.y = y;
    a.status = p.status;
    a.n_out = int(n_out);
    a.n_in = int(n_in);
    a.depth = p.tile.depth;
    a.split = p.tile.split;
    a.seg_len = p.seg_len;
    a.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
    a.drain_limit = std::max<uint32_t>(a.wait_limit, 1u << 16);
    a.test_extra_tx = g_test_extra_tx.load(std::memory_order_relaxed);
    a.stage_tx = uint32_t(p.tile.rpw * full_step_bytes(fmt));
    a.pre = p.tile.pre;
    a.phase = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_phase_mu);
        if (g_phase_buf) {
            a.phase = g_phase_buf + size_t(g_phase_next) * QG_PHASE_SLOT_WORDS;
            g_phase_next = (g_phase_next + 1) % g_phase_slots;
        }
    }
    return QG_OK;
}

qg_status check_common(int fmt, const void* W, int64_t n_out, int64_t n_in, const float* x, int ntok) {
    if (!shape_valid(fmt, n_out, n_in)) return QG_EINVAL;
    if (ntok < 1 || ntok > kMaxNtok) return QG_EINVAL;
    if (!W || !x) return QG_EINVAL;
    if (!aligned(W, 16) || !aligned(x, 16)) return QG_EALIGN;
    return QG_OK;
}

// Launch options (qg_set_launch_options / QGEMV_EARLY_START).
std::atomic<unsigned> g_launch_flags{0};
std::once_flag g_launch_env_once;
}  // namespace

unsigned launch_flags() {
    std::call_once(g_launch_env_once, [] {
        const char* e = std::getenv("QGEMV_EARLY_START");
        if (e && e[0] == '1') g_launch_flags.fetch_or(QG_LAUNCH_EARLY_START);
    });
    return g_launch_flags.load(std::memory_order_relaxed);
}

namespace {

qg_status launch(const Plan& p, const KernelArgs& args, void* stream) {
    KernelArgs a = args;
    void* params[] = {&a};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(p.threads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    if (launch_flags() & QG_LAUNCH_EARLY_START) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    cudaError_t e = cudaLaunchKernelExC(&cfg, p.fn, params);
    if (e != cudaSuccess) { cudaGetLastError(); return QG_ECUDA; }
    return QG_OK;
}

}  // namespace
}  // namespace qg

using namespace qg;

extern "C" {

const char* qg_strerror(qg_status s) {
    switch (s) {
        case QG_OK: return "ok";
        case QG_EINVAL: return "invalid argument (format, size, ntok or null pointer)";
        case QG_EALIGN: return "pointer not aligned (W, x and workspace need 16 bytes; y and argmax 4)";
        case QG_EUNSUPPORTED: return "unsupported shape or device (n_in too large for shared memory?)";
        case QG_EWORKSPACE: return "argmax workspace missing or smaller than qgemv_argmax_workspace_bytes()";
        case QG_ECUDA: return "CUDA runtime error at launch";
        default: return "unknown status";
    }
}

int qg_abi_version(void) { return 1; }

qg_status qgemv(qg_fmt fmt, const void* W, int64_t n_out, int64_t n_in, const float* x, float* y,
                int ntok, void* stream) {
    qg_status st = check_common(fmt, W, n_out, n_in, x, ntok);
    if (st != QG_OK) return st;
    if (!y) return QG_EINVAL;
    if (!aligned(y, 4)) return QG_EALIGN;
    Plan p;
    st = plan_launch_cached(fmt, n_out, n_in, ntok, false, &p);
    if (st != QG_OK) return st;
    KernelArgs a{};
    st = fill_common(a, p, fmt, W, n_out, n_in, x, y);
    if (st != QG_OK) return st;
    return launch(p, a, stream);
}

size_t qgemv_argmax_workspace_bytes(int64_t n_out, int ntok) {
    if (n_out < 1 || ntok < 1 || ntok > kMaxNtok) return 0;
    return 16 + size_t(kMaxGrid) * size_t(ntok) * sizeof(ArgmaxPartial);
}

}  // extern "C"

namespace qg {
namespace {

qg_status argmax_call(int fmt, const void* W, int64_t n_out, int64_t n_in, const float* x, float* y,
                      int32_t* argmax, int ntok, const int32_t* row_ids, void* workspace, size_t workspace_bytes,
                      void* stream) {
    qg_status st = check_common(fmt, W, n_out, n_in, x, ntok);
    if (st != QG_OK) return st;
    if (!argmax) return QG_EINVAL;
    if ((y && !aligned(y, 4)) || !aligned(argmax, 4) || (row_ids && !aligned(row_ids, 4))) return QG_EALIGN;
    if (!workspace || workspace_bytes < qgemv_argmax_workspace_bytes(n_out, ntok)) return QG_EWORKSPACE;
    if (!aligned(workspace, 16)) return QG_EALIGN;
    Plan p;
    st = plan_launch_cached(fmt, n_out, n_in, ntok, true, &p);
    if (st != QG_OK) return st;
    KernelArgs a{};
    st = fill_common(a, p, fmt, W, n_out, n_in, x, y);
    if (st != QG_OK) return st;
    a.argmax = argmax;
    a.row_ids = row_ids;
    a.ticket = static_cast<unsigned int*>(workspace);
    a.partials = reinterpret_cast<ArgmaxPartial*>(static_cast<uint8_t*>(workspace) + 16);
    return launch(p, a, stream);
}

// Row gather: block-strided over the listed rows, each row copied as 16-byte words.
// An id outside [0, n_out) gets a zero row and sets kStatusBadRowId (no access
// outside the source).
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                          const int32_t* __restrict__ ids, long long n_ids,
                                                          long long n_out, int row16, unsigned int* status) {
    for (long long j = blockIdx.x; j < n_ids; j += gridDim.x) {
        const int id = __ldg(ids + j);
        uint4* d = dst + j * row16;
        if (id < 0 || id >= n_out) {
            for (int k = threadIdx.x; k < row16; k += blockDim.x) d[k] = make_uint4(0u, 0u, 0u, 0u);
            if (threadIdx.x == 0) atomicOr(status, kStatusBadRowId);
        } else {
            const uint4* r = src + (long long)id * row16;
            for (int k = threadIdx.x; k < row16; k += blockDim.x) d[k] = __ldg(r + k);
        }
    }
}

}  // namespace
}  // namespace qg

extern "C" {

qg_status qgemv_argmax(qg_fmt fmt, const void* W, int64_t n_out, int64_t n_in, const float* x, float* y,
                       int32_t* argmax, int ntok, void* workspace, size_t workspace_bytes, void* stream) {
    return argmax_call(fmt, W, n_out, n_in, x, y, argmax, ntok, nullptr, workspace, workspace_bytes, stream);
}

qg_status qgemv_argmax_ids(qg_fmt fmt, const void* W_sub, int64_t n_sub, int64_t n_in, const float* x, float* y,
                           int32_t* argmax, int ntok, const int32_t* ids, void* workspace, size_t workspace_bytes,
                           void* stream) {
    if (!ids) return QG_EINVAL;
    return argmax_call(fmt, W_sub, n_sub, n_in, x, y, argmax, ntok, ids, workspace, workspace_bytes, stream);
}

qg_status qg_gather_rows(qg_fmt fmt, const void* W, int64_t n_out, int64_t n_in, const int32_t* ids, int64_t n_ids,
                         void* W_out, void* stream) {
    if (!shape_valid(fmt, n_out, n_in)) return QG_EINVAL;
    if (!W || !ids || !W_out || n_ids < 1 || n_ids > (int64_t(1) << 31) - 1) return QG_EINVAL;
    if (!aligned(W, 16) || !aligned(W_out, 16) || !aligned(ids, 4)) return QG_EALIGN;
    int dev = 0, sms = 0, optin = 0;
    unsigned int* status = nullptr;
    qg_status st = device_info(&dev, &sms, &optin, &status);
    if (st != QG_OK) return st;
    const int64_t stride = row_stride(fmt, n_in);
    const long long grid = std::min<long long>(n_ids, (long long)sms * 8);
    gather_rows_kernel<<<unsigned(grid), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(W), static_cast<uint4*>(W_out), ids, n_ids, n_out, int(stride / 16), status);
    if (cudaGetLastError() != cudaSuccess) return QG_ECUDA;
    return QG_OK;
}

qg_status qg_set_tile_override(const char* spec) {
    read_env_override();
    TileOverride o;
    if (!parse_tile_spec(spec, &o)) return QG_EINVAL;
    std::lock_guard<std::mutex> lk(g_override_mu);
    g_override = o;
    g_override_gen.fetch_add(1);
    return QG_OK;
}

qg_status qg_device_status(int clear, unsigned int* status) {
    if (!status) return QG_EINVAL;
    int dev = 0, sms = 0, optin = 0;
    unsigned int* addr = nullptr;
    qg_status st = device_info(&dev, &sms, &optin, &addr);
    if (st != QG_OK) return st;
    unsigned int v = 0;
    if (cudaMemcpy(&v, addr, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) { cudaGetLastError(); return QG_ECUDA; }
    if (clear && v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(addr, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaGetLastError();
            return QG_ECUDA;
        }
    }
    *status = v;
    return QG_OK;
}

qg_status qg_set_launch_options(unsigned int flags) {
    if (flags & ~unsigned(QG_LAUNCH_EARLY_START)) return QG_EINVAL;
    launch_flags();                       // consume the environment first, then override it
    g_launch_flags.store(flags, std::memory_order_relaxed);
    return QG_OK;
}

qg_status qg_set_wait_limit(uint32_t polls, uint32_t extra_tx_bytes) {
    g_wait_limit.store(polls == 0 ? kWaitLimit : polls, std::memory_order_relaxed);
    g_test_extra_tx.store(extra_tx_bytes, std::memory_order_relaxed);
    return QG_OK;
}

qg_status qg_set_phase_record(unsigned long long* buf, int64_t slots) {
    if (buf && slots < 1) return QG_EINVAL;
    if (buf && !aligned(buf, 8)) return QG_EALIGN;
    std::lock_guard<std::mutex> lk(g_phase_mu);
    g_phase_buf = buf;
    g_phase_slots = buf ? slots : 0;
    g_phase_next = 0;
    return QG_OK;
}

qg_status qg_describe_tile(qg_fmt fmt, int64_t n_out, int64_t n_in, int ntok, char* buf, size_t len) {
    if (!buf || len == 0) return QG_EINVAL;
    if (!shape_valid(fmt, n_out, n_in) || ntok < 1 || ntok > kMaxNtok) return QG_EINVAL;
    Plan p;
    qg_status st = plan_launch(fmt, n_out, n_in, ntok, false, &p);
    if (st != QG_OK) return st;
    std::snprintf(buf, len, "%s,grid=%d", tile_to_string(p.tile).c_str(), p.grid);
    return QG_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ no-allocation variant
// qgemv_argmax_noalloc: the fused LM-head argmax for callers that cannot call
// cudaMalloc.  Its scratch (the CTA ticket and the per-CTA partial maxima) is a
// fixed array in this library's device image instead of a caller-provided
// workspace.  Nothing here allocates: the array exists on every GPU the
// library is loaded on, for the life of the process.
namespace qg {
namespace {

constexpr int kNoAllocMaxGrid = 1024;        // CTAs whose partials fit in the array
constexpr size_t kNoAllocScratchBytes = 16 + size_t(kNoAllocMaxGrid) * kMaxNtok * sizeof(ArgmaxPartial);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch per device, looked up once per device and
// context: a device reset gives the device a new context, in which the library's
// module (and the array) may sit at another address, so a change of the current
// context repeats the lookup.
struct NoAllocSlot {
    std::mutex mu;
    void* ctx = nullptr;
    void* addr = nullptr;
};
NoAllocSlot g_noalloc[kMaxDevices];

// cuCtxGetCurrent, fetched from the driver through the runtime once (the library
// links only the runtime).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
    static const CtxGetCurrentFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return CtxGetCurrentFn(nullptr);
        }
        return reinterpret_cast<CtxGetCurrentFn>(f);
    }();
    return fn;
}

}  // namespace
}  // namespace qg

extern "C" qg_status qgemv_argmax_noalloc(qg_fmt fmt, const void* W, int64_t n_out, int64_t n_in,
                                          const float* x, float* y, int32_t* argmax, int ntok,
                                          void* stream) {
    qg_status st = check_common(fmt, W, n_out, n_in, x, ntok);
    if (st != QG_OK) return st;
    if (!argmax) return QG_EINVAL;
    if ((y && !aligned(y, 4)) || !aligned(argmax, 4)) return QG_EALIGN;

    // Set-up, once per device (and again after a device reset), with that device
    // current: the host-side name of the array is only a stand-in, so ask the runtime
    // for its device address.
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return QG_ECUDA; }
    if (dev < 0 || dev >= kMaxDevices) return QG_EUNSUPPORTED;
    void* scratch = nullptr;
    {
        CUcontext ctx = nullptr;
        const CtxGetCurrentFn get = ctx_get_current();
        if (get && get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
        NoAllocSlot& slot = g_noalloc[dev];
        std::lock_guard<std::mutex> lk(slot.mu);
        if (slot.addr == nullptr || ctx == nullptr || slot.ctx != static_cast<void*>(ctx)) {
            // (The lookup makes the device's primary context current if none was.)
            void* a = nullptr;
            if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess || a == nullptr) {
                cudaGetLastError();
                return QG_ECUDA;
            }
            if (ctx == nullptr && get && get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
            slot.addr = a;
            slot.ctx = ctx;
        }
        scratch = slot.addr;
    }

    Plan p;
    st = plan_launch_cached(fmt, n_out, n_in, ntok, true, &p);
    if (st != QG_OK) return st;
    // The launch needs a ticket plus one partial per CTA and token; refuse a launch
    // geometry (possible only through a tile override) that the array cannot hold.
    const size_t need = 16 + size_t(p.grid) * size_t(ntok) * sizeof(ArgmaxPartial);
    if (need > kNoAllocScratchBytes) return QG_EWORKSPACE;

    KernelArgs a{};
    st = fill_common(a, p, fmt, W, n_out, n_in, x, y);
    if (st != QG_OK) return st;
    // The array keeps whatever the last call left; the ticket must start at zero.
    if (cudaMemsetAsync(scratch, 0, 16, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return QG_ECUDA;
    }
    a.argmax = argmax;
    a.ticket = static_cast<unsigned int*>(scratch);
    a.partials = reinterpret_cast<ArgmaxPartial*>(static_cast<uint8_t*>(scratch) + 16);
    return launch(p, a, stream);
}
