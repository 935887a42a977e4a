// abi.cu -- the C ABI: argument validation, the tile policy, workspace
// management, TMA descriptor encoding and kernel dispatch.
//
// Tile policy.  The pages' prior art (atlas pull request #266, "What it
// does") tiles n >= 4 decode tokens greedily into tiles of 3, then a 2 or 1
// remainder, each tile reading W once (n = 8 -> 3 weight reads).  The default
// here is ONE_PASS: all n <= 16 tokens share one read of W; the greedy tiling
// stays available (NVFP4_TILING_GREEDY_321) to measure against.  Either way
// each pass is one launch of the same kernel on a contiguous token slice, so
// every token's result is computed exactly as a single-token call computes it
// (the same pull request's "Correctness argument").
#include "../../include/nvfp4_gemv.h"
#include "internal.h"

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

namespace nvfp4 {

static thread_local std::string t_last_error;

void set_last_error(const char *msg) { t_last_error = msg ? msg : ""; }

static nvfp4_status fail(nvfp4_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
static nvfp4_status fail(nvfp4_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

static nvfp4_status cuda_fail(cudaError_t e, const char *what) {
    return fail(NVFP4_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ------------------------------------------------------------ device state
struct DeviceState {
    bool ready = false;
    int sms = 0;
    int smem_optin = 0;
    int major = 0, minor = 0;
    unsigned *err_word = nullptr;
};

struct WorkspaceEntry {
    int device;
    cudaStream_t stream;
    void *ptr;
    size_t bytes;
};

static std::mutex g_mutex;
static std::vector<DeviceState> g_devices;
static std::vector<WorkspaceEntry> g_workspaces;

static nvfp4_status device_state(int dev, DeviceState **out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if ((int)g_devices.size() <= dev) g_devices.resize(dev + 1);
    DeviceState &d = g_devices[dev];
    if (!d.ready) {
        cudaError_t e;
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
        if ((e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(smem opt-in)");
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (d.major != 10 || d.minor != 3)
            return fail(NVFP4_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                        d.major, d.minor);
        if ((e = stream_set_smem_limits(d.smem_optin)) != cudaSuccess)
            return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");
        if ((e = tc_set_smem_limit(d.smem_optin)) != cudaSuccess)
            return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory, tcgen05 kernel)");
        if ((e = f4_set_smem_limit(d.smem_optin)) != cudaSuccess)
            return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory, block-scaled FP4 kernel)");
        if ((e = moe_set_smem_limit(d.smem_optin)) != cudaSuccess)
            return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory, grouped expert kernel)");
        if ((e = moe_mma_set_smem_limit(d.smem_optin)) != cudaSuccess)
            return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory, tensor-core expert kernel)");
        if ((e = device_error_word(&d.err_word)) != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(device error word)");
        d.ready = true;
    }
    *out = &d;
    return NVFP4_OK;
}

// Library-owned workspace for (device, stream); allocated and zeroed once.
static nvfp4_status stream_workspace(int dev, cudaStream_t stream, size_t bytes, void **out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    for (auto &w : g_workspaces) {
        if (w.device == dev && w.stream == stream) {
            if (w.bytes >= bytes) {
                *out = w.ptr;
                return NVFP4_OK;
            }
            // Grow: wait for work that may still use the old buffer, then replace it.
            cudaError_t e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize (workspace grow)");
            cudaFree(w.ptr);
            w.ptr = nullptr;
            if ((e = cudaMalloc(&w.ptr, bytes)) != cudaSuccess) return cuda_fail(e, "cudaMalloc (workspace)");
            if ((e = cudaMemsetAsync(w.ptr, 0, bytes, stream)) != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
            w.bytes = bytes;
            *out = w.ptr;
            return NVFP4_OK;
        }
    }
    WorkspaceEntry w{dev, stream, nullptr, bytes};
    cudaError_t e = cudaMalloc(&w.ptr, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc (workspace)");
    if ((e = cudaMemsetAsync(w.ptr, 0, bytes, stream)) != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    g_workspaces.push_back(w);
    *out = w.ptr;
    return NVFP4_OK;
}

// --------------------------------------------------------- TMA descriptors
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static nvfp4_status get_encode_fn(EncodeTiledFn *fn) {
    static EncodeTiledFn cached = nullptr;
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) cached = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!cached)
        return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(err));
    *fn = cached;
    return NVFP4_OK;
}

// 2D uint8 tensor [rows][cols] with row pitch `cols` bytes, box box_cols x box_rows.
static nvfp4_status encode_2d(CUtensorMap *map, const void *ptr, uint64_t cols, uint64_t rows, uint32_t box_cols,
                              uint32_t box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
    EncodeTiledFn fn;
    nvfp4_status st = get_encode_fn(&fn);
    if (st != NVFP4_OK) return st;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return NVFP4_OK;
}

// encode_2d through a small per-thread cache: a decode step calls the same
// few weight matrices over and over, and encoding a tensor map is host work
// on every call's path.  Keyed by everything the map depends on.
struct MapCacheEntry {
    const void *ptr;
    uint64_t cols, rows;
    uint32_t box_cols, box_rows;
    int swizzle;
    CUtensorMap map;
};
static nvfp4_status encode_2d_cached(CUtensorMap *map, const void *ptr, uint64_t cols, uint64_t rows,
                                     uint32_t box_cols, uint32_t box_rows,
                                     CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
    constexpr int kEntries = 32;
    static thread_local MapCacheEntry cache[kEntries];
    static thread_local int used = 0, next = 0;
    for (int i = 0; i < used; ++i) {
        const MapCacheEntry &c = cache[i];
        if (c.ptr == ptr && c.cols == cols && c.rows == rows && c.box_cols == box_cols && c.box_rows == box_rows &&
            c.swizzle == (int)swizzle) {
            *map = c.map;
            return NVFP4_OK;
        }
    }
    nvfp4_status st = encode_2d(map, ptr, cols, rows, box_cols, box_rows, swizzle);
    if (st != NVFP4_OK) return st;
    MapCacheEntry &c = cache[next];
    c = MapCacheEntry{ptr, cols, rows, box_cols, box_rows, (int)swizzle, *map};
    next = (next + 1) % kEntries;
    if (used < kEntries) ++used;
    return NVFP4_OK;
}

// The f16 X of one pass for the tcgen05 kernel with 32 staged tokens (the
// output of its conversion kernel), viewed as 3D {64 k, n tokens, K/64
// k-chunks} (token stride 2K bytes, chunk stride 128 bytes) so that one box
// {64, 32, 4} is one unit's X in the tensor core's 128-byte-swizzled K-major
// layout; tokens past n read as zeros.  (With 8 staged tokens the kernel
// copies X rows itself and needs no map.)
static nvfp4_status encode_x(CUtensorMap *map, const uint16_t *x, int n, int K, int box_tokens) {
    EncodeTiledFn fn;
    nvfp4_status st = get_encode_fn(&fn);
    if (st != NVFP4_OK) return st;
    const cuuint64_t dims[3] = {64, (cuuint64_t)n, (cuuint64_t)K / 64};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_tokens, 4};
    const cuuint32_t estr[3] = {1, 1, 1};
    // a 2-byte element type either way: the copy does not convert (T = 32 maps the f16 X)
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(x), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled (X) failed (CUresult %d)", (int)r);
    return NVFP4_OK;
}

// ------------------------------------------------------------------ policy
struct Plan {
    int variant = kAuto;
    int tiling = NVFP4_TILING_AUTO;
    std::vector<int> tiles;  // tokens per pass
    int ctas = 0;
    int stages = 0;
    int smem = 0;
    long long units = 0;
    int tc_tokens = 0;  // tcgen05 kernel: tokens staged per pass (8, 16 or 32)
    size_t partial_bytes = 0, x16_bytes = 0;
    TcPartition part{};  // tcgen05 kernel: k-groups and their CTAs
    size_t counter_bytes = 0, ws_bytes = 0;
    // block-scaled FP4 kernel: MMA columns of the widest pass, parts bound,
    // and the workspace regions after the partial tiles
    int f4_cols_max = 0, f4_max_seg = 0, f4_max_parts = 0, f4_inflight = 0;
    bool f4_x_resident = false;
    int f4_cluster = 0;  // CTAs per row block when the grid splits every row block evenly (summed in a cluster)
    size_t f4_xq_offset = 0, f4_xt_offset = 0, f4_et_offset = 0;
};

// Largest k-group (unit columns) whose X for 16 tokens fits next to eight
// weight stages; the partition uses it for every n, so results do not depend
// on n.
static int tc_group_limit(int smem_optin) {
    int kg = 32;
    while (kg > 1 && tc_smem_bytes(kMaxStages, 16, kg) > smem_optin) --kg;
    return kg;
}

// Split K into k-groups and the grid into per-group CTA ranges (each group
// gets CTAs in proportion to its units, at least one), and count the row
// blocks any CTA touches.
static nvfp4_status tc_partition(int N, int K, int ctas, int smem_optin, TcPartition *out, int *kg_max_out) {
    TcPartition t{};
    const int KC = K / kTcUnitKHost;
    t.row_blocks = (N + kUnitRows - 1) / kUnitRows;
    const int limit = tc_group_limit(smem_optin);
    t.groups = (KC + limit - 1) / limit;
    if (t.groups > kTcMaxGroups)
        return fail(NVFP4_ERR_UNSUPPORTED, "K = %d needs %d k-groups (at most %d)", K, t.groups, kTcMaxGroups);
    if (ctas < t.groups)
        return fail(NVFP4_ERR_INVALID_ARG, "num_ctas = %d: the tcgen05 kernel needs at least %d CTAs for K = %d", ctas,
                    t.groups, K);
    std::vector<long long> units(t.groups);
    std::vector<int> c(t.groups, 1);
    for (int g = 0; g < t.groups; ++g) {
        int ks, kg;
        tc_group_host(g, t.groups, KC, &ks, &kg);
        units[g] = (long long)t.row_blocks * kg;
    }
    for (int extra = ctas - t.groups; extra > 0; --extra) {
        int best = -1;  // the group with the most units per CTA that can still take a CTA
        for (int g = 0; g < t.groups; ++g) {
            if (c[g] >= units[g]) continue;
            if (best < 0 || units[g] * c[best] > units[best] * c[g]) best = g;
        }
        if (best < 0) break;
        ++c[best];
    }
    t.cstart[0] = 0;
    for (int g = 0; g < t.groups; ++g) t.cstart[g + 1] = t.cstart[g] + c[g];
    t.max_seg = 1;
    for (int g = 0; g < t.groups; ++g) {
        int ks, kg;
        tc_group_host(g, t.groups, KC, &ks, &kg);
        for (int cl = 0; cl < c[g]; ++cl) {
            const long long u0 = (long long)cl * units[g] / c[g], u1 = (long long)(cl + 1) * units[g] / c[g];
            const int segs = (int)((u1 - 1) / kg - u0 / kg + 1);
            if (segs > t.max_seg) t.max_seg = segs;
        }
    }
    // parts of the most-split row block (the reduction kernel holds them all in shared memory)
    if ((long long)t.row_blocks * KC * (ctas + 1) >= (1ll << 32))
        return fail(NVFP4_ERR_UNSUPPORTED, "N = %d, K = %d: too many units for the tcgen05 kernel", N, K);
    t.max_parts = 1;
    for (int rb = 0; rb < t.row_blocks; ++rb) {
        int parts = 0;
        for (int g = 0; g < t.groups; ++g) {
            int ks, kg;
            tc_group_host(g, t.groups, KC, &ks, &kg);
            const long long u = units[g];
            const long long ca = ((long long)(rb * kg + 1) * c[g] - 1) / u, cb = ((long long)(rb * kg + kg) * c[g] - 1) / u;
            parts += (int)(cb - ca + 1);
        }
        if (parts > t.max_parts) t.max_parts = parts;
    }
    if (t.max_parts > kTcMaxParts)
        return fail(NVFP4_ERR_UNSUPPORTED, "a row block would be split into %d parts (at most %d)", t.max_parts,
                    kTcMaxParts);
    *out = t;
    *kg_max_out = (KC + t.groups - 1) / t.groups;
    return NVFP4_OK;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Block-scaled FP4 kernel: stream-K over the row-block-major units of all of
// K (CTA c takes units [c U / C, (c + 1) U / C)); returns the most row-block
// segments of one CTA (its partial-tile slots) and the most parts of one row
// block.
// Default grid of the FP4 kernel.  Split row blocks cost a partial-tile round
// trip and a wait for the slowest part, so a grid that gives every CTA whole
// row blocks (RB CTAs, one row block each) or every row block p equal parts
// (RB p CTAs, KC % p == 0) is taken when it keeps at least 70 % of the SMs
// streaming -- the largest such; otherwise one CTA per SM with stream-K
// ranges.  Measured on GB300: attention qkv (112 row blocks) 13.0 -> 11.1 us
// at n = 1 with 112 CTAs, output projection (40 row blocks of 24 units)
// 12.3 -> 10.4 us at n = 8 with 120 CTAs (3 parts each).
static int f4_default_ctas(int N, int K, int sms) {
    const int RB = (N + kUnitRows - 1) / kUnitRows, KC = K / kTcUnitKHost;
    int best = 0;
    for (int p = 1; p <= 8; ++p) {
        const long long c = (long long)RB * p;
        if (c <= sms && KC % p == 0 && 10 * c >= 7LL * sms && c > best) best = (int)c;
    }
    return best ? best : sms;
}

static nvfp4_status f4_partition(int N, int K, int ctas, int *max_seg, int *max_parts) {
    const long long KC = K / kTcUnitKHost, RB = (N + kUnitRows - 1) / kUnitRows, U = RB * KC;
    if (RB * KC * (ctas + 1) >= (1ll << 40))
        return fail(NVFP4_ERR_UNSUPPORTED, "N = %d, K = %d: too many units for the FP4 kernel", N, K);
    int ms = 1, mp = 1;
    for (long long c = 0; c < ctas; ++c) {
        const long long u0 = c * U / ctas, u1 = (c + 1) * U / ctas;
        if (u1 > u0) {
            const int segs = (int)((u1 - 1) / KC - u0 / KC + 1);
            if (segs > ms) ms = segs;
        }
    }
    for (long long rb = 0; rb < RB; ++rb) {
        const long long ca = ((rb * KC + 1) * ctas - 1) / U, cb = ((rb * KC + KC) * ctas - 1) / U;
        if (cb - ca + 1 > mp) mp = (int)(cb - ca + 1);
    }
    *max_seg = ms;
    *max_parts = mp;
    return NVFP4_OK;
}

// Greedy 3/2/1 token tiling: tiles of 3, then one tile of 2 or 1.
static std::vector<int> greedy_321(int n) {
    std::vector<int> t;
    int left = n;
    while (left >= 3) {
        t.push_back(3);
        left -= 3;
    }
    if (left > 0) t.push_back(left);
    return t;
}

// AUTO's choice of kernel for a fast-path call: the FP4 kernel (passes of
// up to 16 tokens) when K allows it (default), or the tcgen05 kernel only.
enum AutoMode { kAutoDefault = 0, kAutoTcOnly = 1 };
static nvfp4_status make_plan_tokens(int n, int N, int K, bool fast_ok, const nvfp4_gemv_opts &o, int sms,
                                     int smem_optin, int tc_per_pass, AutoMode mode, Plan *plan);

// AUTO picks the FP4 kernel, in passes of up to 16 tokens (one read of W for
// n <= 16; the weights of a pass that another follows are kept in L2), for
// K <= 32768, and the tcgen05 f16 kernel above that.  The tcgen05 kernel's
// 32-token mode is not AUTO's choice for n > 16: on GB300 it showed rare
// run-to-run differences with long unit ranges per CTA whose cause is not
// found.  When the caller declares a scratch size (workspace_bytes) too
// small for the FP4 plan, AUTO takes the tcgen05 kernel, in 8-token passes if
// its 32-token pass does not fit either.
static nvfp4_status make_plan_uncached(int n, int N, int K, bool fast_ok, const nvfp4_gemv_opts &o, int sms,
                                       int smem_optin, Plan *plan);

// Plans through a small per-thread cache keyed by the call's shape, the
// options that shape the plan and the device's limits (planning walks the
// partition, which is host work on every call's path).
struct PlanCacheEntry {
    int n, N, K, sms, smem_optin, variant, tiling, num_ctas, stages, inflight;
    bool fast_ok;
    size_t workspace_bytes;
    Plan plan;
};
static nvfp4_status make_plan(int n, int N, int K, bool fast_ok, const nvfp4_gemv_opts &o, int sms, int smem_optin,
                              Plan *plan) {
    constexpr int kEntries = 16;
    static thread_local PlanCacheEntry cache[kEntries];
    static thread_local int used = 0, next = 0;
    for (int i = 0; i < used; ++i) {
        const PlanCacheEntry &c = cache[i];
        if (c.n == n && c.N == N && c.K == K && c.fast_ok == fast_ok && c.sms == sms && c.smem_optin == smem_optin &&
            c.variant == o.variant && c.tiling == o.tiling && c.num_ctas == o.num_ctas && c.stages == o.stages &&
            c.inflight == o.inflight && c.workspace_bytes == o.workspace_bytes) {
            *plan = c.plan;
            return NVFP4_OK;
        }
    }
    nvfp4_status st = make_plan_uncached(n, N, K, fast_ok, o, sms, smem_optin, plan);
    if (st != NVFP4_OK) return st;
    cache[next] = PlanCacheEntry{n, N, K, sms, smem_optin, o.variant, o.tiling, o.num_ctas, o.stages, o.inflight,
                                 fast_ok, o.workspace_bytes, *plan};
    next = (next + 1) % kEntries;
    if (used < kEntries) ++used;
    return NVFP4_OK;
}

static nvfp4_status make_plan_uncached(int n, int N, int K, bool fast_ok, const nvfp4_gemv_opts &o, int sms,
                                       int smem_optin, Plan *plan) {
    const bool small_ws = o.workspace_bytes != 0;
    auto too_big = [&](const Plan *pl) { return small_ws && o.workspace_bytes < pl->ws_bytes; };
    nvfp4_status st =
        make_plan_tokens(n, N, K, fast_ok, o, sms, smem_optin, kTcMaxTokensPerPass, kAutoDefault, plan);
    if (st == NVFP4_OK && o.variant == kAuto && too_big(plan) && plan->variant == kFp4)
        st = make_plan_tokens(n, N, K, fast_ok, o, sms, smem_optin, kTcMaxTokensPerPass, kAutoTcOnly, plan);
    if (st == NVFP4_OK && plan->variant == kTc && plan->tc_tokens == 32 && too_big(plan))
        st = make_plan_tokens(n, N, K, fast_ok, o, sms, smem_optin, 8, kAutoTcOnly, plan);
    return st;
}

static nvfp4_status make_plan_tokens(int n, int N, int K, bool fast_ok, const nvfp4_gemv_opts &o, int sms,
                                     int smem_optin, int tc_per_pass, AutoMode mode, Plan *plan) {
    Plan p;
    p.variant = o.variant;
    const bool tc_ok = fast_ok;
    if (p.variant == kAuto) {
        const bool fp4_ok = fast_ok && K <= kF4MaxK && mode != kAutoTcOnly;
        p.variant = fp4_ok ? kFp4 : tc_ok ? kTc : kGeneric;
    }
    if ((p.variant == kMma || p.variant == kSimt) && !fast_ok)
        return fail(NVFP4_ERR_INVALID_ARG,
                    "variant %d needs K %% 256 == 0 and 16-byte aligned w_packed, w_scale_e4m3 and x_bf16",
                    p.variant);
    if (p.variant == kTc && !tc_ok)
        return fail(NVFP4_ERR_INVALID_ARG,
                    "the tcgen05 variant needs K %% 256 == 0 and 16-byte aligned w_packed, w_scale_e4m3 and x_bf16");
    if (p.variant == kFp4 && !fast_ok)
        return fail(NVFP4_ERR_INVALID_ARG,
                    "the FP4 variant needs K %% 256 == 0 and 16-byte aligned w_packed, w_scale_e4m3 and x_bf16");
    if (p.variant == kFp4 && K > kF4MaxK)
        return fail(NVFP4_ERR_UNSUPPORTED, "the FP4 variant takes K <= %d", kF4MaxK);
    p.tiling = (o.tiling == NVFP4_TILING_AUTO) ? NVFP4_TILING_ONE_PASS : o.tiling;

    int per_pass = p.variant == kTc ? tc_per_pass : p.variant == kFp4 ? kF4MaxTokensPerPass : kMaxTokensPerPass;
    if (p.variant == kMma || p.variant == kSimt) {
        // largest token count whose X still leaves room for two ring stages
        const int room = smem_optin - stream_smem_bytes(2, 0, K);
        int fit = room / (2 * K);
        if (fit < 1) return fail(NVFP4_ERR_UNSUPPORTED, "K = %d too large for the streaming kernel", K);
        per_pass = fit < per_pass ? fit : per_pass;
    }  // tcgen05: 32 tokens per pass (X streamed per unit) for any K, or 8 (X held per k-group)
    if (p.tiling == NVFP4_TILING_GREEDY_321) {
        p.tiles = greedy_321(n);
    } else {
        for (int left = n; left > 0; left -= per_pass) p.tiles.push_back(left < per_pass ? left : per_pass);
    }
    if (p.variant == kFp4) {
        int max_tile = 0;
        for (int t : p.tiles) max_tile = t > max_tile ? t : max_tile;
        p.units = (long long)((N + kUnitRows - 1) / kUnitRows) * (K / kTcUnitKHost);
        int ctas = o.num_ctas ? o.num_ctas : f4_default_ctas(N, K, sms);
        if (ctas < 1 || ctas > sms) return fail(NVFP4_ERR_INVALID_ARG, "num_ctas must be 0 or 1..%d", sms);
        if ((long long)ctas > p.units) ctas = (int)p.units;
        p.ctas = ctas;
        nvfp4_status st = f4_partition(N, K, ctas, &p.f4_max_seg, &p.f4_max_parts);
        if (st != NVFP4_OK) return st;
        p.f4_cols_max = f4_cols(max_tile);
        {
            // RB p CTAs with KC % p == 0: every CTA holds 1 / p of one row block;
            // the p parts of a row block are consecutive CTAs, one cluster
            const int RBc = (N + kUnitRows - 1) / kUnitRows, KCc = K / kTcUnitKHost;
            const int parts = ctas % RBc == 0 ? ctas / RBc : 0;
            p.f4_cluster = (parts >= 2 && parts <= 8 && KCc % parts == 0) ? parts : 0;
        }
        // leave room on the SM for one X-prep CTA of the next call beside the GEMV
        const int limit = smem_optin - 4096;
        const int KC = K / kTcUnitKHost;
        // small X term blocks stay resident for the whole call (a few bulk
        // copies per CTA instead of one per unit)
        p.f4_x_resident = (long long)KC * f4_slot_bytes(p.f4_cols_max) <= kF4ResidentXMax &&
                          f4_max_stages(p.f4_cols_max, limit, true, KC, p.f4_cluster) >= 4;
        const int max_stages = f4_max_stages(p.f4_cols_max, limit, p.f4_x_resident, KC, p.f4_cluster);
        if (max_stages < 2) return fail(NVFP4_ERR_UNSUPPORTED, "the FP4 kernel does not fit shared memory");
        int stages = max_stages;
        if (o.stages != 0) {
            if (o.stages > max_stages)
                return fail(NVFP4_ERR_INVALID_ARG, "stages = %d does not fit (max %d)", o.stages, max_stages);
            stages = o.stages;
        }
        p.stages = stages;
        p.f4_inflight = o.inflight > 0 ? o.inflight : kF4DefaultInflight;
        p.smem = f4_smem_bytes(stages, p.f4_cols_max, p.f4_x_resident, KC, p.f4_cluster);
        const int RB = (N + kUnitRows - 1) / kUnitRows;
        p.counter_bytes = ws_counter_bytes(sms, RB);
        p.partial_bytes = (size_t)ctas * 2 * kUnitRows * 16 * sizeof(float);  // first and last row block
        p.f4_xq_offset = p.counter_bytes + ((p.partial_bytes + 255) & ~(size_t)255);
        const size_t xq_bytes = (size_t)KC * f4_slot_bytes(p.f4_cols_max);
        p.f4_xt_offset = p.f4_xq_offset + ((xq_bytes + 255) & ~(size_t)255);
        const size_t xt_bytes = (size_t)KC * f4_tab_bytes(p.f4_cols_max);
        p.f4_et_offset = p.f4_xt_offset + ((xt_bytes + 255) & ~(size_t)255);
        p.ws_bytes = p.f4_et_offset + 16 * kF4Terms * sizeof(float);
    } else if (p.variant != kGeneric) {
        int max_tile = 0;
        for (int t : p.tiles) max_tile = t > max_tile ? t : max_tile;
        // tcgen05 staged tokens: 8, else 32 (X pre-converted, streamed per unit).
        // The 16-token mode of the kernel (X converted in place per k-group)
        // returned run-to-run differing, wrong outputs in some row blocks for
        // long unit ranges per CTA on GB300 (cause not found); it is not used.
        const int T = max_tile > 8 ? 32 : 8;
        const int unit_k = p.variant == kTc ? kTcUnitKHost : kUnitK;
        p.units = (long long)((N + kUnitRows - 1) / kUnitRows) * (K / unit_k);
        int ctas = o.num_ctas ? o.num_ctas : sms;
        if (ctas < 1 || ctas > sms) return fail(NVFP4_ERR_INVALID_ARG, "num_ctas must be 0 or 1..%d", sms);
        if ((long long)ctas > p.units) ctas = (int)p.units;
        p.ctas = ctas;
        int kg_max = 0;
        if (p.variant == kTc) {
            nvfp4_status st = tc_partition(N, K, ctas, smem_optin, &p.part, &kg_max);
            if (st != NVFP4_OK) return st;
        }
        auto smem_for = [&](int st) {
            return p.variant == kTc ? tc_smem_bytes(st, T, kg_max) : stream_smem_bytes(st, max_tile, K);
        };
        // the tcgen05 kernel needs an even number of stages (every consumer warp
        // waits on every phase of a stage's barriers)
        const int stage_step = p.variant == kTc ? 2 : 1;
        int stages = kMaxStages;
        while (stages > 2 && smem_for(stages) > smem_optin) stages -= stage_step;
        if (smem_for(stages) > smem_optin) return fail(NVFP4_ERR_UNSUPPORTED, "K = %d does not fit shared memory", K);
        if (o.stages != 0) {
            if (o.stages > stages)
                return fail(NVFP4_ERR_INVALID_ARG, "stages = %d does not fit shared memory (max %d)", o.stages, stages);
            if (o.stages % stage_step != 0)
                return fail(NVFP4_ERR_INVALID_ARG, "stages = %d: the tcgen05 kernel needs an even number", o.stages);
            stages = o.stages;
        }
        p.stages = stages;
        p.smem = smem_for(stages);
        p.tc_tokens = p.variant == kTc ? T : 0;
        p.counter_bytes = ws_counter_bytes(sms, (N + kUnitRows - 1) / kUnitRows);
        p.partial_bytes = p.variant == kTc ? (size_t)ctas * p.part.max_seg * tc_partial_floats(T) * sizeof(float)
                                           : stream_partial_bytes(sms);
        // T = 32: the pass's X as f16 x 2^-8 follows the partial tiles (256-byte aligned)
        p.x16_bytes = (p.variant == kTc && T == 32) ? (size_t)32 * K * 2 : 0;
        p.ws_bytes = p.counter_bytes + ((p.partial_bytes + 255) & ~(size_t)255) + p.x16_bytes;
    }
    *plan = p;
    return NVFP4_OK;
}

static nvfp4_status validate(const void *wp, const void *ws, const void *gs, const void *x, const void *y, int n,
                             int N, int K) {
    if (n < 0) return fail(NVFP4_ERR_INVALID_ARG, "n = %d must be >= 0", n);
    if (N < 1) return fail(NVFP4_ERR_INVALID_ARG, "N = %d must be >= 1", N);
    if (K < 16 || K % 16 != 0) return fail(NVFP4_ERR_INVALID_ARG, "K = %d must be a positive multiple of 16", K);
    if ((long long)N * K / 2 > (1ll << 40)) return fail(NVFP4_ERR_INVALID_ARG, "N * K too large");
    if (n > 0 && (!wp || !ws || !gs || !x || !y)) return fail(NVFP4_ERR_INVALID_ARG, "null pointer argument");
    return NVFP4_OK;
}

static nvfp4_status validate_opts(const nvfp4_gemv_opts &o) {
    if (o.variant < kAuto || o.variant > kFp4) return fail(NVFP4_ERR_INVALID_ARG, "unknown variant %d", o.variant);
    if (o.tiling < NVFP4_TILING_AUTO || o.tiling > NVFP4_TILING_GREEDY_321)
        return fail(NVFP4_ERR_INVALID_ARG, "unknown tiling %d", o.tiling);
    if (o.num_ctas < 0) return fail(NVFP4_ERR_INVALID_ARG, "num_ctas = %d must be >= 0", o.num_ctas);
    if (o.stages != 0 && (o.stages < 2 || o.stages > (o.variant == kFp4 ? kF4MaxStages : kMaxStages)))
        return fail(NVFP4_ERR_INVALID_ARG, "stages must be 0 or 2..%d", o.variant == kFp4 ? kF4MaxStages : kMaxStages);
    if (o.workspace && (reinterpret_cast<uintptr_t>(o.workspace) & 255u) != 0)
        return fail(NVFP4_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    return NVFP4_OK;
}

static nvfp4_gemv_opts default_opts() {
    nvfp4_gemv_opts o;
    std::memset(&o, 0, sizeof o);
    return o;
}

// swiglu: rows 2f, 2f+1 of W are gate_f, up_f; y receives h[n][N/2] (tcgen05 path only).
static nvfp4_status run(const uint8_t *wp, const uint8_t *ws, const float *gs, const uint16_t *x, uint16_t *y, int n,
                        int N, int K, cudaStream_t stream, const nvfp4_gemv_opts *opts, bool swiglu = false) {
    nvfp4_status st = validate(wp, ws, gs, x, y, n, N, K);
    if (st != NVFP4_OK) return st;
    const nvfp4_gemv_opts o = opts ? *opts : default_opts();
    if ((st = validate_opts(o)) != NVFP4_OK || n == 0) return st;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceState *d = nullptr;
    if ((st = device_state(dev, &d)) != NVFP4_OK) return st;

    const bool fast_ok = (K % 256 == 0) && aligned16(wp) && aligned16(ws) && aligned16(x);
    Plan plan;
    if ((st = make_plan(n, N, K, fast_ok, o, d->sms, d->smem_optin, &plan)) != NVFP4_OK) return st;

    if (swiglu && plan.variant != kTc && plan.variant != kFp4)
        return fail(NVFP4_ERR_UNSUPPORTED,
                    "the fused SwiGLU runs on the tcgen05 path only (K %% 256 == 0, 16-byte aligned inputs, variant "
                    "AUTO or TC)");
    if (plan.variant == kGeneric) {
        int t0 = 0;
        for (int tn : plan.tiles) {
            for (int c0 = 0; c0 < tn; c0 += kMaxTokensPerPass) {
                const int cn = (tn - c0) < kMaxTokensPerPass ? (tn - c0) : kMaxTokensPerPass;
                GenericParams gp{wp, ws, gs, x + (size_t)(t0 + c0) * K, y + (size_t)(t0 + c0) * N, cn, N, K};
                if ((e = launch_generic(gp, stream)) != cudaSuccess) return cuda_fail(e, "generic kernel launch");
            }
            t0 += tn;
        }
        return NVFP4_OK;
    }

    // streaming kernels: workspace, descriptors, one launch per token tile
    const size_t ws_bytes = plan.ws_bytes;
    void *work = o.workspace;
    if (work) {
        if (o.workspace_bytes < ws_bytes)
            return fail(NVFP4_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", o.workspace_bytes, ws_bytes);
        if ((reinterpret_cast<uintptr_t>(work) & 255u) != 0)
            return fail(NVFP4_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    } else if ((st = stream_workspace(dev, stream, ws_bytes, &work)) != NVFP4_OK) {
        return st;
    }
    CUtensorMap tw, ts;
    if (plan.variant == kTc || plan.variant == kFp4) {
        if ((st = encode_2d_cached(&tw, wp, (uint64_t)K / 2, (uint64_t)N, 128, kUnitRows,
                                   CU_TENSOR_MAP_SWIZZLE_128B)) != NVFP4_OK)
            return st;
    } else if ((st = encode_2d_cached(&tw, wp, (uint64_t)K / 2, (uint64_t)N, kUnitK / 2, kUnitRows)) != NVFP4_OK) {
        return st;
    }
    if ((st = encode_2d_cached(&ts, ws, (uint64_t)K / 16, (uint64_t)N, 16, kUnitRows)) != NVFP4_OK) return st;

    if (plan.variant == kFp4) {
        F4Params fp;
        fp.gscale = gs;
        fp.counters = static_cast<unsigned *>(work);
        fp.partials = reinterpret_cast<float *>(static_cast<char *>(work) + plan.counter_bytes);
        fp.xq = static_cast<uint8_t *>(work) + plan.f4_xq_offset;
        fp.xtab = static_cast<uint8_t *>(work) + plan.f4_xt_offset;
        fp.xs = reinterpret_cast<float *>(static_cast<char *>(work) + plan.f4_et_offset);
        fp.err = d->err_word;
        fp.N = N;
        fp.K = K;
        fp.KC = K / kTcUnitKHost;
        fp.ctas = plan.ctas;
        fp.row_blocks = (N + kUnitRows - 1) / kUnitRows;
        fp.max_seg = plan.f4_max_seg;
        fp.stages = plan.stages;
        fp.swiglu = swiglu ? 1 : 0;
        fp.inflight = plan.f4_inflight;
        fp.x_resident = plan.f4_x_resident ? 1 : 0;
        fp.cluster = plan.f4_cluster;
        const size_t y_stride_f4 = swiglu ? (size_t)N / 2 : (size_t)N;
        int t0 = 0;
        for (int tn : plan.tiles) {
            fp.y = y + (size_t)t0 * y_stride_f4;
            fp.n = tn;
            fp.cols = f4_cols(tn);
            fp.w_keep = (t0 + tn < n) ? 1 : 0;  // the next pass re-reads W: from L2, not HBM
            if ((e = launch_fp4(tw, ts, x + (size_t)t0 * K, fp,
                                f4_smem_bytes(plan.stages, fp.cols, plan.f4_x_resident, fp.KC, plan.f4_cluster),
                                stream)) !=
                cudaSuccess)
                return cuda_fail(e, "FP4 kernel launch");
            t0 += tn;
        }
        return NVFP4_OK;
    }

    StreamParams sp;
    sp.gscale = gs;
    sp.counters = static_cast<unsigned *>(work);
    sp.partials = reinterpret_cast<float *>(static_cast<char *>(work) + plan.counter_bytes);
    uint16_t *const x16 = reinterpret_cast<uint16_t *>(static_cast<char *>(work) + plan.counter_bytes +
                                                       ((plan.partial_bytes + 255) & ~(size_t)255));
    sp.err = d->err_word;
    sp.units = plan.units;
    sp.ctas = plan.ctas;
    sp.N = N;
    sp.K = K;
    sp.KC = K / (plan.variant == kTc ? kTcUnitKHost : kUnitK);
    sp.stages = plan.stages;
    sp.swiglu = swiglu ? 1 : 0;
    const size_t y_stride = swiglu ? (size_t)N / 2 : (size_t)N;
    int t0 = 0;
    for (int tn : plan.tiles) {
        sp.x = x + (size_t)t0 * K;
        sp.y = y + (size_t)t0 * y_stride;
        sp.n = tn;
        sp.w_keep = (t0 + tn < n) ? 1 : 0;  // the next pass re-reads W: from L2, not HBM
        sp.y_vec2 = (N % 2 == 0) && ((reinterpret_cast<uintptr_t>(sp.y) & 3u) == 0);
        if (plan.variant == kTc) {
            CUtensorMap tx;
            memset(&tx, 0, sizeof tx);
            if (plan.tc_tokens == 32) {
                // the pass's X converted once to f16 x 2^-8; the GEMV streams it per unit
                if ((e = launch_tc_x16(sp.x, x16, tn, K, d->err_word, stream)) != cudaSuccess)
                    return cuda_fail(e, "X conversion kernel launch");
                if ((st = encode_x(&tx, x16, tn, K, 32)) != NVFP4_OK) return st;
            }
            e = launch_tc(tw, ts, tx, sp, plan.part, plan.tc_tokens, plan.smem, stream);
        } else {
            e = launch_stream(plan.variant, tw, ts, sp, plan.smem, stream);
        }
        if (e != cudaSuccess) return cuda_fail(e, "streaming kernel launch");
        t0 += tn;
    }
    return NVFP4_OK;
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status nvfp4_gemv_batched(const uint8_t *w_packed, const uint8_t *w_scale_e4m3,
                                           const float *w_global_scale_f32, const uint16_t *x_bf16, uint16_t *y_bf16,
                                           int n, int N, int K, cudaStream_t stream) {
    return run(w_packed, w_scale_e4m3, w_global_scale_f32, x_bf16, y_bf16, n, N, K, stream, nullptr);
}

extern "C" nvfp4_status nvfp4_gemv_batched_ex(const uint8_t *w_packed, const uint8_t *w_scale_e4m3,
                                              const float *w_global_scale_f32, const uint16_t *x_bf16,
                                              uint16_t *y_bf16, int n, int N, int K, cudaStream_t stream,
                                              const nvfp4_gemv_opts *opts) {
    return run(w_packed, w_scale_e4m3, w_global_scale_f32, x_bf16, y_bf16, n, N, K, stream, opts);
}

extern "C" nvfp4_status nvfp4_gemv_swiglu(const uint8_t *w_packed, const uint8_t *w_scale_e4m3,
                                          const float *w_global_scale_f32, const uint16_t *x_bf16, uint16_t *h_bf16,
                                          int n, int F, int K, cudaStream_t stream) {
    if (F < 1 || F > (1 << 29)) return fail(NVFP4_ERR_INVALID_ARG, "F = %d must be in [1, 2^29]", F);
    return run(w_packed, w_scale_e4m3, w_global_scale_f32, x_bf16, h_bf16, n, 2 * F, K, stream, nullptr, true);
}

extern "C" nvfp4_status nvfp4_ffn_swiglu(const uint8_t *w_gu_packed, const uint8_t *w_gu_scale_e4m3,
                                         const float *w_gu_global_scale_f32, const uint8_t *w_down_packed,
                                         const uint8_t *w_down_scale_e4m3, const float *w_down_global_scale_f32,
                                         const uint16_t *x_bf16, uint16_t *h_bf16, uint16_t *y_bf16, int n, int D,
                                         int F, cudaStream_t stream) {
    if (!w_down_packed || !w_down_scale_e4m3 || !w_down_global_scale_f32 || !y_bf16)
        return fail(NVFP4_ERR_INVALID_ARG, "null pointer argument");
    if (D < 16 || D % 16 != 0 || F < 16 || F % 16 != 0)
        return fail(NVFP4_ERR_INVALID_ARG, "D = %d and F = %d must be positive multiples of 16", D, F);
    nvfp4_status st = nvfp4_gemv_swiglu(w_gu_packed, w_gu_scale_e4m3, w_gu_global_scale_f32, x_bf16, h_bf16, n, F,
                                        D, stream);
    if (st != NVFP4_OK) return st;
    return run(w_down_packed, w_down_scale_e4m3, w_down_global_scale_f32, h_bf16, y_bf16, n, D, F, stream, nullptr);
}

// Host-only planning (no CUDA calls when the device state is unknown: SM count
// and shared memory default to the GB300 figures then).
static nvfp4_status plan_host(int n, int N, int K, const nvfp4_gemv_opts *opts, Plan *plan, int *sms_out) {
    nvfp4_status st = validate((void *)1, (void *)1, (void *)1, (void *)1, (void *)1, n, N, K);
    if (st != NVFP4_OK) return st;
    const nvfp4_gemv_opts o = opts ? *opts : default_opts();
    if ((st = validate_opts(o)) != NVFP4_OK) return st;
    int sms = 152, smem = 232448;
    int dev = 0, count = 0;
    if (cudaGetDeviceCount(&count) == cudaSuccess && count > 0 && cudaGetDevice(&dev) == cudaSuccess) {
        DeviceState *d = nullptr;
        if (device_state(dev, &d) == NVFP4_OK) {
            sms = d->sms;
            smem = d->smem_optin;
        }
    }
    cudaGetLastError();  // planning must not leave a sticky runtime error behind
    *sms_out = sms;
    return make_plan(n > 0 ? n : 1, N, K, K % 256 == 0, o, sms, smem, plan);
}

extern "C" nvfp4_status nvfp4_gemv_workspace_size(int n, int N, int K, const nvfp4_gemv_opts *opts, size_t *bytes) {
    if (!bytes) return fail(NVFP4_ERR_INVALID_ARG, "null bytes pointer");
    Plan plan;
    int sms = 0;
    nvfp4_status st = plan_host(n, N, K, opts, &plan, &sms);
    if (st != NVFP4_OK) return st;
    *bytes = plan.variant == kGeneric ? 0 : plan.ws_bytes;
    return NVFP4_OK;
}

namespace nvfp4 {
int workspace_layout(int n, int N, int K, const void *opts, size_t *counter_bytes, size_t *total_bytes) {
    Plan plan;
    int sms = 0;
    nvfp4_status st = plan_host(n, N, K, static_cast<const nvfp4_gemv_opts *>(opts), &plan, &sms);
    if (st != NVFP4_OK) return st;
    *counter_bytes = plan.variant == kGeneric ? 0 : plan.counter_bytes;
    *total_bytes = plan.variant == kGeneric ? 0 : plan.ws_bytes;
    return NVFP4_OK;
}
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_gemv_plan(int n, int N, int K, const nvfp4_gemv_opts *opts,
                                        nvfp4_gemv_plan_info *info) {
    if (!info) return fail(NVFP4_ERR_INVALID_ARG, "null info pointer");
    Plan plan;
    int sms = 0;
    nvfp4_status st = plan_host(n, N, K, opts, &plan, &sms);
    if (st != NVFP4_OK) return st;
    std::memset(info, 0, sizeof *info);
    info->variant = plan.variant;
    info->tiling = plan.tiling;
    info->passes = (int)plan.tiles.size();
    for (int i = 0; i < info->passes && i < 16; ++i) info->tile_tokens[i] = plan.tiles[i];
    info->num_ctas = plan.ctas;
    info->stages = plan.stages;
    info->smem_bytes = plan.smem;
    info->units = plan.units;
    return NVFP4_OK;
}

// GPU quantizer entry points: validation as nvfp4_quantize_ref, plus device
// pointer alignment (16 B for the weights, 8 B for the packed codes).
template <typename TW>
static nvfp4_status quantize_gpu(const TW *w, int N, int K, uint8_t *w_packed, uint8_t *w_scale,
                                 float *w_global_scale, cudaStream_t stream, bool bf16) {
    if (!w || !w_packed || !w_scale || !w_global_scale) return fail(NVFP4_ERR_INVALID_ARG, "null pointer argument");
    if (N < 1) return fail(NVFP4_ERR_INVALID_ARG, "N = %d must be >= 1", N);
    if (K < 16 || K % 16 != 0) return fail(NVFP4_ERR_INVALID_ARG, "K = %d must be a positive multiple of 16", K);
    if ((long long)N * K > (1ll << 40)) return fail(NVFP4_ERR_INVALID_ARG, "N * K too large");
    if (!aligned16(w) || (reinterpret_cast<uintptr_t>(w_packed) & 7u) != 0 ||
        (reinterpret_cast<uintptr_t>(w_global_scale) & 3u) != 0)
        return fail(NVFP4_ERR_MISALIGNED, "weights must be 16-byte aligned, packed codes 8-byte aligned");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceState *d = nullptr;
    nvfp4_status st = device_state(dev, &d);
    if (st != NVFP4_OK) return st;
    e = bf16 ? launch_quantize_bf16(reinterpret_cast<const uint16_t *>(w), N, K, w_packed, w_scale, w_global_scale,
                                    d->err_word, d->sms, stream)
             : launch_quantize_f32(reinterpret_cast<const float *>(w), N, K, w_packed, w_scale, w_global_scale,
                                   d->err_word, d->sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "quantizer launch");
    return NVFP4_OK;
}

extern "C" nvfp4_status nvfp4_quantize(const float *w_f32, int N, int K, uint8_t *w_packed, uint8_t *w_scale_e4m3,
                                       float *w_global_scale_f32, cudaStream_t stream) {
    return quantize_gpu(w_f32, N, K, w_packed, w_scale_e4m3, w_global_scale_f32, stream, false);
}

extern "C" nvfp4_status nvfp4_quantize_bf16(const uint16_t *w_bf16, int N, int K, uint8_t *w_packed,
                                            uint8_t *w_scale_e4m3, float *w_global_scale_f32, cudaStream_t stream) {
    return quantize_gpu(w_bf16, N, K, w_packed, w_scale_e4m3, w_global_scale_f32, stream, true);
}

extern "C" nvfp4_status nvfp4_moe_gemv_grouped(const uint8_t *w_packed, const uint8_t *w_scale_e4m3,
                                               const float *w_global_scale_f32, const uint16_t *x_bf16,
                                               const int32_t *expert_offsets, const int32_t *sorted_token,
                                               uint16_t *y_bf16, int E, int A, int n_tokens, int N, int K,
                                               int swiglu, cudaStream_t stream) {
    if (!w_packed || !w_scale_e4m3 || !w_global_scale_f32 || !x_bf16 || !expert_offsets || !sorted_token || !y_bf16)
        return fail(NVFP4_ERR_INVALID_ARG, "null pointer argument");
    if (E < 1 || E > kMoeMaxExperts || A < 0 || n_tokens < 1 || N < 1)
        return fail(NVFP4_ERR_INVALID_ARG, "E = %d (1..%d), A = %d, n_tokens = %d, N = %d out of range", E,
                    kMoeMaxExperts, A, n_tokens, N);
    if (swiglu != 0 && swiglu != 1) return fail(NVFP4_ERR_INVALID_ARG, "swiglu must be 0 or 1");
    if (N % 16 != 0) return fail(NVFP4_ERR_INVALID_ARG, "N = %d must be a multiple of 16", N);
    if (K < 32 || K % 32 != 0 || K > kMoeMaxK)
        return fail(NVFP4_ERR_INVALID_ARG, "K = %d must be a multiple of 32 in [32, %d]", K, kMoeMaxK);
    if ((long long)E * N > (1ll << 31) || (long long)A * N > (1ll << 40))
        return fail(NVFP4_ERR_INVALID_ARG, "E * N or A * N too large");
    if (!aligned16(w_packed) || !aligned16(w_scale_e4m3) || !aligned16(x_bf16) ||
        (reinterpret_cast<uintptr_t>(y_bf16) & 1u) != 0)
        return fail(NVFP4_ERR_MISALIGNED, "weights, scales and X must be 16-byte aligned");
    if (A == 0) return NVFP4_OK;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceState *d = nullptr;
    nvfp4_status st = device_state(dev, &d);
    if (st != NVFP4_OK) return st;
    MoeParams p;
    p.w = w_packed;
    p.s = w_scale_e4m3;
    p.gs = w_global_scale_f32;
    p.x = x_bf16;
    p.off = expert_offsets;
    p.tok = sorted_token;
    p.y = y_bf16;
    p.err = d->err_word;
    p.E = E;
    p.A = A;
    p.ntok = n_tokens;
    p.N = N;
    p.K = K;
    p.swiglu = swiglu;
    // K % 256 == 0: the streaming tensor-core kernel (W as 128-byte-swizzled TMA boxes)
    if (moe_mma_plan(N, K, d->smem_optin, &p.item_rows, &p.stages, &p.tok_pass)) {
        CUtensorMap tw;
        if ((st = encode_2d(&tw, w_packed, (uint64_t)K / 2, (uint64_t)E * N, 128, (uint32_t)p.item_rows,
                            CU_TENSOR_MAP_SWIZZLE_128B)) != NVFP4_OK)
            return st;
        p.ctas = d->sms;
        p.rows_per_cta = p.row_groups = 0;
        if ((e = launch_moe_mma(tw, p, stream)) != cudaSuccess) return cuda_fail(e, "grouped expert kernel launch");
        return NVFP4_OK;
    }
    const int out_rows = swiglu ? N / 2 : N;
    p.item_rows = p.stages = p.tok_pass = p.ctas = 0;
    p.rows_per_cta = moe_rows_per_cta(K, swiglu != 0, d->smem_optin);
    if (p.rows_per_cta == 0)
        return fail(NVFP4_ERR_UNSUPPORTED, "K = %d: the staged tokens and 16 weight rows do not fit shared memory", K);
    p.row_groups = (out_rows + p.rows_per_cta - 1) / p.rows_per_cta;
    if ((long long)E * p.row_groups > 0x7FFFFFFF) return fail(NVFP4_ERR_INVALID_ARG, "too many experts x rows");
    if ((e = launch_moe(p, stream)) != cudaSuccess) return cuda_fail(e, "grouped expert kernel launch");
    return NVFP4_OK;
}

extern "C" nvfp4_status nvfp4_device_error(cudaStream_t stream, int *code) {
    if (!code) return fail(NVFP4_ERR_INVALID_ARG, "null code pointer");
    *code = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceState *d = nullptr;
    nvfp4_status st = device_state(dev, &d);
    if (st != NVFP4_OK) return st;
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned word = 0;
    if ((e = cudaMemcpy(&word, d->err_word, sizeof word, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy (device error word)");
    *code = (int)word;
    if (word == 0) return NVFP4_OK;
    const unsigned zero = 0;
    cudaMemcpy(d->err_word, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if ((word & 7u) == 0 && (word & 128u) != 0)  // a debug-bounds check failed
        return fail(NVFP4_ERR_DEVICE_BOUNDS, "a device index check of the debug-bounds build failed and its access "
                    "was skipped (error word 0x%x)", word);
    if ((word & 7u) == 0 && (word & 64u) != 0)
        return fail(NVFP4_ERR_UNSUPPORTED, "the GEMV found its dynamic shared memory off a 1024-byte boundary "
                    "and computed nothing (error word 0x%x)", word);
    if ((word & 7u) == 0)
        return fail(NVFP4_ERR_DEVICE_INPUT, "a kernel met an input it cannot use (error word 0x%x)", word);
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        for (auto &w : g_workspaces)
            if (w.device == dev) cudaMemset(w.ptr, 0, w.bytes);
    }
    return fail(NVFP4_ERR_DEVICE_TIMEOUT, "a kernel gave up waiting on a barrier (error word 0x%x)", word);
}

extern "C" nvfp4_status nvfp4_selftest_wait_timeout(cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceState *d = nullptr;
    nvfp4_status st = device_state(dev, &d);
    if (st != NVFP4_OK) return st;
    if ((e = launch_selftest_wait_timeout(d->err_word, stream)) != cudaSuccess)
        return cuda_fail(e, "self-test kernel launch");
    return NVFP4_OK;
}

extern "C" const char *nvfp4_last_error(void) { return t_last_error.c_str(); }

extern "C" int nvfp4_version(void) { return 100; }
