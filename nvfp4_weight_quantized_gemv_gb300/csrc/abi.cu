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

// ------------------------------------------------------------------ policy
struct Plan {
    int variant = kAuto;
    int tiling = NVFP4_TILING_AUTO;
    std::vector<int> tiles;  // tokens per pass
    int ctas = 0;
    int stages = 0;
    int smem = 0;
    long long units = 0;
    int tc_tokens = 0;  // tcgen05 kernel: tokens staged per pass (8 or 16)
};

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

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

static nvfp4_status make_plan(int n, int N, int K, bool fast_ok, const nvfp4_gemv_opts &o, int sms, int smem_optin,
                              Plan *plan) {
    Plan p;
    p.variant = o.variant;
    const bool tc_ok = fast_ok;
    if (p.variant == kAuto) p.variant = tc_ok ? kTc : (fast_ok ? kMma : kGeneric);
    if ((p.variant == kMma || p.variant == kSimt) && !fast_ok)
        return fail(NVFP4_ERR_INVALID_ARG,
                    "variant %d needs K %% 256 == 0 and 16-byte aligned w_packed, w_scale_e4m3 and x_bf16",
                    p.variant);
    if (p.variant == kTc && !tc_ok)
        return fail(NVFP4_ERR_INVALID_ARG,
                    "the tcgen05 variant needs K %% 256 == 0 and 16-byte aligned w_packed, w_scale_e4m3 and x_bf16");
    p.tiling = (o.tiling == NVFP4_TILING_AUTO) ? NVFP4_TILING_ONE_PASS : o.tiling;

    int per_pass = kMaxTokensPerPass;
    if (p.variant == kMma || p.variant == kSimt) {
        // largest token count whose X still leaves room for two ring stages
        const int room = smem_optin - stream_smem_bytes(2, 0, K);
        int fit = room / (2 * K);
        if (fit < 1) return fail(NVFP4_ERR_UNSUPPORTED, "K = %d too large for the streaming kernel", K);
        per_pass = fit < per_pass ? fit : per_pass;
    } else if (p.variant == kTc) {
        if (tc_smem_bytes(2, 16, K) <= smem_optin) per_pass = 16;
        else if (tc_smem_bytes(2, 8, K) <= smem_optin) per_pass = 8;
        else return fail(NVFP4_ERR_UNSUPPORTED, "K = %d too large for the tcgen05 kernel", K);
    }
    if (p.tiling == NVFP4_TILING_GREEDY_321) {
        p.tiles = greedy_321(n);
    } else {
        for (int left = n; left > 0; left -= per_pass) p.tiles.push_back(left < per_pass ? left : per_pass);
    }
    if (p.variant != kGeneric) {
        int max_tile = 0;
        for (int t : p.tiles) max_tile = t > max_tile ? t : max_tile;
        const int T = max_tile > 8 ? 16 : 8;
        auto smem_for = [&](int st) {
            return p.variant == kTc ? tc_smem_bytes(st, T, K) : stream_smem_bytes(st, max_tile, K);
        };
        int stages = kMaxStages;
        while (stages > 2 && smem_for(stages) > smem_optin) --stages;
        if (o.stages != 0) {
            if (o.stages > stages)
                return fail(NVFP4_ERR_INVALID_ARG, "stages = %d does not fit shared memory (max %d)", o.stages, stages);
            stages = o.stages;
        }
        p.stages = stages;
        p.smem = smem_for(stages);
        p.tc_tokens = p.variant == kTc ? T : 0;
        const int unit_k = p.variant == kTc ? kTcUnitKHost : kUnitK;
        p.units = (long long)((N + kUnitRows - 1) / kUnitRows) * (K / unit_k);
        int ctas = o.num_ctas ? o.num_ctas : sms;
        if (ctas < 1 || ctas > sms) return fail(NVFP4_ERR_INVALID_ARG, "num_ctas must be 0 or 1..%d", sms);
        if ((long long)ctas > p.units) ctas = (int)p.units;
        p.ctas = ctas;
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
    if (o.variant < kAuto || o.variant > kTc) return fail(NVFP4_ERR_INVALID_ARG, "unknown variant %d", o.variant);
    if (o.tiling < NVFP4_TILING_AUTO || o.tiling > NVFP4_TILING_GREEDY_321)
        return fail(NVFP4_ERR_INVALID_ARG, "unknown tiling %d", o.tiling);
    if (o.num_ctas < 0) return fail(NVFP4_ERR_INVALID_ARG, "num_ctas = %d must be >= 0", o.num_ctas);
    if (o.stages != 0 && (o.stages < 2 || o.stages > kMaxStages))
        return fail(NVFP4_ERR_INVALID_ARG, "stages must be 0 or 2..%d", kMaxStages);
    if (o.workspace && (reinterpret_cast<uintptr_t>(o.workspace) & 255u) != 0)
        return fail(NVFP4_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    return NVFP4_OK;
}

static nvfp4_gemv_opts default_opts() {
    nvfp4_gemv_opts o;
    std::memset(&o, 0, sizeof o);
    return o;
}

static nvfp4_status run(const uint8_t *wp, const uint8_t *ws, const float *gs, const uint16_t *x, uint16_t *y, int n,
                        int N, int K, cudaStream_t stream, const nvfp4_gemv_opts *opts) {
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
    const size_t fixed_bytes = stream_workspace_bytes(d->sms);
    const size_t ws_bytes = fixed_bytes + (plan.variant == kTc ? tc_xbuf_bytes(K) : 0);
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
    if (plan.variant == kTc) {
        if ((st = encode_2d(&tw, wp, (uint64_t)K / 2, (uint64_t)N, 128, kUnitRows, CU_TENSOR_MAP_SWIZZLE_128B)) !=
            NVFP4_OK)
            return st;
    } else if ((st = encode_2d(&tw, wp, (uint64_t)K / 2, (uint64_t)N, kUnitK / 2, kUnitRows)) != NVFP4_OK) {
        return st;
    }
    if ((st = encode_2d(&ts, ws, (uint64_t)K / 16, (uint64_t)N, 16, kUnitRows)) != NVFP4_OK) return st;

    StreamParams sp;
    sp.gscale = gs;
    sp.counters = static_cast<unsigned *>(work);
    sp.partials = reinterpret_cast<float *>(static_cast<char *>(work) + stream_counter_bytes(d->sms));
    sp.xf16 = reinterpret_cast<const uint16_t *>(static_cast<char *>(work) + fixed_bytes);
    sp.err = d->err_word;
    sp.units = plan.units;
    sp.ctas = plan.ctas;
    sp.N = N;
    sp.K = K;
    sp.KC = K / (plan.variant == kTc ? kTcUnitKHost : kUnitK);
    sp.stages = plan.stages;
    int t0 = 0;
    for (int tn : plan.tiles) {
        sp.x = x + (size_t)t0 * K;
        sp.y = y + (size_t)t0 * N;
        sp.n = tn;
        sp.y_vec2 = (N % 2 == 0) && ((reinterpret_cast<uintptr_t>(sp.y) & 3u) == 0);
        e = plan.variant == kTc ? launch_tc(tw, ts, sp, plan.tc_tokens, plan.smem, stream)
                                : launch_stream(plan.variant, tw, ts, sp, plan.smem, stream);
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
    *bytes = plan.variant == kGeneric ? 0
                                      : stream_workspace_bytes(sms) + (plan.variant == kTc ? tc_xbuf_bytes(K) : 0);
    return NVFP4_OK;
}

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
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        for (auto &w : g_workspaces)
            if (w.device == dev) cudaMemset(w.ptr, 0, w.bytes);
    }
    return fail(NVFP4_ERR_DEVICE_TIMEOUT, "a kernel gave up waiting on a barrier (error word 0x%x)", word);
}

extern "C" const char *nvfp4_last_error(void) { return t_last_error.c_str(); }

extern "C" int nvfp4_version(void) { return 100; }
