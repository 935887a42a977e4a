// gemv_noalloc.cu -- nvfp4_gemv_batched_noalloc: the batched GEMV without any
// device allocation, for callers that cannot call cudaMalloc.
//
// Who needs it: engines that reserve (nearly) all device memory up front in
// their own pool, so a library cudaMalloc would fail or fragment that pool;
// code that must not allocate once serving has started, because cudaMalloc
// can synchronize the whole device; and plugins that only ever receive
// pointers from a host program that owns all device memory.  The default
// entry point allocates a small workspace on the first call per stream; this
// one never does.
//
// How: the kernels' scratch (split-tile counters and fp32 partial tiles)
// lives in the file-scope device array below (8 MiB, held by every GPU that
// loads the library until the process exits); a call whose plan needs more
// is refused.  Its device address comes from
// cudaGetSymbolAddress, taken once per device with that device current, on
// the first call on that device.  Each call then clears the counters with
// cudaMemsetAsync on the caller's stream and runs the ordinary streaming path
// with this array as the caller-provided workspace.
//
// All calls on a device share the one array: calls that can overlap on the
// GPU (different streams without ordering between them) race on it and may
// return wrong results.  Serialize them, or use nvfp4_gemv_batched_ex with a
// workspace per stream.
#include "../../include/nvfp4_gemv.h"
#include "internal.h"

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

namespace nvfp4 {
void set_last_error(const char *msg);

namespace {

// counters + fp32 partial tiles: enough for 160 SMs with up to six row-block
// segments per CTA (6 x 8 KiB partial tiles each) and 16384 row blocks.
constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

nvfp4_status noalloc_fail(nvfp4_status st, const std::string &msg) {
    set_last_error(msg.c_str());
    return st;
}

}  // namespace
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_gemv_batched_noalloc(const uint8_t *w_packed, const uint8_t *w_scale_e4m3,
                                                   const float *w_global_scale_f32, const uint16_t *x_bf16,
                                                   uint16_t *y_bf16, int n, int N, int K, cudaStream_t stream) {
    using namespace nvfp4;
    // Bad arguments and n == 0 are answered by the ordinary validation, which
    // returns before anything is allocated or enqueued.
    const bool args_ok = n > 0 && N >= 1 && K >= 16 && K % 16 == 0 && w_packed && w_scale_e4m3 &&
                         w_global_scale_f32 && x_bf16 && y_bf16;
    if (!args_ok)
        return nvfp4_gemv_batched_ex(w_packed, w_scale_e4m3, w_global_scale_f32, x_bf16, y_bf16, n, N, K, stream,
                                     nullptr);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return noalloc_fail(NVFP4_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return noalloc_fail(NVFP4_ERR_UNSUPPORTED, "nvfp4_gemv_batched_noalloc: device ordinal too large");
    size_t counter_bytes = 0, needed = 0;
    nvfp4_gemv_opts cap;  // plan within the static scratch (AUTO falls back to a smaller plan if it is too small)
    std::memset(&cap, 0, sizeof cap);
    cap.workspace_bytes = kNoAllocScratchBytes;
    // Inputs off 16-byte alignment (or K % 256 != 0) take the generic kernel,
    // which needs no scratch: size the call only when the fast path runs.
    const auto a16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    const bool fast = K % 256 == 0 && a16(w_packed) && a16(w_scale_e4m3) && a16(x_bf16);
    if (fast) {
        const int st = workspace_layout(n, N, K, &cap, &counter_bytes, &needed);
        if (st != NVFP4_OK) return (nvfp4_status)st;
    }
    if (needed > kNoAllocScratchBytes) {
        char buf[256];
        std::snprintf(buf, sizeof buf,
                      "nvfp4_gemv_batched_noalloc: this call needs %zu bytes of scratch; the static scratch holds %zu",
                      needed, kNoAllocScratchBytes);
        return noalloc_fail(NVFP4_ERR_WORKSPACE, buf);
    }
    void *ptr = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        if (!g_noalloc_ptr[dev]) {
            // Set-up, once per device, with that device current: the symbol's
            // host-side name is not a device address, so ask the runtime for it.
            void *p = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess)
                return noalloc_fail(NVFP4_ERR_CUDA, std::string("cudaGetSymbolAddress(no-alloc scratch): ") +
                                                        cudaGetErrorString(e));
            g_noalloc_ptr[dev] = p;
        }
        ptr = g_noalloc_ptr[dev];
    }
    // The split-tile counters must start at zero; the array keeps whatever the
    // last call left, so clear them on this stream before the kernels run.
    if (counter_bytes && (e = cudaMemsetAsync(ptr, 0, counter_bytes, stream)) != cudaSuccess)
        return noalloc_fail(NVFP4_ERR_CUDA, std::string("cudaMemsetAsync(no-alloc counters): ") +
                                                cudaGetErrorString(e));
    nvfp4_gemv_opts o;
    std::memset(&o, 0, sizeof o);
    o.workspace = ptr;
    o.workspace_bytes = kNoAllocScratchBytes;
    return nvfp4_gemv_batched_ex(w_packed, w_scale_e4m3, w_global_scale_f32, x_bf16, y_bf16, n, N, K, stream, &o);
}
