// internal.h -- declarations shared by the library's translation units.
// Not installed, not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace nvfp4 {

// Work decomposition of the streaming kernels: a unit is 128 output rows by
// 128 k (64 bytes of every packed row plus 8 scale bytes per row).
constexpr int kUnitRows = 128;
constexpr int kUnitK = 128;
constexpr int kConsumerWarps = 4;                    // each owns 32 of the 128 rows
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one TMA producer warp
constexpr int kWTileBytes = kUnitRows * (kUnitK / 2);   // 8192
constexpr int kSTileBytes = kUnitRows * 16;             // 2048 (16 scale bytes = 256 k)
constexpr int kStageBytes = kWTileBytes + kSTileBytes;  // 10240
constexpr int kMaxStages = 8;
constexpr int kMaxTokensPerPass = 16;
constexpr int kSlotFloats = 32 * 16;  // one warp's partial tile: 32 lanes x 16 fp32
constexpr int kCountersPerCta = 8;    // split-tile counters per CTA (one per fixup warp)

enum Variant : int { kAuto = 0, kMma = 1, kSimt = 2, kGeneric = 3, kTc = 4 };

struct StreamParams {
    const uint16_t *x;   // [n][K] bf16, 16-byte aligned
    uint16_t *y;         // [n][N] bf16
    const float *gscale; // device scalar
    const uint16_t *xf16;  // tcgen05 kernel: X converted to f16, [K/256][T][256] core-matrix slices
    float *partials;     // [C][2][kConsumerWarps][kSlotFloats]
    unsigned *counters;  // [C][kConsumerWarps]
    unsigned *err;       // device error word
    long long units;     // ceil(N/128) * (K/128)
    int ctas;            // grid size (== number of unit ranges)
    int n, N, K, KC;     // KC = K / 128
    int stages;
    int y_vec2;          // bf16x2 stores allowed (N even and y 4-byte aligned)
};

struct GenericParams {
    const uint8_t *w;
    const uint8_t *s;
    const float *gscale;
    const uint16_t *x;
    uint16_t *y;
    int n, N, K;
};

// Shared-memory bytes of one streaming-kernel CTA.
inline int stream_smem_bytes(int stages, int n, int K) {
    return 1024 /* alignment slack */ + stages * kStageBytes + n * K * 2 + stages * 16 + 64;
}

// Workspace layout for a device with `max_ctas` SMs (independent of the grid
// size of any one call, so counters always sit at the same place):
//   [0, counter_bytes)          unsigned counters[max_ctas][kCountersPerCta]
//   [counter_bytes, ...)        float partials[max_ctas][2][kConsumerWarps * kSlotFloats]
inline size_t stream_counter_bytes(int max_ctas) {
    return ((size_t)max_ctas * kCountersPerCta * sizeof(unsigned) + 255) & ~(size_t)255;
}
inline size_t stream_workspace_bytes(int max_ctas) {
    return stream_counter_bytes(max_ctas) + (size_t)max_ctas * 2 * kConsumerWarps * kSlotFloats * sizeof(float);
}
// The tcgen05 path also keeps X converted to f16 (16 tokens x K) after that.
inline size_t tc_xbuf_bytes(int K) { return ((size_t)K * 16 * 2 + 255) & ~(size_t)255; }

cudaError_t launch_stream(int variant, const CUtensorMap &tw, const CUtensorMap &ts, const StreamParams &p,
                          int smem, cudaStream_t stream);
cudaError_t launch_generic(const GenericParams &p, cudaStream_t stream);
cudaError_t stream_set_smem_limits(int smem_optin);
cudaError_t device_error_word(unsigned **ptr);  // device address of the error word

// tcgen05 kernel (gemv_tc.cu): units of 128 rows x 256 k; T = 8 or 16 staged tokens.
constexpr int kTcUnitKHost = 256;
int tc_smem_bytes(int stages, int T, int K);
cudaError_t tc_set_smem_limit(int smem_optin);
// Converts X (n rows of bf16) into p.xf16 and then launches the GEMV with
// programmatic dependent launch, so the GEMV's weight stream starts while X is
// being converted.
cudaError_t launch_tc(const CUtensorMap &tw, const CUtensorMap &ts, const StreamParams &p, int T, int smem,
                      cudaStream_t stream);

}  // namespace nvfp4
