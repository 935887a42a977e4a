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
constexpr int kTcMaxTokensPerPass = 32;  // tcgen05 kernel with the X ring
constexpr int kSlotFloats = 32 * 16;  // one warp's partial tile: 32 lanes x 16 fp32
constexpr int kCountersPerCta = 8;    // split-tile counters per CTA (one per fixup warp)

enum Variant : int { kAuto = 0, kMma = 1, kSimt = 2, kGeneric = 3, kTc = 4, kFp4 = 5 };

struct StreamParams {
    const uint16_t *x;   // [n][K] bf16, 16-byte aligned
    uint16_t *y;         // [n][N] bf16
    const float *gscale; // device scalar
    float *partials;     // [C][2][kConsumerWarps][kSlotFloats]
    unsigned *counters;  // [C][kConsumerWarps]
    unsigned *err;       // device error word
    long long units;     // ceil(N/128) * (K/128)
    int ctas;            // grid size (== number of unit ranges)
    int n, N, K, KC;     // KC = K / 128
    int stages;
    int y_vec2;          // bf16x2 stores allowed (N even and y 4-byte aligned)
    int swiglu;          // tcgen05 only: rows 2f, 2f+1 are gate_f, up_f; y is h[n][N/2] = silu(gate) * up
    int w_keep;          // tcgen05 only: another pass over the same weights follows (keep them in L2)
};

// Block-scaled FP4 tensor-core path (gemv_fp4.cu).  Per pass of up to 16
// tokens: fp4_xprep_kernel writes each token's activations as kF4Terms NVFP4
// terms -- E2M1 codes, one power-of-two UE4M3 scale per 16-element block
// (shared by the token's terms) and one fp32 scale per (token, term), MMA
// columns 8t + j -- into the workspace, then the GEMV streams the stored W
// and S tiles straight into tcgen05.mma kind::mxf4nvf4.  Workspace per unit
// column of 256 k: the codes [cols][128 B] (128-byte swizzled rows) and the
// block scales [cols / 8 tokens][16 B]; then the term scales [16][kF4Terms]
// floats.
constexpr int kF4Terms = 8;
constexpr int kF4MaxTokensPerPass = 16;
constexpr int kF4MaxCols = 128;              // 16 tokens x 8 terms
constexpr int kF4MaxStages = 16;
constexpr int kF4XOffHost = 16384 + 2048;    // X codes inside a ring stage, after the W and S tiles
constexpr int kF4MaxK = 32768;               // the X-prep kernel reads a whole row in one round of loads
constexpr int kF4DefaultInflight = 4;
constexpr int kF4MiscBytes = 32 + 16 * kF4Terms * 4 + 64;  // flags and counters, the term scales, slack
inline int f4_cols(int n) { return 16 * ((n * kF4Terms + 15) / 16); }
#ifdef __CUDACC__
#define NVFP4_HD __host__ __device__
#else
#define NVFP4_HD
#endif
NVFP4_HD inline int f4_slot_bytes(int cols) { return 128 * cols; }  // one unit column's X codes
NVFP4_HD inline int f4_tab_bytes(int cols) { return 2 * cols; }     // its block scales: cols / 8 tokens x 16
constexpr int kF4BlockHeadroom = 256;        // largest activation block scale, 2^8 (UE4M3 spans 2^-9 .. 2^8)
constexpr int kF4XGroup = 4;                 // unit columns per bulk copy of resident X codes
constexpr int kF4ResidentXMax = 112 * 1024;  // largest X code block kept resident in shared memory
inline int f4_dstride(int cols) { return cols <= 32 ? 32 : cols <= 64 ? 64 : 128; }
inline int f4_issuers(int cols) { return cols <= 64 ? 2 : 1; }
struct F4Params {
    uint16_t *y;          // [n][N] bf16 (swiglu: [n][N/2])
    const float *gscale;  // device scalar g
    uint8_t *xq;          // X codes: [K/256][f4_slot_bytes(cols)]
    uint8_t *xtab;        // X block scales: [K/256][f4_tab_bytes(cols)], UE4M3 byte per (token, 16-k block)
    float *xs;            // [16][kF4Terms] the tokens' term scales
    float *partials;      // [ctas][2][128 rows][16] fp32 parts of split row blocks (first, last)
    unsigned *counters;   // [row_blocks] parts completed (zero between calls)
    unsigned *err;        // device error word
    int n, N, K, KC;      // KC = K / 256
    int ctas, row_blocks, max_seg, stages, cols, swiglu, w_keep;
    int inflight;         // weight stages requested and not yet landed, at most
    int x_resident;       // 1: all unit columns' X codes stay in shared memory; 0: streamed with each stage
    int cluster;          // p >= 2: every row block is split over p consecutive CTAs, launched as one
                          // cluster that sums the parts through distributed shared memory; 0: no clusters
};
// Cluster sums of split row blocks (p CTAs per row block): the CTA of rank k
// sums the rows of epilogue warps q with q % p == k; its peers push their
// parts of those rows into its receive area, [p - 1 senders][f4_red_rows(p)
// rows][16 fp32], after the misc area (16-byte aligned).
inline int f4_red_rows(int p) { return p >= 2 ? 32 * ((4 + p - 1) / p) : 0; }
inline int f4_red_bytes(int p) { return p >= 2 ? (p - 1) * f4_red_rows(p) * 64 + 16 : 0; }
int f4_smem_bytes(int stages, int cols, bool x_resident, int KC, int cluster = 0);
int f4_max_stages(int cols, int smem_limit, bool x_resident, int KC, int cluster = 0);  // 0: does not fit
cudaError_t f4_set_smem_limit(int smem_optin);
// X prep then GEMV, both with programmatic dependent launch.
cudaError_t launch_fp4(const CUtensorMap &tw, const CUtensorMap &ts, const uint16_t *x, const F4Params &p, int smem,
                       cudaStream_t stream);

// Grouped read-once GEMV over routed experts (moe_gemv.cu).
struct MoeParams {
    const uint8_t *w;   // [E][N][K/2]
    const uint8_t *s;   // [E][N][K/16]
    const float *gs;    // [E] global scales
    const uint16_t *x;  // [ntok][K] bf16
    const int *off;     // [E + 1] assignment offsets per expert
    const int *tok;     // [A] token of each assignment, grouped by expert
    uint16_t *y;        // [A][N] (or [A][N/2] with swiglu)
    unsigned *err;      // device error word
    int E, A, ntok, N, K, swiglu;
    int rows_per_cta;   // SIMT kernel: output rows (gate/up pairs with swiglu) per CTA
    int row_groups;     // SIMT kernel: CTAs per expert
    int item_rows;      // tensor-core kernel: W rows per streamed item (128, 64, 32 or 16)
    int stages;         // tensor-core kernel: items in flight per CTA (ring slots)
    int tok_pass;       // tensor-core kernel: tokens staged per pass over an item (<= 16)
    int ctas;           // tensor-core kernel: persistent grid (one CTA per SM)
};
constexpr int kMoeMaxK = 7168;
constexpr int kMoeMaxExperts = 1024;
constexpr int kMoeMaxStages = 8;
constexpr int kMoeMmaStaticSmem = 5 * 1024;  // the tensor-core kernel's static shared memory, rounded up
// Tensor-core kernel (moe_mma.cu, K % 256 == 0): plan, shared memory, launch.
bool moe_mma_plan(int N, int K, int smem_optin, int *item_rows, int *stages, int *tok_pass);
int moe_mma_smem_bytes(const MoeParams &p);
cudaError_t moe_mma_set_smem_limit(int smem_optin);
cudaError_t launch_moe_mma(const CUtensorMap &tw, const MoeParams &p, cudaStream_t stream);
int moe_smem_bytes(int K, int rows_per_cta, bool swiglu);
int moe_rows_per_cta(int K, bool swiglu, int smem_optin);  // 0: K too large for shared memory
cudaError_t moe_set_smem_limit(int smem_optin);
cudaError_t launch_moe(const MoeParams &p, cudaStream_t stream);

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

// Workspace layout.  One zeroed counter region at offset 0 serves every
// variant (each call leaves the counters it used at zero again):
//   [0, counter_bytes)    unsigned counters: [sms][kCountersPerCta] for the
//                         mma.sync / SIMT kernels, [row blocks][kConsumerWarps]
//                         for the tcgen05 kernel
//   [counter_bytes, ...)  float partial tiles of kConsumerWarps * kSlotFloats:
//                         [sms][2] (mma.sync / SIMT) or [grid][max_seg] (tcgen05)
inline size_t ws_counter_bytes(int sms, int row_blocks) {
    const size_t a = (size_t)sms * kCountersPerCta, b = (size_t)row_blocks * kConsumerWarps;
    return ((a > b ? a : b) * sizeof(unsigned) + 255) & ~(size_t)255;
}
inline size_t stream_partial_bytes(int sms) { return (size_t)sms * 2 * kConsumerWarps * kSlotFloats * sizeof(float); }

// GPU quantizer (quantize_gpu.cu): three launches on `stream`; err = device error word.
cudaError_t launch_quantize_f32(const float *w, int N, int K, uint8_t *packed, uint8_t *scale, float *global_scale,
                                unsigned *err, int sms, cudaStream_t stream);
cudaError_t launch_quantize_bf16(const uint16_t *w, int N, int K, uint8_t *packed, uint8_t *scale,
                                 float *global_scale, unsigned *err, int sms, cudaStream_t stream);

cudaError_t launch_stream(int variant, const CUtensorMap &tw, const CUtensorMap &ts, const StreamParams &p,
                          int smem, cudaStream_t stream);
cudaError_t launch_generic(const GenericParams &p, cudaStream_t stream);
cudaError_t stream_set_smem_limits(int smem_optin);
cudaError_t device_error_word(unsigned **ptr);  // device address of the error word
cudaError_t launch_selftest_wait_timeout(unsigned *err, cudaStream_t stream);  // selftest.cu

// tcgen05 kernel (gemv_tc.cu): units of 128 rows x 256 k; T = 8 or 16 staged
// tokens; an even number of weight stages.  K is cut into `groups` k-groups
// (tc_group_host: the first KC % groups get one unit column more); the CTAs
// [cstart[g], cstart[g+1]) stream group g.  max_seg bounds the row blocks any
// one CTA touches (its partial-tile slots).
constexpr int kTcUnitKHost = 256;
constexpr int kTcMaxGroups = 32;
constexpr int kTcMaxParts = 256;   // most parts of one split row block
// fp32 partial tile of one (CTA, row-block segment) of the tcgen05 kernel:
// 128 rows x max(T, 16) tokens
#ifdef __CUDACC__
__host__ __device__
#endif
constexpr int tc_partial_floats(int T) { return kUnitRows * (T < 16 ? 16 : T); }
constexpr int kTcReduceChunk = 4;  // partial tiles whose loads the reduction keeps in flight at once
struct TcPartition {
    int groups;
    int max_seg;
    int max_parts;
    int row_blocks;
    int cstart[kTcMaxGroups + 1];
};
int tc_smem_bytes(int stages, int T, int kg_max);
void tc_group_host(int g, int groups, int KC, int *kstart, int *kg);
cudaError_t tc_set_smem_limit(int smem_optin);
// Launches the GEMV with programmatic dependent launch: it may start (and
// stream weights) while the kernel ahead of it on the stream is finishing; it
// reads X and writes the workspace and Y only after that kernel completes.
// tx (T = 16 only): the pass's bf16 X (p.x) as a 3D tensor {64 k, n tokens,
// K/64}, box {64, 16, 4} = one unit, 128-byte swizzle (tokens past n read as
// zeros).  With T = 8 the kernel bulk-copies X rows from p.x itself.
// Launches the GEMV and then the split-row reduction, both with programmatic
// dependent launch.
// T = 32: tx views the pass's f16 X (written by launch_tc_x16) with box
// {64, 32, 4}.
cudaError_t launch_tc(const CUtensorMap &tw, const CUtensorMap &ts, const CUtensorMap &tx, const StreamParams &p,
                      const TcPartition &part, int T, int smem, cudaStream_t stream);
// x16[t][k] = f16(x[t][k] * 2^-8) for the 32-token kernel (programmatic
// dependent launch; |x| >= 2^24 sets device error bit 8).  x, x16 16-byte
// aligned, n * K a multiple of 8.
cudaError_t launch_tc_x16(const uint16_t *x, uint16_t *x16, int n, int K, unsigned *err, cudaStream_t stream);

// Workspace a call needs (host-side plan; no GPU work): bytes of the zeroed
// counter region at offset 0 and in total.  Returns an nvfp4_status.
int workspace_layout(int n, int N, int K, const void *opts, size_t *counter_bytes, size_t *total_bytes);

}  // namespace nvfp4
