/*
 * nvfp4_gemv.h -- C ABI of the GB300 (sm_103a) NVFP4 batched decode GEMV.
 *
 * The operation (atlas pull request #266, "perf(decode): n>=4 tiled QKV +
 * o_proj GEMV for NVFP4 batched decode", section "What it does"): for a tile
 * of n concurrent decode tokens, compute the attention projection
 *
 *     Y[t, r] = bf16( g * sum_{k<K} X[t, k] * E2M1(W[r, k]) * E4M3(S[r, k/16]) )
 *
 * for t < n, r < N, reading the NVFP4 weight matrix from HBM once for all n
 * tokens instead of once per token.  The same pull request's section
 * "Correctness argument" and its review thread's "Numeric identity" caveat fix
 * the invariant this library keeps: a batched call returns, bit for bit, what
 * n single-token (n == 1) calls of the same variant return.
 *
 * Data layout (all row-major, no padding, no swizzle):
 *   w_packed       [N][K/2] bytes   E2M1 codes; element 2i of a row is the LOW
 *                                    nibble of byte i, element 2i+1 the high one.
 *   w_scale_e4m3   [N][K/16] bytes  one E4M3 scale per 16 consecutive k.
 *   w_global_scale 1 float          fp32 global scale g.
 *   x_bf16         [n][K] bf16      activations (uint16 bit patterns).
 *   y_bf16         [n][N] bf16      output, fully overwritten.
 * E2M1: 1 sign, 2 exponent, 1 mantissa bit (OCP Microscaling Formats v1.0).
 * E4M3: bias 7, max 448, S.1111.111 = NaN (OCP 8-bit floating point).
 *
 * Conventions shared by every entry point:
 *   - The caller owns every buffer; the library never frees or keeps them.
 *   - Device calls are asynchronous on `stream` and never synchronize it.
 *   - y_bf16 must not overlap any input.
 *   - On a non-OK status nothing was launched, and nvfp4_last_error() returns
 *     a message for this thread.
 *   - Pointers named "device" must be device (or managed) memory of the
 *     current device; pointers named "host" must be host memory.
 */
#ifndef NVFP4_GEMV_H
#define NVFP4_GEMV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nvfp4_status {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,     /* null pointer, bad size, K % 16 != 0, ... */
    NVFP4_ERR_MISALIGNED = 2,      /* device quantizer buffers unaligned (the GEMV takes a slower kernel instead) */
    NVFP4_ERR_UNSUPPORTED = 3,     /* device is not sm_103, or option not available */
    NVFP4_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed; see nvfp4_last_error() */
    NVFP4_ERR_DEVICE_TIMEOUT = 5,  /* a kernel gave up waiting on a barrier (see nvfp4_device_error) */
    NVFP4_ERR_WORKSPACE = 6,       /* caller workspace too small */
    NVFP4_ERR_DEVICE_INPUT = 7,    /* a kernel met an input it cannot use (see nvfp4_device_error) */
    NVFP4_ERR_DEVICE_BOUNDS = 8    /* debug-bounds build: a device index check failed (see nvfp4_device_error) */
} nvfp4_status;

/* Kernel variants (selectable through nvfp4_gemv_opts; AUTO picks per shape). */
typedef enum nvfp4_variant {
    NVFP4_VARIANT_AUTO = 0,
    NVFP4_VARIANT_MMA = 1,      /* TMA ring + register dequant + mma.sync f16 tensor cores */
    NVFP4_VARIANT_SIMT = 2,     /* TMA ring + register dequant + fp32 CUDA-core FMAs */
    NVFP4_VARIANT_GENERIC = 3,  /* plain loads, any K % 16 == 0 and any alignment */
    NVFP4_VARIANT_TC = 4,       /* TMA ring + dequant into tensor memory + tcgen05.mma kind::f16 */
    NVFP4_VARIANT_FP4 = 5       /* TMA ring straight into block-scaled tcgen05.mma kind::mxf4nvf4 (W as
                                   stored, X as a sum of 8 NVFP4 terms written by a small prep kernel);
                                   AUTO's choice for K <= 32768 */
} nvfp4_variant;

/* Token tiling.  ONE_PASS streams W once for all n tokens (chunks of up to 16
 * tokens when n > 16 or shared memory is short).  GREEDY_321 is the pages'
 * prior art (atlas #266, "What it does"): tiles of 3 tokens, then a 2 or 1
 * remainder, each tile re-reading W -- kept to measure against. */
typedef enum nvfp4_tiling {
    NVFP4_TILING_AUTO = 0,
    NVFP4_TILING_ONE_PASS = 1,
    NVFP4_TILING_GREEDY_321 = 2
} nvfp4_tiling;

typedef struct nvfp4_gemv_opts {
    int variant;             /* nvfp4_variant */
    int tiling;              /* nvfp4_tiling */
    int num_ctas;            /* 0 = one CTA per SM; else 1..#SMs (persistent grid size) */
    int stages;              /* 0 = as many TMA ring stages as shared memory allows; else 2..8 */
    void *workspace;         /* NULL = library-owned per-stream workspace; else device memory */
    size_t workspace_bytes;  /* size of `workspace` (see nvfp4_gemv_workspace_size); if nonzero (with or without
                                `workspace`) the plan keeps its scratch within it: when the FP4 plan needs
                                more, AUTO takes the tcgen05 kernel, in 8-token passes if its 32-token pass
                                needs more too */
    int inflight;            /* FP4 kernel: most weight stages requested and not yet landed per CTA (0 = default) */
} nvfp4_gemv_opts;

/* Launch plan the library would use (for tests and benchmarks). */
typedef struct nvfp4_gemv_plan_info {
    int variant;         /* resolved nvfp4_variant */
    int tiling;          /* resolved nvfp4_tiling */
    int passes;          /* weight passes (token tiles) */
    int tile_tokens[16]; /* tokens per pass (first 16 passes) */
    int num_ctas;        /* grid size of each launch */
    int stages;          /* TMA ring stages */
    int smem_bytes;      /* dynamic shared memory per CTA */
    long long units;     /* work units (128 rows x 128 k; 128 x 256 for TC) per pass */
} nvfp4_gemv_plan_info;

/*
 * Y[n][N] = X[n][K] . W^T with NVFP4 W (see the file header for the formula).
 *
 * w_packed, w_scale_e4m3, w_global_scale_f32, x_bf16: device, read only.
 * y_bf16: device, written.  n >= 0 (n == 0 is a no-op), N >= 1, K >= 16 and
 * K % 16 == 0.  Any n is accepted.  The fast paths need K % 256 == 0 and
 * 16-byte aligned w_packed, w_scale_e4m3 and x_bf16 (other inputs take the
 * GENERIC kernel).  For K <= 32768 AUTO takes the FP4 kernel: one read of W
 * for up to 16 tokens (passes of 16 above, the weights of a pass that another
 * follows kept in L2), each token's activations written as 8 NVFP4 terms
 * (every 16-element block with its own power-of-two scale, so the full bf16
 * range is taken; a block's terms leave at most 1.5e-7 of its largest entry)
 * by a small prep kernel launched ahead of the GEMV.  Every output equals the
 * single-token call's bit for bit, whatever n.  For K > 32768 it takes the
 * tcgen05 f16 kernel (one read of W per 8 tokens, or per 32 with X converted
 * by one extra small kernel per pass; on request also for smaller K, where it
 * showed rare run-to-run differences with long unit ranges per CTA on GB300).
 * The streaming CUDA-core kernels (MMA, SIMT) take up to 16 tokens per pass
 * (fewer when n * K is too large for shared memory), each pass re-reading W.
 * The tcgen05 path scales X by 2^-8 before its f16 conversion: entries with
 * |x| >= 65520 * 2^8 (about 1.68e7) are out of its range and set the device
 * error word (nvfp4_device_error), and entries below 2^-6 lose relative
 * precision in f16 subnormals.  The MMA and SIMT kernels convert X to f16 too
 * (scaled down by a power of two only when some |x| would overflow), with the
 * same loss for small entries.  The FP4 and GENERIC kernels have neither.
 * The GEMV kernels are launched with programmatic dependent launch: when the
 * kernel ahead of them on `stream` allows its dependents to start early, the
 * GEMV begins reading w_packed and w_scale_e4m3 before that kernel finishes
 * (it reads x_bf16, w_global_scale_f32 and its workspace and writes y_bf16 only
 * after that kernel has completed).  So the weights must be written either by
 * a non-kernel operation (a copy, a memset) or by a kernel that completes
 * before the call's first kernel is launched, or one that allows its
 * dependents to start only after its last write to them (this library's
 * kernels do: the quantizer's last kernel writes before it allows them).
 * Uses a library-owned workspace tied to `stream`, allocated on the first call
 * on that stream (make that first call before capturing `stream` in a graph).
 * Calls on different streams may run concurrently.
 * Returns NVFP4_OK or an error status; never synchronizes.
 */
nvfp4_status nvfp4_gemv_batched(const uint8_t *w_packed, const uint8_t *w_scale_e4m3,
                                const float *w_global_scale_f32, const uint16_t *x_bf16,
                                uint16_t *y_bf16, int n, int N, int K, cudaStream_t stream);

/* Same as nvfp4_gemv_batched with explicit options (NULL = defaults).  With a
 * caller workspace, concurrent calls must use distinct workspaces; the first
 * use of a workspace must see it zeroed (cudaMemset), and every completed call
 * leaves it zeroed again. */
nvfp4_status nvfp4_gemv_batched_ex(const uint8_t *w_packed, const uint8_t *w_scale_e4m3,
                                   const float *w_global_scale_f32, const uint16_t *x_bf16,
                                   uint16_t *y_bf16, int n, int N, int K, cudaStream_t stream,
                                   const nvfp4_gemv_opts *opts);

/*
 * nvfp4_gemv_batched without any device allocation.  The pages have no
 * counterpart: this entry point exists for callers that cannot call cudaMalloc
 * -- engines that reserve nearly all device memory in their own pool up front
 * (a library allocation would fail or fragment it), code that must not
 * allocate once serving has started (cudaMalloc can synchronize the device),
 * and plugins that only receive pointers from a host program owning all
 * device memory.
 * Arguments, layout, ownership and validation as nvfp4_gemv_batched; the
 * caller still passes every input and output buffer.  The kernels' scratch
 * (split-tile counters and fp32 partial tiles) is a static device array
 * inside the library of 8 MiB (8,388,608 bytes, held by every GPU that loads
 * the library until the process exits); a call whose plan needs more scratch
 * than that (nvfp4_gemv_workspace_size) gets NVFP4_ERR_WORKSPACE.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current: make that
 * first call before any stream capture.  Each call clears the counters with
 * cudaMemsetAsync on `stream`.  All calls on a device share the array, so
 * calls that can overlap on the GPU race and may return wrong results:
 * serialize them (one stream), or use nvfp4_gemv_batched_ex with a workspace
 * per stream.  Never calls cudaMalloc or cudaFree.
 */
nvfp4_status nvfp4_gemv_batched_noalloc(const uint8_t *w_packed, const uint8_t *w_scale_e4m3,
                                        const float *w_global_scale_f32, const uint16_t *x_bf16,
                                        uint16_t *y_bf16, int n, int N, int K, cudaStream_t stream);

/*
 * Gate/up projection with the SwiGLU activation fused into its output, for
 * the dense FFN of the speculative-verify step over m = 4..8 draft tokens that
 * runs through batched GEMV (rustdoc of spark_model/layers/mod.rs, the
 * FfnComponent enum's dense SwiGLU variant and the can_forward_km /
 * try_forward_km methods).  The SwiGLU form is the usual one; the pages name
 * it without a formula:
 *
 *     h[t, f] = bf16( silu(G[t, f]) * U[t, f] ),   silu(a) = a / (1 + exp(-a)),
 *
 * with G and U the fp32 GEMV results (x g, not rounded to bf16 first) of the
 * gate and up rows, and silu and the product in fp32.
 *
 * w_packed [2F][K/2], w_scale_e4m3 [2F][K/16]: the gate and up matrices with
 * their rows interleaved -- row 2f is gate row f, row 2f+1 is up row f -- and
 * one global scale for both (quantize the interleaved matrix as one tensor,
 * e.g. with nvfp4_quantize_bf16).  x_bf16 [n][K]; h_bf16 [n][F] is written.
 * Same conventions and errors as nvfp4_gemv_batched (same invariant: a batched
 * call equals n single-token calls bit for bit); runs on the tensor-core
 * paths only (FP4, or tcgen05 for K > 32768), so K % 256 != 0 or unaligned
 * inputs give NVFP4_ERR_UNSUPPORTED.
 * F >= 1.
 */
nvfp4_status nvfp4_gemv_swiglu(const uint8_t *w_packed, const uint8_t *w_scale_e4m3,
                               const float *w_global_scale_f32, const uint16_t *x_bf16, uint16_t *h_bf16,
                               int n, int F, int K, cudaStream_t stream);

/*
 * Dense SwiGLU FFN of n tokens (the verify FFN above): h = nvfp4_gemv_swiglu
 * (W_gu, x), then y = W_down . h with nvfp4_gemv_batched -- two calls on
 * `stream`, each reading its weights once for all n tokens.
 * x_bf16 [n][D], h_bf16 [n][F] (device scratch owned by the caller, written),
 * y_bf16 [n][D] (written); W_gu as in nvfp4_gemv_swiglu with K = D; W_down
 * [D][F/2] packed, [D][F/16] scales.  D and F: positive multiples of 16 (256
 * for the fast path of each call).  Errors as the two calls.
 */
nvfp4_status nvfp4_ffn_swiglu(const uint8_t *w_gu_packed, const uint8_t *w_gu_scale_e4m3,
                              const float *w_gu_global_scale_f32, const uint8_t *w_down_packed,
                              const uint8_t *w_down_scale_e4m3, const float *w_down_global_scale_f32,
                              const uint16_t *x_bf16, uint16_t *h_bf16, uint16_t *y_bf16, int n, int D, int F,
                              cudaStream_t stream);

/*
 * Grouped read-once GEMV over routed experts, for MoE decode (rustdoc of
 * spark_model/layers/mod.rs, moe_grouped_decode_min_rows: with the tokens
 * sorted by expert, the grouped path reads every routed expert's weights one
 * time for all of its tokens rather than one time per token).  For every expert e and every assignment j in
 * [expert_offsets[e], expert_offsets[e+1]):
 *
 *     Y[j, r] = bf16( g_e * sum_k X[sorted_token[j], k] * E2M1(W_e[r, k]) * E4M3(S_e[r, k/16]) )
 *
 * or, with swiglu = 1, H[j, f] = bf16(silu(Y'[j, 2f]) * Y'[j, 2f+1]) from the
 * unrounded values Y' (rows interleaved gate/up as in nvfp4_gemv_swiglu).
 * Each assignment's sum is computed in a fixed order that does not depend on
 * the other tokens routed to the same expert.  The routing weights and the
 * combine of a token's expert outputs are not part of this call.
 *
 * w_packed [E][N][K/2], w_scale_e4m3 [E][N][K/16]: device, 16-byte aligned;
 * w_global_scale_f32 [E]: device; x_bf16 [n_tokens][K]: device, 16-byte
 * aligned; expert_offsets [E+1] and sorted_token [A] (int32): device;
 * y_bf16 [A][N] (swiglu: [A][N/2]): device, written, row j = assignment j.
 * 1 <= E <= 1024, A >= 0 (0: no-op), n_tokens >= 1, N a positive multiple
 * of 16, K a multiple of 32 in [32, 7168].  K % 256 == 0: a persistent grid
 * (one CTA per SM) streams the row blocks of the experts that have tokens
 * through a ring of shared-memory slots (TMA) and multiplies on tensor cores
 * (mma.sync, f16 x f16 -> fp32); other K: one CTA per (expert, row block),
 * bulk-copied, SIMT FMAs (whose 16 staged tokens, 8 with swiglu, and 16
 * weight rows must fit shared memory: K <= 5632 without swiglu).  Either
 * way each routed expert is read once whatever its token count.
 * Asynchronous on `stream`; one launch.  Errors: NVFP4_ERR_INVALID_ARG,
 * NVFP4_ERR_MISALIGNED, NVFP4_ERR_UNSUPPORTED (K too large), NVFP4_ERR_CUDA.
 * Offsets outside [0, A] or decreasing and token indices outside
 * [0, n_tokens) are skipped by the kernel and set bit 32 of the device error
 * word (nvfp4_device_error).
 */
nvfp4_status nvfp4_moe_gemv_grouped(const uint8_t *w_packed, const uint8_t *w_scale_e4m3,
                                    const float *w_global_scale_f32, const uint16_t *x_bf16,
                                    const int32_t *expert_offsets, const int32_t *sorted_token, uint16_t *y_bf16,
                                    int E, int A, int n_tokens, int N, int K, int swiglu, cudaStream_t stream);

/* Bytes of device workspace a call with these options needs (opts may be NULL). */
nvfp4_status nvfp4_gemv_workspace_size(int n, int N, int K, const nvfp4_gemv_opts *opts,
                                       size_t *bytes);

/* Describe the launches nvfp4_gemv_batched_ex would make, without launching.
 * Pointer alignment is taken as 16 bytes (the fast path's requirement). */
nvfp4_status nvfp4_gemv_plan(int n, int N, int K, const nvfp4_gemv_opts *opts,
                             nvfp4_gemv_plan_info *info);

/*
 * Host-side NVFP4 quantizer for making test data (not on the GEMV path).  It
 * produces the weight format of the file header as the test workloads state
 * it: E2M1 values, one E4M3 scale per 16-element K block equal to the block's
 * max |w| / 6 in units of the fp32 global scale, and g = amax / (6 * 448) so
 * that the largest block scale is E4M3's largest value (the pages give the
 * format and leave the scale choice open; this is the plainest reading).
 * w: host fp32 [N][K]; w_packed: host [N][K/2]; w_scale: host [N][K/16];
 * global_scale: host, 1 float.  amax = max|w|; g = amax / (6 * 448) in fp32
 * (1 when amax == 0); s = E4M3_rne_sat(blockabsmax / (6 g)); code =
 * E2M1_rne_sat(w / (E4M3(s) g)), code 0 when the magnitude rounds to 0 or s is
 * 0.  All arithmetic fp32.  Non-finite input -> NVFP4_ERR_INVALID_ARG.
 */
nvfp4_status nvfp4_quantize_ref(const float *w, int N, int K, uint8_t *w_packed, uint8_t *w_scale,
                                float *global_scale);

/*
 * Device NVFP4 quantizer: the runtime requantization of BF16 (or fp32)
 * attention weights to FP4 that the pages' measurements depend on (atlas pull
 * request #266, conversation, "Tiebreaker: the win is the BF16->FP4 requant
 * path").  Same formula and fp32 rounding as nvfp4_quantize_ref (every
 * division and product correctly rounded, no fused multiply-add), so for the
 * same weights it writes the same bytes and the same g.  nvfp4_quantize_bf16
 * takes bf16 weights (uint16 bit patterns), widened exactly to fp32 first.
 *
 * w_f32 / w_bf16: device [N][K], read only, 16-byte aligned.
 * w_packed: device [N][K/2], written, 8-byte aligned (layout of the file header).
 * w_scale_e4m3: device [N][K/16], written.
 * w_global_scale_f32: device, 1 float, 4-byte aligned, written (it holds amax
 *   between the launches, so it must not be read by other work until the call's
 *   launches on `stream` are done).
 * N >= 1, K >= 16, K % 16 == 0, N * K <= 2^40.  No output may overlap w.
 * Three asynchronous launches on `stream` (amax reduction, block quantizer,
 * finish) plus a 4-byte memset of w_global_scale_f32; no workspace.
 * Errors: NVFP4_ERR_INVALID_ARG (null pointer, bad size), NVFP4_ERR_MISALIGNED
 * (alignment above), NVFP4_ERR_CUDA.  A non-finite weight cannot be detected
 * before launch: it sets bit 16 of the device error word (nvfp4_device_error
 * then returns NVFP4_ERR_DEVICE_INPUT) and the outputs are not meaningful.
 */
nvfp4_status nvfp4_quantize(const float *w_f32, int N, int K, uint8_t *w_packed, uint8_t *w_scale_e4m3,
                            float *w_global_scale_f32, cudaStream_t stream);
nvfp4_status nvfp4_quantize_bf16(const uint16_t *w_bf16, int N, int K, uint8_t *w_packed,
                                 uint8_t *w_scale_e4m3, float *w_global_scale_f32, cudaStream_t stream);

/* Synchronize `stream`, then report and clear the library's device error word
 * (one word per device, shared by every stream).  *code receives the raw word
 * (0 = no error); its bits:
 *   1, 2, 4  a GEMV kernel gave up on a wait (TMA stage full / stage free /
 *            copies in flight at exit) after about 2 s;
 *   8        a GEMV met |x| >= 65520 * 2^8 (see nvfp4_gemv_batched);
 *   16       the device quantizer met a non-finite weight;
 *   32       the grouped expert GEMV met bad routing data;
 *   64       a tcgen05 or FP4 GEMV found its dynamic shared memory off a
 *            1024-byte boundary and computed nothing (a platform fault, never
 *            expected);
 *   128      (only the library built with -DNVFP4_DEBUG_BOUNDS,
 *            libnvfp4_gemv_debug.so) a device check of a computed workspace
 *            index (partial tile, split-row counter) failed and the access was
 *            skipped.
 * Returns NVFP4_ERR_DEVICE_TIMEOUT when any of bits 1, 2, 4 is set (the
 * library then also re-zeroes its own workspaces so later calls start clean),
 * else NVFP4_ERR_DEVICE_BOUNDS when bit 128 is set, else NVFP4_ERR_UNSUPPORTED
 * when bit 64 is set, else NVFP4_ERR_DEVICE_INPUT when bit 8, 16 or 32 is set,
 * else NVFP4_OK. */
nvfp4_status nvfp4_device_error(cudaStream_t stream, int *code);

/* Self-test of the failure path (no fault involved): enqueues on `stream` one
 * kernel whose single thread waits on a shared-memory barrier phase that
 * nothing completes; like every wait in the library's kernels it gives up
 * after about 2 s and sets bit 1 of the device error word, so that a later
 * nvfp4_device_error returns NVFP4_ERR_DEVICE_TIMEOUT (and re-zeroes the
 * workspaces) while the CUDA context stays usable.  Asynchronous; returns
 * NVFP4_OK or NVFP4_ERR_CUDA. */
nvfp4_status nvfp4_selftest_wait_timeout(cudaStream_t stream);

/* Message for the last non-OK status returned on this thread ("" if none):
 * which argument or check failed, or the CUDA call and its error string.  The
 * pointer stays valid until the next library call on this thread. */
const char *nvfp4_last_error(void);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int nvfp4_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GEMV_H */
