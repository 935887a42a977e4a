// gemv_tc.cu -- the tcgen05 (5th-generation tensor core) NVFP4 batched GEMV.
//
// Computes Y[t, r] = g * sum_k X[t, k] * E2M1(W[r, k]) * E4M3(S[r, k/16]) for all
// n <= 16 tokens from ONE pass over W (atlas pull request #266, "What it
// does": each tile of decode tokens reads the projection weight once; here
// the tile is all n tokens), and up to 32 tokens per pass in a 32-token mode
// (below) for the mid-M widths.
//
// Work split.  The weight matrix is cut into units of 128 rows x 256 k (128 B
// of every packed row + 16 scale bytes per row).  K is cut into `groups`
// k-groups of at most ten units, so that one group's slice of X for 16 tokens
// stays resident in shared memory; the CTAs [cstart[g], cstart[g+1]) of the
// persistent grid stream the units of group g in row-block-major order, each
// CTA owning an equal contiguous range ("stream-K" within the group), so every
// SM moves the same bytes.  A row block held whole by one CTA is finished
// there; the parts of a split row block are published as fp32 tiles with
// plain stores (no waiting inside the GEMV) and a small reduction kernel that
// follows sums them in CTA order (fixed order: deterministic, and independent
// of n, since the partition does not depend on n).
//
// X: each CTA stages the bf16 rows of its k-group's slice of X itself and
// converts them to f16 times 2^-8 (exact: a power of two) in the tensor
// core's K-major 128-byte-swizzled operand layout (8-token atoms of 1024 B).
// With n <= 8 (T = 8) the X warp fetches each token's whole slice with one
// bulk copy into a staging area, and the epilogue warps convert it into the
// swizzled layout; rows n..7 are zeroed beforehand.  No separate conversion
// kernel or X buffer in global memory.  With 9 to 32 tokens (T = 32) the
// group's X would not fit beside the weight ring: X is converted once per
// pass by tc_x16_kernel into the workspace and the X warp streams each unit's
// {64 k, 32 tokens, 4} box into a ring of kTcXRing slots, which the unit's
// two issuers release with a commit; same partition, so the results equal
// those of n <= 8 calls bit for bit.  (A 16-token mode that converted X in
// place per k-group returned run-to-run differing outputs in some row blocks
// on GB300 for long unit ranges per CTA; it was removed, its cause not found.)
//
// Warp roles (576 threads, one CTA per SM):
//   warp 0       weight producer: 2D TMA loads of the unit's W tile
//                (128B-swizzled) and scale tile into a ring of S stages.
//   warp 1       X loads (see above).
//   warps 2-5    MMA issuers.  Unit i uses tensor-memory A buffer i % 2;
//                each buffer has two issuers, one per 128-k half, each with
//                its own fp32 accumulators in tensor memory per row-block
//                segment buffer (summed by the epilogue in fixed order), so
//                the two halves' MMAs run concurrently and every barrier of
//                a buffer half has one waiter that sees each of its phases.
//                8 x tcgen05.mma.kind::f16 per half unit, M = 128 weight
//                rows, N = 16 token columns, K = 16; A from tensor memory,
//                B (= X) from shared memory.
//   warps 6-13   dequantise: thread = weight row; warp set b (warps 6-9,
//                10-13) converts the units of A buffer b, warp (lane quarter
//                q) all 256 k of rows 32q..32q+31 into f16 (E2M1 cvt times
//                the E4M3 block scale: exact) with four tcgen05.st of 32
//                columns, handing each 128-k half over as it is stored.
//   warps 14-17  X conversion (bf16 -> f16 x 2^-8 in shared memory, unit by
//                unit in the order the CTA uses them), then the epilogue:
//                per finished row-block segment, tcgen05.ld of the
//                issuers' accumulators, summed in a fixed order, then either
//                x g x 2^8 and bf16 store (whole row block) or an fp32
//                partial tile -- off the streaming path.
//
// With n <= 8 only tokens 0-7 are staged and the MMA's tokens 8-15 read a
// 1024-byte zero block.  The 2^-8 prescale of X keeps |x| up to
// 65504 * 2^8 ~ 1.68e7 finite in f16; larger entries set the device error
// word (the output is then not meaningful).
//
// Programmatic dependent launch: the kernel lets the next kernel on the stream
// (the split-row reduction) launch as soon as its CTAs are set up -- the
// reduction needs no shared memory and few registers, so its CTAs sit next to
// the GEMV CTAs, waiting for this grid, and never keep the next call's GEMV
// off an SM -- and it starts its own weight stream before the kernel ahead of
// it has finished; X, the global scale, the workspace and Y are touched only
// after griddepcontrol.wait.  Weights and scales are therefore read as
// constants of the call.
//
// Every wait is bounded (2 s of %globaltimer); on a timeout the kernel sets
// the device error word, skips the remaining work, waits (bounded) for its
// own copies and MMAs, and frees its tensor memory before exiting.
#include "internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

#include <cuda_bf16.h>

namespace nvfp4 {

namespace {

constexpr int kTcUnitK = 256;                    // k per unit (128 packed bytes per row)
constexpr int kTcWBytes = kUnitRows * 128;       // 16384
constexpr int kTcSBytes = kUnitRows * 16;        // 2048
constexpr int kTcABufs = 2;                      // A buffers, 128 columns each
constexpr int kTcIssuersPerBuf = 2;              // MMA issuers per A buffer (each takes 1 / this of its parts)
constexpr int kTcAColsPerUnit = kTcUnitK / 2;    // two f16 per 32-bit column
constexpr int kTcIssuers = kTcABufs * kTcIssuersPerBuf;
constexpr int kTcDCol = kTcABufs * kTcAColsPerUnit;  // accumulators [issuer][segment buffer 2][16 cols] from here
constexpr uint32_t kTcTmemCols = 512;
constexpr int kTcWarpProducer = 0;
constexpr int kTcWarpX = 1;
constexpr int kTcWarpIssuer0 = kTcWarpX + 1;                    // issuers: warps 2 ..
constexpr int kTcWarpDequant0 = kTcWarpIssuer0 + kTcIssuers;    // dequant: the next 16 warps
// Eight dequant warps in two sets of four: set b converts the units of A
// buffer b, a warp all 256 k of its 32 rows, so each warp has two units'
// time per unit it converts (its per-unit latencies -- barrier round trips,
// shared-memory loads, the tensor-memory store -- overlap with the other
// set's unit).
constexpr int kTcDequantWarps = 8;
constexpr int kTcWarpEpilogue0 = kTcWarpDequant0 + kTcDequantWarps;  // epilogue: warps 14..17
constexpr int kTcEpilogueWarps = 4;
constexpr int kTcThreads = (kTcWarpEpilogue0 + kTcEpilogueWarps) * 32;  // 576
// Registers: the GEMV keeps room for one warp of the reduction kernel (at
// most kTcReduceRegs registers a thread) on every SM sub-partition (16 K
// registers each; warp w sits on sub-partition w % 4), so that a reduction CTA
// fits beside it.
constexpr int kTcReduceRegs = 96;
constexpr int kTcWarpsPerSmsp = (kTcThreads / 32 + 3) / 4;
constexpr int kTcMaxRegs = ((16384 - 32 * kTcReduceRegs) / (32 * kTcWarpsPerSmsp)) & ~7;
static_assert(kTcMaxRegs >= 64, "register budget");
constexpr float kTcXScale = 1.0f / 256.0f;       // 2^-8 applied to X before the f16 cast
constexpr float kTcXUnscale = 256.0f;
constexpr unsigned kDevErrXRange = 8u;           // some |x| >= 65520 * 2^8
constexpr unsigned kDevErrSmemBase = 64u;        // dynamic shared memory not 1024-byte aligned
// 32 staged tokens (n = 17..32): X is not resident but streamed per unit
// through a ring of kTcXRing slots, already converted to f16 x 2^-8 by
// tc_x16_kernel (the k-group partition stays that of n <= 16, so results do
// not depend on n).
constexpr int kTcXRing = 4;
// x-barrier slots: one per unit column of the group (T <= 16) or ring slot (T = 32)
__host__ __device__ constexpr int tc_xbars(int KG) { return KG > kTcXRing ? KG : kTcXRing; }

static_assert(kTcDCol + kTcIssuers * 2 * 32 <= (int)kTcTmemCols, "tensor memory (up to 32 token columns)");

// Each A buffer is handed from the dequant warps to its issuer, and back, in
// kTcAParts parts of 256 / kTcAParts k (the lane-quarter warps of those k
// quarters), so MMAs start once a part is converted and a part is refilled as
// soon as its MMAs are done.  Two parts measured best (four: more commits and
// barrier round trips per unit for no shorter cycle).
constexpr int kTcAParts = 2;
constexpr int kTcStepsPerPart = 16 / kTcAParts;  // MMA k-steps (16 k each) per part
constexpr int kTcPartsPerIssuer = kTcAParts / kTcIssuersPerBuf;
static_assert(kTcPartsPerIssuer * kTcIssuersPerBuf == kTcAParts, "issuers split a buffer's parts evenly");

// barriers: full[S] empty[S] xloaded[XB] xfull[XB] afull[B][P] aempty[B][P] dfull[I][2] dempty[2] final[I] xreq
// (B A buffers, P parts, I issuers, XB = tc_xbars(KG))
__host__ __device__ constexpr int tc_barrier_count(int S, int KG) {
    return 2 * S + 2 * tc_xbars(KG) + 2 * kTcABufs * kTcAParts + 2 * kTcIssuers + 2 + kTcIssuers + 1;
}
// Weight stages requested before X: the rest of the ring is requested only
// once the X warp has requested X, so that X does not queue behind a full
// ring of weight traffic from this SM (0, 2, 4, 8 measured: 4 is best).
constexpr int kTcStagesBeforeX = 4;
constexpr int kTcXConverterWarps = kTcEpilogueWarps;  // the epilogue warps convert X before their epilogue work

// Group g of `groups` k-groups over KC unit columns: first unit column and width.
__host__ __device__ inline void tc_group(int g, int groups, int KC, int *kstart, int *kg) {
    const int q = KC / groups, r = KC % groups;
    *kg = q + (g < r ? 1 : 0);
    *kstart = g * q + (g < r ? g : r);
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, int c0, int c1, int c2, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}

// Plain bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Output of one finished row `row` (this lane's) for all tokens: y = bf16(v *
// gs), or, with p.swiglu, the gated form -- the rows 2f (gate) and 2f + 1 (up)
// of a pair sit in lanes 2i and 2i + 1 of the calling warp, and the even lane
// stores h[t][f] = bf16(silu(gate) * up), silu(a) = a / (1 + exp(-a)), in fp32.
// Every lane of the warp must call it (the pair exchange is a shuffle).
// v[j] is token t0 + j.
__device__ __forceinline__ void tc_store_row(const StreamParams &p, const float (&v)[16], int row, float gs,
                                             int t0 = 0) {
    const int lane = threadIdx.x & 31;
    if (!p.swiglu) {
        if (row < p.N) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int t = t0 + j;
                if (t < p.n) {
                    __nv_bfloat16 hv = __float2bfloat16_rn(v[j] * gs);
                    p.y[(size_t)t * p.N + row] = *reinterpret_cast<uint16_t *>(&hv);
                }
            }
        }
        return;
    }
    const int F = p.N >> 1;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int t = t0 + j;
        const float a = v[j] * gs;
        const float up = __shfl_down_sync(0xffffffffu, a, 1);
        if (t < p.n && (lane & 1) == 0 && row < p.N) {
            const float h = a / (1.0f + expf(-a)) * up;
            __nv_bfloat16 hv = __float2bfloat16_rn(h);
            p.y[(size_t)t * F + (row >> 1)] = *reinterpret_cast<uint16_t *>(&hv);
        }
    }
}

// Two bf16 (one 32-bit word) -> two f16 of x * 2^-8.  `bad` collects, in
// bits 15 and 31, finite entries with |x| >= 2^24: the only bf16 values whose
// scaled f16 would overflow (65520 * 2^8 lies between 2^24 - 2^16 and 2^24).
// Per 15-bit magnitude m: m + 0x3480 reaches bit 15 iff m >= 0x4B80 (2^24) and
// m + 0x0080 iff m >= 0x7F80 (inf or NaN); neither sum carries out of its half.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, uint32_t &bad) {
    const uint32_t m = w & 0x7FFF7FFFu;
    bad |= (m + 0x34803480u) & ~(m + 0x00800080u) & 0x80008000u;
    const float lo = __uint_as_float(w << 16) * kTcXScale;
    const float hi = __uint_as_float(w & 0xFFFF0000u) * kTcXScale;
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

}  // namespace

// X area: kg_max units x 16 token rows x 512 B -- the f16 X (8 rows) plus the
// bf16 staging (8 rows) for T = 8; for T = 32, kTcXRing slots of 32 token
// rows x 512 B.
// The dynamic shared memory starts 1024-byte aligned (the kernel checks it),
// so no alignment slack is reserved: the GEMV then leaves room on its SM for a
// reduction CTA (its 1 KB of reserved shared memory).
__host__ __device__ inline int tc_xarea_bytes(int T, int kg_max) {
    return T == 32 ? kTcXRing * 32 * 512 : kg_max * 16 * 512;
}
int tc_smem_bytes(int stages, int T, int kg_max) {
    return stages * (kTcWBytes + kTcSBytes) + tc_xarea_bytes(T, kg_max) + 1024 + 8 * tc_barrier_count(stages, kg_max) +
           64;
}

void tc_group_host(int g, int groups, int KC, int *kstart, int *kg) { tc_group(g, groups, KC, kstart, kg); }

// At most kTcMaxRegs registers a thread, so that a reduction CTA can sit
// beside the GEMV CTA (see the launch notes above).
template <int T>  // staged tokens: 8 (n <= 8) or 32 (X ring, pre-converted)
__global__ void __maxnreg__(kTcMaxRegs)
    gemv_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_s,
                   const __grid_constant__ CUtensorMap tmap_x, const StreamParams p, const TcPartition part) {
    static_assert(T == 8 || T == 32, "staged tokens");
    constexpr bool kRing = T == 32;        // X streamed per unit through kTcXRing slots
    constexpr int kAcc = T < 16 ? 16 : T;  // accumulator columns per (issuer, segment buffer)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t sW = smem_u32(smem_raw);
    if (sW & 1023u) {  // the swizzled tiles need a 1024-byte aligned base; never expected
        griddep_wait();
        if (threadIdx.x == 0) atomicOr(p.err, kDevErrSmemBase);
        return;
    }
    uint8_t *const base = smem_raw;
    const int S = p.stages;                              // even (every dequant warp sees every phase)
    const int KC = p.KC;
    const int G = part.groups;

    // ---- this CTA's group and unit range
    int grp = 0;
    while (grp + 1 < G && part.cstart[grp + 1] <= (int)blockIdx.x) ++grp;
    int kstart, kg;
    tc_group(grp, G, KC, &kstart, &kg);
    const int kg_max = (KC + G - 1) / G;
    const int cg = part.cstart[grp + 1] - part.cstart[grp];
    const long long ug = (long long)part.row_blocks * kg;
    const int cl = (int)blockIdx.x - part.cstart[grp];
    const long long u0 = (long long)cl * ug / cg;
    const int count = (int)((long long)(cl + 1) * ug / cg - u0);
    const int rb0 = (int)(u0 / kg), kl0 = (int)(u0 - (long long)rb0 * kg);  // first row block, column in group
    const int nx = count < kg ? count : kg;              // X units this CTA uses

    constexpr uint32_t xslot = (uint32_t)T * 512;       // one unit's X: 4 boxes of T tokens x 64 k (128 B rows)
    const int xb = tc_xbars(kg_max);                     // x-barrier slots
    constexpr uint32_t xbox = (uint32_t)T * 128;
    const uint32_t sS = sW + S * kTcWBytes;
    const uint32_t sX = sS + S * kTcSBytes;             // X of the group [kg_max units], 1024-byte aligned
    const uint32_t sStage = sX + kg_max * xslot;        // T = 8: bf16 rows [8 tokens][kg_max * 256 k]
    const uint32_t stage_pitch = (uint32_t)kg_max * 512; // bytes per staged token row
    const uint32_t sZero = sX + tc_xarea_bytes(T, kg_max);  // 1024 zero bytes (one swizzle atom)
    const uint32_t sFull = sZero + 1024;                // W + scales of a stage landed
    const uint32_t sEmpty = sFull + 8 * S;              // dequant warps done with W + scales, count 16
    // T <= 16: [unit column] X landed (TMA, one phase) / f16 X ready (converter warps);
    // T = 32: [ring slot] X landed (TMA) / slot free (commits of the unit's issuers)
    const uint32_t sXLoaded = sEmpty + 8 * S;
    const uint32_t sXFull = sXLoaded + 8 * xb;
    const uint32_t sAFull = sXFull + 8 * xb;            // [buffer][part], count = warps per part
    const uint32_t sAEmpty = sAFull + 8 * kTcABufs * kTcAParts;   // [buffer][part], count 1 (commit)
    const uint32_t sDFull = sAEmpty + 8 * kTcABufs * kTcAParts;   // [issuer][segment buffer], count 1 (commit)
    const uint32_t sDEmpty = sDFull + 16 * kTcIssuers;  // [segment buffer], count 4 (epilogue warps)
    const uint32_t sFinal = sDEmpty + 16;               // [issuer], count 1 (commit)
    const uint32_t sXReq = sFinal + 8 * kTcIssuers;     // X requested (X warp), count 1
    const uint32_t sMisc = sXReq + 8;                   // [0] tensor-memory base
    uint32_t *const misc = reinterpret_cast<uint32_t *>(base + (sMisc - sW));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // The weight stream starts first: the producer thread sets up the ring's
    // barriers and requests the first stages before anything else (the ring is
    // touched by no other thread before the CTA barrier below).
    // Weights are read once per call: streamed with evict-first, except in a
    // pass that another pass over the same weights follows (n > 16), which
    // leaves them in L2 (evict-last) so that the next pass does not read HBM.
    const uint64_t w_policy = p.w_keep ? l2_policy_evict_last() : l2_policy_evict_first();
    int w_rb = rb0, w_kl = kl0, issued = 0;
    auto issue_w = [&](int i) {
        const int slot = i % S;
        const uint32_t full = sFull + 8 * slot;
        const int kc = kstart + w_kl;
        mbar_arrive_expect_tx(full, kTcWBytes + kTcSBytes);
        tma_load_2d(sW + slot * kTcWBytes, &tmap_w, kc * 128, w_rb * kUnitRows, full, w_policy);
        tma_load_2d(sS + slot * kTcSBytes, &tmap_s, kc * 16, w_rb * kUnitRows, full, w_policy);
        if (++w_kl == kg) {
            w_kl = 0;
            ++w_rb;
        }
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(sFull + 8 * s, 1);
            mbar_init(sEmpty + 8 * s, kTcDequantWarps / kTcABufs);
        }
        fence_barrier_init();
        const int pre = count < kTcStagesBeforeX ? count : (kTcStagesBeforeX < S ? kTcStagesBeforeX : S);
        for (; issued < pre; ++issued) issue_w(issued);
        for (int s = 0; s < xb; ++s) {
            mbar_init(sXLoaded + 8 * s, 1);
            mbar_init(sXFull + 8 * s, kRing ? kTcIssuersPerBuf : kTcXConverterWarps);
        }
        for (int b = 0; b < kTcABufs * kTcAParts; ++b) {
            mbar_init(sAFull + 8 * b, kTcDequantWarps / kTcABufs);
            mbar_init(sAEmpty + 8 * b, 1);
        }
        for (int d = 0; d < 2 * kTcIssuers; ++d) mbar_init(sDFull + 8 * d, 1);
        for (int d = 0; d < 2; ++d) mbar_init(sDEmpty + 8 * d, kTcEpilogueWarps);
        for (int h = 0; h < kTcIssuers; ++h) mbar_init(sFinal + 8 * h, 1);
        mbar_init(sXReq, 1);
        fence_barrier_init();
    }
    if (T == 32 && warp == kTcWarpX && lane == 0) prefetch_tensormap(&tmap_x);  // T = 8 uses no X map
    if (warp == kTcWarpIssuer0) {
        tc::tmem_alloc(sMisc, kTcTmemCols);
        tc::tmem_relinquish();
    }
    if (threadIdx.x < 64) sts128(sZero + threadIdx.x * 16, make_uint4(0, 0, 0, 0));
    fence_proxy_async_smem();  // the zero block is read by the tensor core
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = misc[0];
    // The reduction may launch now: its CTAs fit next to this one and only
    // wait (griddepcontrol.wait) until this grid has finished.
    if (threadIdx.x == 0) griddep_launch_dependents();

    // X conversion by the epilogue warps (converter cv = 0..3), unit column
    // by unit column in the order the CTA uses them; each warp arrives on a
    // column's barrier once its share of the column is stored.
    //   T = 8:  rows t < n of column l come from the bf16 staging row of
    //           token t (lane = 16-byte chunk of the column's 512 bytes) and
    //           go to the chunk's swizzled position; rows n..7 are zeroed by
    //           zero_x_pad before the wait for X.
    auto zero_x_pad = [&](int cv) {
        if (T != 8) return;
        const int pad = T - p.n;
        const int items = nx * 4 * pad * 8;  // 16-byte chunks
        for (int j = cv * 32 + lane; j < items; j += kTcXConverterWarps * 32) {
            const int c = j & 7, rowbox = j >> 3;  // rowbox = (column i * 4 + box b) * pad + (t - n)
            const int tp = rowbox % pad, ib = rowbox / pad;
            const int l = (kl0 + (ib >> 2)) % kg;
            sts128(sX + l * xslot + (ib & 3) * xbox + (p.n + tp) * 128 + c * 16, make_uint4(0, 0, 0, 0));
        }
    };
    auto convert_x = [&](int cv) -> bool {
        uint32_t bad = 0;
        bool ok = true;
        if (T == 8 && __any_sync(0xffffffffu, !mbar_wait_bounded(sXLoaded, 0))) ok = false;
        for (int i = 0; i < nx && ok && T == 8; ++i) {  // per column, so the MMAs can start early
            const int l = (kl0 + i) % kg;
            const uint32_t dst_box = sX + l * xslot + (uint32_t)(lane >> 3) * xbox;
            for (int t = cv; t < p.n; t += kTcXConverterWarps) {
                uint4 v = lds128(sStage + t * stage_pitch + l * 512 + lane * 16);
                v.x = bf16x2_to_f16x2_scaled(v.x, bad);
                v.y = bf16x2_to_f16x2_scaled(v.y, bad);
                v.z = bf16x2_to_f16x2_scaled(v.z, bad);
                v.w = bf16x2_to_f16x2_scaled(v.w, bad);
                sts128(dst_box + t * 128 + ((uint32_t)((lane & 7) ^ (t & 7)) << 4), v);
            }
            fence_proxy_async_smem();  // the tensor core reads these bytes through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(sXFull + 8 * l);
        }
        if (bad) atomicOr(p.err, kDevErrXRange);
        return ok;
    };

    if (warp == kTcWarpProducer) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            if (issued < count && !mbar_wait_bounded(sXReq, 0)) atomicOr(p.err, kDevErrTimeoutEmpty);
            for (; issued < count; ++issued) {
                if (!mbar_wait_bounded(sEmpty + 8 * (issued % S), ((issued / S) - 1) & 1)) {
                    atomicOr(p.err, kDevErrTimeoutEmpty);
                    break;
                }
                issue_w(issued);
            }
            // wait (bounded) for the most recent copy into every stage before exiting
            const int lo = issued > S ? issued - S : 0;
            for (int i = lo; i < issued; ++i) {
                if (!mbar_wait_bounded(sFull + 8 * (i % S), (i / S) & 1)) {
                    atomicOr(p.err, kDevErrTimeoutDrain);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp == kTcWarpX) {
        // ------------------------------------------------------------------- X
        // The unit in column l of the group sits at sX + l * xslot.
        griddep_wait();  // X may be the output of the kernel ahead of this one
        if (kRing && lane == 0) {
            // unit i's X (its unit column of the group) into ring slot i % kTcXRing,
            // once both issuers of the slot's previous unit have committed
            const uint64_t policy = l2_policy_evict_last();  // every CTA of the group reads the same X
            const int first = count < kTcXRing ? count : kTcXRing;
            int loaded = 0;
            for (; loaded < count; ++loaded) {
                const int slot = loaded % kTcXRing;
                if (loaded >= kTcXRing &&
                    !mbar_wait_bounded(sXFull + 8 * slot, ((loaded / kTcXRing) - 1) & 1)) {
                    atomicOr(p.err, kDevErrTimeoutEmpty);
                    break;
                }
                const int l = (kl0 + loaded) % kg;
                mbar_arrive_expect_tx(sXLoaded + 8 * slot, xslot);
                tma_load_3d(sX + slot * xslot, &tmap_x, 0, 0, (kstart + l) * 4, sXLoaded + 8 * slot, policy);
                if (loaded == first - 1) mbar_arrive(sXReq);  // the producer may request the rest of its ring
            }
            if (loaded < first) mbar_arrive(sXReq);
            // wait (bounded) for the copies in flight before the warp leaves
            for (int i = loaded > kTcXRing ? loaded - kTcXRing : 0; i < loaded; ++i) {
                if (!mbar_wait_bounded(sXLoaded + 8 * (i % kTcXRing), (i / kTcXRing) & 1)) {
                    atomicOr(p.err, kDevErrTimeoutDrain);
                    break;
                }
            }
        } else if (lane == 0) {
            const uint64_t policy = l2_policy_evict_last();  // every CTA of the group reads the same X
            // T = 8: one bulk copy per token, its kg units of the group (contiguous in X)
            const uint32_t bytes = (uint32_t)kg * 512;
            mbar_arrive_expect_tx(sXLoaded, bytes * (uint32_t)p.n);
            for (int t = 0; t < p.n; ++t)
                bulk_load(sStage + t * stage_pitch, p.x + (size_t)t * p.K + (size_t)kstart * kTcUnitK, bytes,
                          sXLoaded, policy);
            mbar_arrive(sXReq);  // the producer may request the rest of the weight ring
            // wait (bounded) for the copies before the warp leaves (the conversion may give up)
            if (!mbar_wait_bounded(sXLoaded, 0)) atomicOr(p.err, kDevErrTimeoutDrain);
        }
        __syncwarp();
    } else if (warp < kTcWarpDequant0) {
        // ---------------------------------------------------------- MMA issuers
        const int w = warp - kTcWarpIssuer0;  // accumulator of this issuer
        const int a = w / kTcIssuersPerBuf;   // its A buffer: units i with i % kTcABufs == a
        const int p0 = (w % kTcIssuersPerBuf) * kTcPartsPerIssuer;  // its parts of each unit
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_f16_f32(kUnitRows, kAcc);
            bool ok = true;
            int seg = 0, kl = kl0;
            for (int i = 0; i < count && ok; ++seg) {
                // segment: units [i, iend] of one row block
                int iend = i + (kg - kl) - 1;
                if (iend > count - 1) iend = count - 1;
                const int sb = seg & 1;
                if (seg >= 2 && !mbar_wait_bounded(sDEmpty + 8 * sb, ((seg >> 1) - 1) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t d_tmem = tbase + kTcDCol + w * 2 * kAcc + sb * kAcc;
                bool first = true;
                int ib = i + ((a - i % kTcABufs) + kTcABufs) % kTcABufs;  // first unit of this issuer
                for (; ib <= iend; ib += kTcABufs) {
                    const int l = kl + (ib - i);  // unit column within the group
                    const int xs = ib % kTcXRing;  // T = 32: ring slot of unit ib
                    if (kRing ? !mbar_wait_bounded(sXLoaded + 8 * xs, (ib / kTcXRing) & 1)
                              : !mbar_wait_bounded(sXFull + 8 * l, 0)) {
                        ok = false;
                        break;
                    }
                    const uint32_t xbase = kRing ? sX + xs * xslot : sX + l * xslot;
                    const uint32_t a_tmem = tbase + a * kTcAColsPerUnit;
                    const unsigned par = (ib / kTcABufs) & 1;
#pragma unroll
                    for (int part = p0; part < p0 + kTcPartsPerIssuer; ++part) {
                        // descriptors of the part's 64-k boxes: tokens 8-15 are the next
                        // atom (T == 32) or the zero block (T == 8)
                        constexpr int kBoxes = kTcStepsPerPart / 4;
                        uint64_t bd[kBoxes];
#pragma unroll
                        for (int h = 0; h < kBoxes; ++h) {
                            const uint32_t box = xbase + (uint32_t)(part * kBoxes + h) * xbox;
                            bd[h] = tc::smem_desc_sw128(box, (T == 32) ? 1024u : (sZero - box));
                        }
                        if (!mbar_wait_bounded(sAFull + 8 * (a * kTcAParts + part), par)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
#pragma unroll
                        for (int j = 0; j < kTcStepsPerPart; ++j) {
                            // k-step s = part * steps + j: box s/4, bytes 32*(s%4) into each
                            // 128-byte row (the start-address field counts 16-byte units and
                            // does not carry)
                            const int s = part * kTcStepsPerPart + j;
                            const uint64_t bdesc = bd[j >> 2] + (uint64_t)(2 * (j & 3));
                            tc::mma_f16_ts(d_tmem, a_tmem + s * 8, bdesc, idesc, !(first && part == p0 && j == 0));
                        }
                        tc::commit(sAEmpty + 8 * (a * kTcAParts + part));
                    }
                    if (!ok) break;
                    if (kRing) tc::commit(sXFull + 8 * xs);  // the X slot may be refilled once these MMAs are done
                    first = false;
                }
                // every issuer closes every segment, so the epilogue sees each phase
                tc::commit(sDFull + 8 * (w * 2 + sb));
                kl = 0;
                i = iend + 1;
            }
            if (!ok) atomicOr(p.err, kDevErrTimeoutFull);
            tc::commit(sFinal + 8 * w);
            if (!mbar_wait_bounded(sFinal + 8 * w, 0)) atomicOr(p.err, kDevErrTimeoutDrain);
        }
        __syncwarp();
    } else if (warp < kTcWarpEpilogue0) {
        // ------------------------------------------------------------ dequant
        // Two sets of four warps: set ab converts the units of A buffer ab
        // (i % 2 == ab), a warp (lane quarter lq) all 256 k of rows
        // 32 lq .. 32 lq + 31; each warp has two units' time for one.
        const int e = warp - kTcWarpDequant0;  // 0 .. kTcDequantWarps - 1
        const int lq = warp & 3;               // tensor-memory lane quarter this warp may access
        const int ab = e >> 2;                 // its A buffer: units i with i % kTcABufs == ab
        const int r = 32 * lq + lane;          // row within the unit
        const uint32_t lane_bits = (uint32_t)(32 * lq) << 16;
        const uint32_t w_row = (uint32_t)r * 128, w_sw = (uint32_t)(r & 7);
        const uint8_t *const s_row = base + (sS - sW) + r * 16;
        bool ok = true;
        int slot = ab % S;               // ring stage of unit i (advanced by kTcABufs per unit)
        uint32_t fpar = 0, apar = 1;     // parities to wait for: full[slot]; aempty from round 1 on
        for (int i = ab; i < count; i += kTcABufs) {
            if (__any_sync(0xffffffffu, !mbar_wait_bounded(sFull + 8 * slot, fpar))) {
                ok = false;
                break;
            }
            const uint32_t wst = sW + slot * kTcWBytes + w_row;
            uint4 wv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) wv[j] = lds128(wst + ((((uint32_t)j) ^ w_sw) << 4));
            const uint4 s16 = *reinterpret_cast<const uint4 *>(s_row + slot * kTcSBytes);
            __syncwarp();
            if (lane == 0) mbar_arrive(sEmpty + 8 * slot);  // the weight stage may be refilled
            slot += kTcABufs;
            if (slot >= S) {  // S is even: every set sees every other stage, each phase
                slot -= S;
                fpar ^= 1u;
            }
            const uint32_t svs[4] = {s16.x, s16.y, s16.z, s16.w};
#pragma unroll
            for (int part = 0; part < kTcAParts; ++part) {
                if (i >= kTcABufs &&
                    __any_sync(0xffffffffu, !mbar_wait_bounded(sAEmpty + 8 * (ab * kTcAParts + part), apar))) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();  // the tensor-memory stores below follow the MMAs that read this part
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {  // 64 k (32 columns) per store
                    const int h = part * 2 + h2;
                    const uint32_t s01 = e4m3x2_to_f16x2(svs[h]), s23 = e4m3x2_to_f16x2(svs[h] >> 16);
                    const uint32_t sc[4] = {dup_lo(s01), dup_hi(s01), dup_lo(s23), dup_hi(s23)};
                    const uint32_t words[8] = {wv[2 * h].x, wv[2 * h].y, wv[2 * h].z, wv[2 * h].w,
                                               wv[2 * h + 1].x, wv[2 * h + 1].y, wv[2 * h + 1].z, wv[2 * h + 1].w};
                    uint32_t v[32];
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        uint32_t f;
                        switch (q & 3) {
                            case 0: f = e2m1x2_to_f16x2<0>(words[q >> 2]); break;
                            case 1: f = e2m1x2_to_f16x2<1>(words[q >> 2]); break;
                            case 2: f = e2m1x2_to_f16x2<2>(words[q >> 2]); break;
                            default: f = e2m1x2_to_f16x2<3>(words[q >> 2]); break;
                        }
                        v[q] = hmul2_u32(f, sc[q >> 3]);  // column q holds k pair (2q, 2q+1); 8 columns per scale block
                    }
                    tc::st_32x32b_x32(tbase + lane_bits + ab * kTcAColsPerUnit + h * 32, v);
                }
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(sAFull + 8 * (ab * kTcAParts + part));
            }
            if (!ok) break;
            apar ^= 1u;  // the next unit of this buffer waits for the phase of this one
        }
        if (!ok && lane == 0) atomicOr(p.err, kDevErrTimeoutFull);
    } else {
        // ----------------------------------------------------------- epilogue
        const int lq = warp & 3;
        const uint32_t lane_bits = (uint32_t)(32 * lq) << 16;
        zero_x_pad(warp - kTcWarpEpilogue0);
        griddep_wait();  // X, the global scale, the workspace and Y belong to this call from here on
        if (!convert_x(warp - kTcWarpEpilogue0) && lane == 0) atomicOr(p.err, kDevErrTimeoutFull);
        const float gs = ld_dep_f32(p.gscale) * kTcXUnscale;
        (void)KC;
        int seg = 0, kl = kl0, rb = rb0;
        for (int i = 0; i < count; ++seg) {
            int iend = i + (kg - kl) - 1;
            if (iend > count - 1) iend = count - 1;
            const int kfirst = kl, klast = kl + (iend - i);
            const int sb = seg & 1;
            // segment `seg`: row block rb, unit columns [kfirst, klast] of the group
            bool ok = true;
#pragma unroll
            for (int q = 0; q < kTcIssuers; ++q) ok = ok && mbar_wait_bounded(sDFull + 8 * (q * 2 + sb), (seg >> 1) & 1);
            if (__any_sync(0xffffffffu, !ok)) {
                if (lane == 0) atomicOr(p.err, kDevErrTimeoutFull);
                break;
            }
            tc::fence_after_sync();
            const int len = iend - i + 1;
            const int row = rb * kUnitRows + 32 * lq + lane;
            const bool whole = G == 1 && kfirst == 0 && klast == kg - 1;
            float *const mine = p.partials + ((size_t)blockIdx.x * part.max_seg + (rb - rb0)) * tc_partial_floats(T) +
                                (size_t)(32 * lq + lane) * T;
#pragma unroll
            for (int c = 0; c < kAcc / 16; ++c) {  // 16 token columns at a time
                float v[16];
                bool have = false;
#pragma unroll
                for (int q = 0; q < kTcIssuers; ++q) {  // fixed order: issuer 0, 1, ...
                    const int qb = q / kTcIssuersPerBuf;  // the A buffer (unit residue) of issuer q
                    const bool contributed = len >= kTcABufs || ((qb - i % kTcABufs + kTcABufs) % kTcABufs) < len;
                    if (!contributed) continue;
                    uint32_t d[16];
                    tc::ld_32x32b_x16(tbase + lane_bits + kTcDCol + q * 2 * kAcc + sb * kAcc + c * 16, d);
                    tc::wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = have ? v[j] + __uint_as_float(d[j]) : __uint_as_float(d[j]);
                    have = true;
                }
                if (c == kAcc / 16 - 1) {  // every accumulator column of the segment is read
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sDEmpty + 8 * sb);
                }
                if (whole) {
                    tc_store_row(p, v, row, gs, 16 * c);  // the whole row block is this segment: finish it here
                } else {
                    // one part of a split row block: publish the fp32 tile (T tokens per row);
                    // the reduction kernel that follows sums the parts in CTA order
                    float4 *const dst = reinterpret_cast<float4 *>(mine + 16 * c);
                    const bool in = nvfp4_in_bounds(rb - rb0 >= 0 && rb - rb0 < part.max_seg, p.err);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (in && q < T / 4)
                            __stcg(dst + q, make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
                }
            }
            i = iend + 1;
            kl = 0;
            ++rb;
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kTcWarpIssuer0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tbase, kTcTmemCols);
    }
}

// Split row blocks: one CTA per row block, one thread per row.  The parts of
// row block rb are the unit ranges of CTAs [ca, cb] of every k-group, taken
// in CTA order; part (CTA c) sits in c's slot for rb (c's partial tiles are
// indexed by row block from its first one).  Each thread walks that list
// itself and fetches its row of 64 / T parts at a time into registers (all
// those loads in flight together: one memory round trip per chunk), then sums
// them in order.  No shared memory and at most kTcReduceRegs registers a
// thread, so a reduction CTA fits on an SM next to a GEMV CTA: it can be resident (and
// waiting) before the GEMV finishes, and it never keeps the next call's GEMV
// CTA off an SM.  Row blocks finished whole by the GEMV (a single part) are
// skipped.  Index arithmetic is 32-bit: the planner keeps row_blocks * KC *
// (grid + 1) below 2^32.
struct TcPartCursor {  // walks the parts of one row block in (group, CTA) order
    unsigned rb, g, c, cb, cs, cg, u, kg;
    int G, KC;
    __device__ void enter_group(const TcPartition &part) {
        int ks, kgi;
        tc_group((int)g, G, KC, &ks, &kgi);
        kg = (unsigned)kgi;
        cs = (unsigned)part.cstart[g];
        cg = (unsigned)part.cstart[g + 1] - cs;
        u = (unsigned)part.row_blocks * kg;
        c = ((rb * kg + 1) * cg - 1) / u;
        cb = ((rb * kg + kg) * cg - 1) / u;
    }
    __device__ unsigned parts_in_group() const { return cb - c + 1; }
    // slot of the current part, then advance; call at most the number of parts times
    __device__ int next(const TcPartition &part) {
        const unsigned rbf = (c * u / cg) / kg;  // that CTA's first row block
        const int slot = (int)((cs + c) * (unsigned)part.max_seg + (rb - rbf));
        if (++c > cb && (int)(g + 1) < G) {
            ++g;
            enter_group(part);
        }
        return slot;
    }
};

// One sweep of the reduction over a row block's parts: tokens h*TT .. h*TT+TT-1
// of this thread's row, 64 / TT parts' loads in flight at a time, summed in
// part order (CTA order, group-major), then stored.
template <int T, int TT>
__device__ __forceinline__ void tc_reduce_sweep(const StreamParams &p, const TcPartition &part, TcPartCursor cur,
                                                int np, int r, int row, int h) {
    constexpr int kChunk = 64 / TT;  // parts whose loads are in flight together
    constexpr int kQ = TT / 4;       // float4 per row of a part and sweep
    cur.g = 0;
    cur.enter_group(part);
    float acc[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) acc[t] = 0.f;
    for (int j0 = 0; j0 < np; j0 += kChunk) {
        float4 f[kChunk][kQ];
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
            if (j0 + j < np) {
                const int tile = cur.next(part);
                const float4 *src = reinterpret_cast<const float4 *>(
                    p.partials + (size_t)tile * tc_partial_floats(T) + (size_t)r * T + h * TT);
                const bool in = nvfp4_in_bounds(tile >= 0 && tile < p.ctas * part.max_seg, p.err);
#pragma unroll
                for (int q = 0; q < kQ; ++q) f[j][q] = in ? __ldcg(src + q) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
            if (j0 + j >= np) break;
#pragma unroll
            for (int q = 0; q < kQ; ++q) {
                // parts are summed in CTA order; the first one replaces the zeros
                const bool first = j0 + j == 0;
                acc[4 * q] = first ? f[j][q].x : acc[4 * q] + f[j][q].x;
                acc[4 * q + 1] = first ? f[j][q].y : acc[4 * q + 1] + f[j][q].y;
                acc[4 * q + 2] = first ? f[j][q].z : acc[4 * q + 2] + f[j][q].z;
                acc[4 * q + 3] = first ? f[j][q].w : acc[4 * q + 3] + f[j][q].w;
            }
        }
    }
    tc_store_row(p, acc, row, ld_dep_f32(p.gscale) * kTcXUnscale, h * TT);
}

template <int T>
__global__ void __maxnreg__(kTcReduceRegs) tc_reduce_kernel(const StreamParams p, const TcPartition part) {
    griddep_launch_dependents();
    constexpr int TT = T < 16 ? T : 16;  // tokens summed per sweep over the parts (T = 32: two sweeps)
    TcPartCursor cur;
    cur.rb = blockIdx.x;
    cur.G = part.groups;
    cur.KC = p.KC;
    int np = 0;
    for (cur.g = 0; (int)cur.g < cur.G; ++cur.g) {
        cur.enter_group(part);
        np += (int)cur.parts_in_group();
    }
    // Every CTA waits for the GEMV, also those with nothing to sum: this grid
    // must not complete before the GEMV does, since the next kernel on the
    // stream (possibly the next call, reading Y) waits only for this one.
    griddep_wait();
    if (np <= 1) return;  // finished whole by the GEMV
    const int r = threadIdx.x, row = (int)cur.rb * kUnitRows + r;
    if constexpr (T == 32) {
        tc_reduce_sweep<T, TT>(p, part, cur, np, r, row, 0);
        tc_reduce_sweep<T, TT>(p, part, cur, np, r, row, 1);
    } else {
        tc_reduce_sweep<T, TT>(p, part, cur, np, r, row, 0);
    }
}

// X of one pass as f16 x 2^-8 for the 32-token kernel (which stages no bf16):
// 8 elements (16 bytes) per thread and step; |x| >= 2^24 sets error bit 8.
__global__ void __launch_bounds__(256) tc_x16_kernel(const uint16_t *__restrict__ x, uint16_t *__restrict__ x16,
                                                     long long chunks, unsigned *err) {
    griddep_wait();  // X may be the output of the kernel ahead of this one
    griddep_launch_dependents();
    uint32_t bad = 0;
    for (long long c = (long long)blockIdx.x * 256 + threadIdx.x; c < chunks; c += (long long)gridDim.x * 256) {
        uint4 v = ld_dep_v4(reinterpret_cast<const uint4 *>(x) + c);
        v.x = bf16x2_to_f16x2_scaled(v.x, bad);
        v.y = bf16x2_to_f16x2_scaled(v.y, bad);
        v.z = bf16x2_to_f16x2_scaled(v.z, bad);
        v.w = bf16x2_to_f16x2_scaled(v.w, bad);
        reinterpret_cast<uint4 *>(x16)[c] = v;
    }
    if (bad) atomicOr(err, kDevErrXRange);
}

cudaError_t launch_tc_x16(const uint16_t *x, uint16_t *x16, int n, int K, unsigned *err, cudaStream_t stream) {
    const long long chunks = (long long)n * K / 8;
    long long blocks = (chunks + 255) / 256;
    if (blocks > 1024) blocks = 1024;
    if (blocks < 1) blocks = 1;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_x16_kernel, x, x16, chunks, err);
}

cudaError_t tc_set_smem_limit(int smem_optin) {
    cudaError_t e = cudaFuncSetAttribute(gemv_tc_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gemv_tc_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
}

cudaError_t launch_tc(const CUtensorMap &tw, const CUtensorMap &ts, const CUtensorMap &tx, const StreamParams &p,
                      const TcPartition &part, int T, int smem, cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ctas);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (T != 8 && T != 32) return cudaErrorInvalidValue;
    cudaError_t e = T == 32 ? cudaLaunchKernelEx(&cfg, gemv_tc_kernel<32>, tw, ts, tx, p, part)
                            : cudaLaunchKernelEx(&cfg, gemv_tc_kernel<8>, tw, ts, tx, p, part);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t rc = {};
    rc.gridDim = dim3(part.row_blocks);
    rc.blockDim = dim3(kUnitRows);
    rc.stream = stream;
    rc.attrs = attr;
    rc.numAttrs = 1;
    return T == 32 ? cudaLaunchKernelEx(&rc, tc_reduce_kernel<32>, p, part)
                   : cudaLaunchKernelEx(&rc, tc_reduce_kernel<8>, p, part);
}

}  // namespace nvfp4
