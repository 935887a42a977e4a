// gemv_tc.cu -- the tcgen05 (5th-generation tensor core) NVFP4 batched GEMV.
//
// Computes Y[t, r] = g * sum_k X[t, k] * E2M1(W[r, k]) * E4M3(S[r, k/16]) for all
// n <= 16 tokens from ONE pass over W (atlas pull request #266, "What it
// does": each tile of decode tokens reads the projection weight once; here
// the tile is all n tokens).
//
// Work split: the weight matrix is cut into units of 128 rows x 256 k (128 B
// of every packed row + 16 scale bytes per row).  Units are ordered
// row-block-major and CTA c of the persistent grid owns units
// [c*U/C, (c+1)*U/C) ("stream-K"), so every SM moves the same bytes for any
// (N, K).  A row block whose units span several CTAs is finished by the last
// CTA to arrive, which sums the fp32 partial tiles in CTA order (fixed order:
// deterministic, and independent of n).
//
// Warp roles (576 threads, one CTA per SM):
//   warp 0       weight producer: 2D TMA loads of the unit's W tile
//                (128B-swizzled) and scale tile into a ring of S stages.
//   warps 1-4    MMA issuers, one per 64-k sub-unit of the unit (warp 1 also
//                owns the 512 tensor-memory columns): 4 x tcgen05.mma.kind::f16
//                per unit, M = 128 weight rows, N = 16 token columns, K = 16; A
//                from tensor memory, B (= X) from shared memory, fp32
//                accumulators in tensor memory per (row-block segment buffer,
//                issuer).  One issuing thread retires one such MMA only every
//                ~50 cycles, so four issuers share the work.
//   warp 5       X producer: one bulk copy per unit of its X slice.
//   warps 6-13   dequantise: thread = weight row; each warp owns a 32-row
//                quarter (its tensor-memory lane quarter) and one 128-k half;
//                E2M1 -> f16 (cvt) times the E4M3 block scale (exact), stored
//                with tcgen05.st.  A is handed to the issuers in 64-k
//                sub-units (12 tensor-memory buffers of 128 rows x 64 k), so
//                a buffer is held only for one sub-unit's dequant + MMAs.
//   warps 14-17  epilogue: per finished row-block segment, tcgen05.ld of the
//                four issuers' accumulators, summed in a fixed order, split
//                fixup, x g x 2^8, bf16 store -- off the streaming path.
//
// X: a small kernel that runs first (xconvert_kernel) converts X to f16
// (times 2^-8) in the canonical no-swizzle K-major layout of 8-token x 16-byte
// core matrices, one 256-k slice after another; the producer fetches each
// unit's slice (T tokens x 256 k, one bulk copy) into an X ring of its own
// (released when the unit's MMAs complete, so the weight stages are refilled
// as soon as the dequant warps have read them).  With
// n <= 8 only tokens 0-7 are kept and the MMA's tokens 8-15 read a 256-byte
// zero block.  The GEMV is launched with programmatic dependent launch: its
// weight stream starts at once and only the X copies wait for the conversion.
//
// X is scaled by 2^-8 before the f16 conversion (exact: a power of two), so
// |x| up to 65504 * 2^8 ~ 1.68e7 stays finite; larger entries set the device
// error word (the output is then not meaningful).  Every wait is bounded
// (2 s of %globaltimer); on a timeout the kernel sets the device error word,
// skips the remaining work, waits (bounded) for its own copies and MMAs, and
// frees its tensor memory before exiting.
#include "internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

#include <cuda_bf16.h>

namespace nvfp4 {

namespace {

constexpr int kTcUnitK = 256;                    // k per unit (128 packed bytes per row)
constexpr int kTcWBytes = kUnitRows * 128;       // 16384
constexpr int kTcSBytes = kUnitRows * 16;        // 2048
constexpr int kTcSubK = 64;                      // k per A sub-unit
constexpr int kTcSubs = kTcUnitK / kTcSubK;      // 4 sub-units per unit
constexpr int kTcASub = 12;                      // A sub-buffers of 32 columns (128 rows x 64 k)
constexpr int kTcAColsPerSub = kTcSubK / 2;      // 32 (two f16 per 32-bit column)
constexpr int kTcIssuers = kTcSubs;              // one MMA issuer per sub-unit
constexpr int kTcDCol = kTcASub * kTcAColsPerSub;  // 384: accumulators [segment buffer 2][issuer 4][16 cols]
constexpr int kTcXSlotsMax = 16;                 // X ring slots (bounded by shared memory)
constexpr uint32_t kTcTmemCols = 512;
constexpr int kTcWarpProducer = 0;
constexpr int kTcWarpIssuer0 = 1;                // issuers: warps 1..4
constexpr int kTcWarpXProducer = kTcWarpIssuer0 + kTcIssuers;  // 5
constexpr int kTcWarpDequant0 = kTcWarpXProducer + 1;         // dequant: warps 6..13
constexpr int kTcDequantWarps = 8;
constexpr int kTcWarpEpilogue0 = kTcWarpDequant0 + kTcDequantWarps;  // epilogue: warps 14..17
constexpr int kTcEpilogueWarps = 4;
constexpr int kTcThreads = (kTcWarpEpilogue0 + kTcEpilogueWarps) * 32;  // 576
constexpr float kTcXScale = 1.0f / 256.0f;       // 2^-8 applied to X before the f16 cast
constexpr float kTcXUnscale = 256.0f;
constexpr unsigned kDevErrXRange = 8u;           // some |x| >= 65520 * 2^8

// barriers: full[S] empty[S] xfull[SX] xempty[SX] afull[NA] aempty[NA] dfull[issuer][2] dempty[2] final[issuer]
__host__ __device__ constexpr int tc_barrier_count(int S, int SX) {
    return 2 * S + 2 * SX + 2 * kTcASub + 2 * kTcIssuers + 2 + kTcIssuers;
}

__device__ __forceinline__ int cta_of_unit_tc(long long u, long long U, int C) {
    return (int)(((u + 1) * (long long)C - 1) / U);
}

__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, bool &range) {
    const float lo = __uint_as_float(w << 16) * kTcXScale;
    const float hi = __uint_as_float(w & 0xFFFF0000u) * kTcXScale;
    range |= (fabsf(lo) >= 65520.f && isfinite(lo)) || (fabsf(hi) >= 65520.f && isfinite(hi));
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// X[t][k] (bf16, t < n) -> xf[k / 256] slice of T*256 f16: (t/8)*4096 + ((k%256)/8)*128 + (t%8)*16 + (k%8)*2
// bytes, times 2^-8; tokens n..T-1 are zero.  One thread per 8 consecutive k.
__global__ void __launch_bounds__(256) xconvert_kernel(const uint16_t *__restrict__ x, uint16_t *__restrict__ xf, int n,
                                                       int K, int T, unsigned *err) {
    griddep_launch_dependents();  // the GEMV may start its weight stream now
    const int groups = K >> 3;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= T * groups) return;
    const int t = i / groups, kb = i - t * groups;
    uint4 o = make_uint4(0, 0, 0, 0);
    bool range = false;
    if (t < n) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)t * K + (size_t)kb * 8));
        o = make_uint4(bf16x2_to_f16x2_scaled(v.x, range), bf16x2_to_f16x2_scaled(v.y, range),
                       bf16x2_to_f16x2_scaled(v.z, range), bf16x2_to_f16x2_scaled(v.w, range));
    }
    const size_t off = (size_t)(kb >> 5) * (T * 512) + (t >> 3) * 4096 + (kb & 31) * 128 + (t & 7) * 16;
    *reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(xf) + off) = o;
    if (range) atomicOr(err, kDevErrXRange);
}

}  // namespace

// X ring depth for a weight ring of `stages`: a few more slots than weight
// stages, because an X slot is held until its unit's MMAs complete.
__host__ __device__ int tc_xslots(int stages, int T) {
    const int sx = stages + 4;
    const int cap = T == 16 ? 10 : kTcXSlotsMax;
    return sx < cap ? sx : cap;
}

int tc_smem_bytes(int stages, int T, int K) {
    (void)K;
    const int xslot = T * 512;
    const int sx = tc_xslots(stages, T);
    return 1024 + stages * (kTcWBytes + kTcSBytes) + sx * xslot + 256 + 8 * tc_barrier_count(stages, sx) + 64;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    gemv_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_s,
                   const StreamParams p, const int T) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t sW = (raw_addr + 1023u) & ~1023u;
    uint8_t *const base = smem_raw + (sW - raw_addr);
    const int S = p.stages;
    const uint32_t xslot = (uint32_t)T * 512;           // one unit's X: T tokens x 256 k f16
    const uint32_t sS = sW + S * kTcWBytes;
    const int SX = tc_xslots(S, T);
    const uint32_t sX = sS + S * kTcSBytes;             // X slots [SX]
    const uint32_t sZero = sX + SX * xslot;             // 256 zero bytes
    const uint32_t sFull = sZero + 256;                 // W + scales of a stage landed
    const uint32_t sEmpty = sFull + 8 * S;              // dequant warps done with W + scales, count 8
    const uint32_t sXFull = sEmpty + 8 * S;             // X slot landed
    const uint32_t sXEmpty = sXFull + 8 * SX;           // all issuers' MMAs done with the X slot, count 4
    const uint32_t sAFull = sXEmpty + 8 * SX;           // [sub-buffer], count 4
    const uint32_t sAEmpty = sAFull + 8 * kTcASub;      // [sub-buffer], count 1 (commit)
    const uint32_t sDFull = sAEmpty + 8 * kTcASub;      // [issuer][dbuf], count 1 (commit)
    const uint32_t sDEmpty = sDFull + 16 * kTcIssuers;  // [dbuf], count 4 (epilogue warps)
    const uint32_t sFinal = sDEmpty + 16;               // [issuer], count 1 (commit)
    const uint32_t sMisc = sFinal + 8 * kTcIssuers;     // [0] tensor-memory base
    uint32_t *const misc = reinterpret_cast<uint32_t *>(base + (sMisc - sW));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KC = p.K / kTcUnitK;
    const long long u0 = (long long)blockIdx.x * p.units / p.ctas;
    const long long u1 = (long long)(blockIdx.x + 1) * p.units / p.ctas;
    const int count = (int)(u1 - u0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(sFull + 8 * s, 1);
            mbar_init(sEmpty + 8 * s, kTcDequantWarps);
        }
        for (int s = 0; s < SX; ++s) {
            mbar_init(sXFull + 8 * s, 1);
            mbar_init(sXEmpty + 8 * s, kTcIssuers);
        }
        for (int b = 0; b < kTcASub; ++b) {
            mbar_init(sAFull + 8 * b, kTcDequantWarps / 2);
            mbar_init(sAEmpty + 8 * b, 1);
        }
        for (int d = 0; d < 2 * kTcIssuers; ++d) mbar_init(sDFull + 8 * d, 1);
        for (int d = 0; d < 2; ++d) mbar_init(sDEmpty + 8 * d, kTcEpilogueWarps);
        for (int h = 0; h < kTcIssuers; ++h) mbar_init(sFinal + 8 * h, 1);
        fence_barrier_init();
    }
    if (warp == kTcWarpProducer && lane == 0) {
        prefetch_tensormap(&tmap_w);
        prefetch_tensormap(&tmap_s);
    }
    if (warp == kTcWarpIssuer0) {
        tc::tmem_alloc(sMisc, kTcTmemCols);
        tc::tmem_relinquish();
    }
    if (threadIdx.x < 16) sts128(sZero + threadIdx.x * 16, make_uint4(0, 0, 0, 0));
    fence_proxy_async_smem();  // the zero block is read by the tensor core
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = misc[0];

    if (warp == kTcWarpProducer) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            auto issue_w = [&](int i) {
                const long long u = u0 + i;
                const int rb = (int)(u / KC), kc = (int)(u - (long long)rb * KC);
                const int slot = i % S;
                const uint32_t full = sFull + 8 * slot;
                mbar_arrive_expect_tx(full, kTcWBytes + kTcSBytes);
                tma_load_2d(sW + slot * kTcWBytes, &tmap_w, kc * 128, rb * kUnitRows, full, policy);
                tma_load_2d(sS + slot * kTcSBytes, &tmap_s, kc * 16, rb * kUnitRows, full, policy);
            };
            const int first = count < S ? count : S;
            int issued = 0;
            for (; issued < first; ++issued) issue_w(issued);
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
    } else if (warp < kTcWarpXProducer) {
        // ---------------------------------------------------------- MMA issuers
        const int su = warp - kTcWarpIssuer0;  // the 64-k sub-unit of every unit this warp multiplies
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_f16_f32(kUnitRows, 16);
            // B descriptor of k-step 0 of the sub-unit; each further k-step moves
            // the start 256 bytes on (and, with T == 8, the stride offset to the
            // zero block 256 bytes back): a constant 64-bit delta.
            const uint64_t step = (T == 16) ? (uint64_t)16 : ((uint64_t)16 - ((uint64_t)16 << 32));
            int seg = -1;
            bool any = false;
            for (int i = 0; i < count; ++i) {
                const int kc = (int)((u0 + i) % KC);
                const int xs = i % SX;
                const int g = i * kTcSubs + su;  // global sub-unit sequence number
                const int sb = g % kTcASub;
                const bool seg_start = (i == 0 || kc == 0);
                if (seg_start) {
                    ++seg;
                    if (seg >= 2 && !mbar_wait_bounded(sDEmpty + 8 * (seg & 1), ((seg >> 1) - 1) & 1)) {
                        atomicOr(p.err, kDevErrTimeoutFull);
                        break;
                    }
                }
                if (!mbar_wait_bounded(sXFull + 8 * xs, (i / SX) & 1) ||
                    !mbar_wait_bounded(sAFull + 8 * sb, (g / kTcASub) & 1)) {
                    atomicOr(p.err, kDevErrTimeoutFull);
                    break;
                }
                tc::fence_after_sync();
                const uint32_t start = sX + xs * xslot + su * 1024;
                const uint64_t d0 = tc::smem_desc_noswizzle(start, 128, (T == 16) ? 4096u : (sZero - start));
                const uint32_t d_tmem = tbase + kTcDCol + (seg & 1) * 64 + su * 16;
                const uint32_t a_tmem = tbase + sb * kTcAColsPerSub;
#pragma unroll
                for (int s = 0; s < kTcSubK / 16; ++s)
                    tc::mma_f16_ts(d_tmem, a_tmem + s * 8, d0 + (uint64_t)s * step, idesc, !(seg_start && s == 0));
                tc::commit(sAEmpty + 8 * sb);
                tc::commit(sXEmpty + 8 * xs);
                if (kc == KC - 1 || i == count - 1) tc::commit(sDFull + 8 * (su * 2 + (seg & 1)));
                any = true;
            }
            if (any) {
                tc::commit(sFinal + 8 * su);
                if (!mbar_wait_bounded(sFinal + 8 * su, 0)) atomicOr(p.err, kDevErrTimeoutDrain);
            }
        }
        __syncwarp();
    } else if (warp == kTcWarpXProducer) {
        // ---------------------------------------------------------- X producer
        if (lane == 0) {
            auto issue_x = [&](int i) {
                const int kc = (int)((u0 + i) % KC), slot = i % SX;
                const uint32_t bar = sXFull + 8 * slot;
                mbar_arrive_expect_tx(bar, xslot);
                bulk_copy_g2s(sX + slot * xslot, reinterpret_cast<const uint8_t *>(p.xf16) + (size_t)kc * xslot, xslot,
                              bar);
            };
            griddep_wait();  // X is written by the conversion kernel that runs first
            int xissued = 0;
            for (; xissued < count; ++xissued) {
                if (xissued >= SX && !mbar_wait_bounded(sXEmpty + 8 * (xissued % SX), ((xissued / SX) - 1) & 1)) {
                    atomicOr(p.err, kDevErrTimeoutEmpty);
                    break;
                }
                issue_x(xissued);
            }
            const int lo = xissued > SX ? xissued - SX : 0;
            for (int i = lo; i < xissued; ++i) {
                if (!mbar_wait_bounded(sXFull + 8 * (i % SX), (i / SX) & 1)) {
                    atomicOr(p.err, kDevErrTimeoutDrain);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp < kTcWarpEpilogue0) {
        // ------------------------------------------------------------ dequant
        const int e = warp - kTcWarpDequant0;  // 0..7
        const int lq = warp & 3;               // tensor-memory lane quarter this warp may access
        const int kh = e >> 2;                 // which 128-k half of the unit
        const int r = 32 * lq + lane;          // row within the unit
        const uint32_t lane_bits = (uint32_t)(32 * lq) << 16;
        bool ok = true;
        for (int i = 0; i < count && ok; ++i) {
            const int slot = i % S;
            if (__any_sync(0xffffffffu, !mbar_wait_bounded(sFull + 8 * slot, (i / S) & 1))) {
                ok = false;
                break;
            }
            // 128 k of row r: 64 packed bytes in 4 swizzled 16-byte chunks, 8 scale bytes
            const uint32_t wrow = sW + slot * kTcWBytes + r * 128;
            const uint2 sv = *reinterpret_cast<const uint2 *>(base + (sS - sW) + slot * kTcSBytes + r * 16 + kh * 8);
            uint4 wv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) wv[j] = lds128(wrow + (uint32_t)(((kh * 4 + j) ^ (r & 7)) << 4));
            __syncwarp();
            if (lane == 0) mbar_arrive(sEmpty + 8 * slot);  // the weight stage may be refilled
            const uint32_t s01 = e4m3x2_to_f16x2(sv.x), s23 = e4m3x2_to_f16x2(sv.x >> 16);
            const uint32_t s45 = e4m3x2_to_f16x2(sv.y), s67 = e4m3x2_to_f16x2(sv.y >> 16);
            const uint32_t sc[8] = {dup_lo(s01), dup_hi(s01), dup_lo(s23), dup_hi(s23),
                                    dup_lo(s45), dup_hi(s45), dup_lo(s67), dup_hi(s67)};
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
                const int g = i * kTcSubs + kh * 2 + sub;
                const int sb = g % kTcASub;
                if (g >= kTcASub &&
                    __any_sync(0xffffffffu, !mbar_wait_bounded(sAEmpty + 8 * sb, ((g / kTcASub) - 1) & 1))) {
                    ok = false;
                    break;
                }
                const uint32_t a_col = tbase + lane_bits + sb * kTcAColsPerSub;
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int j = sub * 2 + jj;
                    const uint32_t words[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
                    uint32_t a[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        uint32_t f;
                        switch (q & 3) {
                            case 0: f = e2m1x2_to_f16x2<0>(words[q >> 2]); break;
                            case 1: f = e2m1x2_to_f16x2<1>(words[q >> 2]); break;
                            case 2: f = e2m1x2_to_f16x2<2>(words[q >> 2]); break;
                            default: f = e2m1x2_to_f16x2<3>(words[q >> 2]); break;
                        }
                        a[q] = hmul2_u32(f, sc[2 * j + (q >> 3)]);
                    }
                    tc::st_32x32b_x16(a_col + jj * 16, a);
                }
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(sAFull + 8 * sb);
            }
        }
        if (!ok && lane == 0) atomicOr(p.err, kDevErrTimeoutFull);
    } else {
        // ----------------------------------------------------------- epilogue
        const int lq = warp & 3;
        const uint32_t lane_bits = (uint32_t)(32 * lq) << 16;
        const float gs = __ldg(p.gscale) * kTcXUnscale;
        int seg = -1, kfirst = 0;
        for (int i = 0; i < count; ++i) {
            const long long u = u0 + i;
            const int rb = (int)(u / KC), kc = (int)(u - (long long)rb * KC);
            if (i == 0 || kc == 0) {
                ++seg;
                kfirst = kc;
            }
            if (!(kc == KC - 1 || i == count - 1)) continue;
            // segment `seg` of row block rb covers unit columns [kfirst, kc]
            bool ok = true;
#pragma unroll
            for (int q = 0; q < kTcIssuers; ++q)
                ok = ok && mbar_wait_bounded(sDFull + 8 * (q * 2 + (seg & 1)), (seg >> 1) & 1);
            if (__any_sync(0xffffffffu, !ok)) {
                if (lane == 0) atomicOr(p.err, kDevErrTimeoutFull);
                break;
            }
            tc::fence_after_sync();
            uint32_t d0[16], d1[16], d2[16], d3[16];
            const uint32_t dcol = tbase + lane_bits + kTcDCol + (seg & 1) * 64;
            tc::ld_32x32b_x16(dcol, d0);
            tc::ld_32x32b_x16(dcol + 16, d1);
            tc::ld_32x32b_x16(dcol + 32, d2);
            tc::ld_32x32b_x16(dcol + 48, d3);
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(sDEmpty + 8 * (seg & 1));
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)  // fixed order: sub-units 0, 1, 2, 3
                v[j] = ((__uint_as_float(d0[j]) + __uint_as_float(d1[j])) + __uint_as_float(d2[j])) +
                       __uint_as_float(d3[j]);

            const int row = rb * kUnitRows + 32 * lq + lane;
            if (!(kfirst == 0 && kc == KC - 1)) {
                // split row block: partial tile, last CTA to arrive sums in CTA order
                const long long ufirst = (long long)rb * KC;
                const int cfirst = cta_of_unit_tc(ufirst, p.units, p.ctas);
                const int clast = cta_of_unit_tc(ufirst + KC - 1, p.units, p.ctas);
                const int slot = ((int)blockIdx.x == cfirst) ? 1 : 0;
                const size_t tile = (size_t)kConsumerWarps * kSlotFloats;  // 2048 floats per (CTA, slot)
                float4 *mine = reinterpret_cast<float4 *>(p.partials + ((size_t)blockIdx.x * 2 + slot) * tile +
                                                          lq * 512 + lane * 16);
#pragma unroll
                for (int q = 0; q < 4; ++q) mine[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                __threadfence();
                __syncwarp();
                unsigned old = 0;
                if (lane == 0) old = atomicAdd(&p.counters[cfirst * kCountersPerCta + lq], 1u);
                old = __shfl_sync(0xffffffffu, old, 0);
                if (old != (unsigned)(clast - cfirst)) continue;  // another CTA finishes this row block
                __threadfence();
                for (int c = cfirst; c <= clast; ++c) {
                    const int sl = (c == cfirst) ? 1 : 0;
                    const float4 *src = reinterpret_cast<const float4 *>(p.partials + ((size_t)c * 2 + sl) * tile +
                                                                         lq * 512 + lane * 16);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 f = __ldcg(src + q);
                        if (c == cfirst) {
                            v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
                        } else {
                            v[4 * q] += f.x; v[4 * q + 1] += f.y; v[4 * q + 2] += f.z; v[4 * q + 3] += f.w;
                        }
                    }
                }
                if (lane == 0) atomicExch(&p.counters[cfirst * kCountersPerCta + lq], 0u);
            }
            if (row < p.N) {
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    if (t < p.n) {
                        __nv_bfloat16 h = __float2bfloat16_rn(v[t] * gs);
                        p.y[(size_t)t * p.N + row] = *reinterpret_cast<uint16_t *>(&h);
                    }
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kTcWarpIssuer0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tbase, kTcTmemCols);
    }
}

cudaError_t tc_set_smem_limit(int smem_optin) {
    return cudaFuncSetAttribute(gemv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
}

cudaError_t launch_tc(const CUtensorMap &tw, const CUtensorMap &ts, const StreamParams &p, int T, int smem,
                      cudaStream_t stream) {
    const int items = T * (p.K >> 3);
    xconvert_kernel<<<(items + 255) / 256, 256, 0, stream>>>(p.x, const_cast<uint16_t *>(p.xf16), p.n, p.K, T,
                                                             p.err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ctas);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_tc_kernel, tw, ts, p, T);
}

}  // namespace nvfp4
