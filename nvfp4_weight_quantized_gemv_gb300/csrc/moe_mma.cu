// moe_mma.cu -- the grouped read-once NVFP4 expert GEMV (MoE decode) on
// tensor cores, for K % 256 == 0 (other K take moe_gemv.cu's SIMT kernel).
//
// Same operation as moe_gemv.cu (rustdoc of spark_model/layers/mod.rs,
// moe_grouped_decode_min_rows: the grouped arm reads each routed expert once,
// on tokens sorted by expert):
//
//     Y[j, r] = bf16( g_e * sum_k X[tok[j], k] * E2M1(W_e[r, k]) * E4M3(S_e[r, k/16]) )
//
// for every expert e and assignment j in [off[e], off[e+1]) (or the SwiGLU of
// the interleaved gate/up rows).
//
// Work split.  An item is (expert with tokens, block of item_rows W rows);
// the items, in expert order, are cut into equal contiguous ranges, one per
// CTA of a persistent grid (one CTA per SM; experts without tokens cost
// nothing).  One producer thread streams each item into a ring of `stages`
// shared-memory slots: the W rows as K/256 TMA boxes of 128 bytes x item_rows
// rows (128-byte swizzle, so that the fragment loads below hit distinct
// banks) and the scale rows with one bulk copy.  The consumer warps stage the
// expert's token rows of X as f16 x 2^-8 (row pitch padded by 64 bytes) when
// the expert changes, then compute with mma.sync.m16n8k16 (f16 in, fp32
// accumulate): warp (row group gi, k part kp) owns 16 W rows and a contiguous
// 1/kparts of the 32-k chunks; per chunk each lane converts the 4 k-pairs it
// needs for rows g and g+8 (E2M1 cvt times the E4M3 scale: exact in f16) and
// issues two MMAs per group of 8 tokens.  Within a chunk, lane quad q holds
// k = 8q..8q+7; the MMA's k index is a fixed permutation of those (the same
// for A and B), which the sum does not depend on.  k parts are summed in
// order through shared memory by the kp = 0 warp, which stores the outputs.
// Each output's sum therefore has a fixed order that does not depend on the
// other tokens routed to the expert.
//
// Bad routing data (an offset outside [0, A] or decreasing, a token index
// outside [0, n)) is skipped and sets bit 32 of the device error word; every
// wait is bounded (2 s), a timeout sets an error bit and the CTA winds down.
#include "internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace nvfp4 {

namespace {

constexpr unsigned kDevErrRoutingMma = 32u;
constexpr unsigned kDevErrXRangeMma = 8u;
constexpr int kMmaWarps = 8;                        // consumer warps
constexpr int kMmaThreads = (kMmaWarps + 1) * 32;   // + the producer warp
constexpr int kMmaConsumerThreads = kMmaWarps * 32;

__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled_moe(uint32_t w, uint32_t &bad) {
    const uint32_t m = w & 0x7FFF7FFFu;
    bad |= (m + 0x34803480u) & ~(m + 0x00800080u) & 0x80008000u;  // finite |x| >= 2^24
    __half2 h = __floats2half2_rn(__uint_as_float(w << 16) * (1.0f / 256.0f),
                                  __uint_as_float(w & 0xFFFF0000u) * (1.0f / 256.0f));
    return *reinterpret_cast<uint32_t *>(&h);
}

// One 32-bit word of packed codes (4 k-pairs) times its scale (f16, dup'ed).
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t sc2, uint32_t (&a)[4]) {
    a[0] = hmul2_u32(e2m1x2_to_f16x2<0>(w), sc2);
    a[1] = hmul2_u32(e2m1x2_to_f16x2<1>(w), sc2);
    a[2] = hmul2_u32(e2m1x2_to_f16x2<2>(w), sc2);
    a[3] = hmul2_u32(e2m1x2_to_f16x2<3>(w), sc2);
}

// Bytes 0 and 2 of `w` (two E4M3 scales) -> f16x2 {byte 0, byte 2}.
__device__ __forceinline__ uint32_t scales02_to_f16x2(uint32_t w) {
    return e4m3x2_to_f16x2(__byte_perm(w, 0u, 0x0020));
}

template <bool SWIGLU>
__global__ void __launch_bounds__(kMmaThreads, 1)
    moe_mma_kernel(const __grid_constant__ CUtensorMap tmap_w, const MoeParams p) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ __align__(8) unsigned long long bars[2 * kMoeMaxStages];
    __shared__ int act[kMoeMaxExperts + 1];  // active experts in order; act[kMoeMaxExperts] = their count
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;  // warp kMmaWarps: the producer
    const uint32_t base = (smem_u32(sm) + 1023u) & ~1023u;       // the ring's TMA boxes need 1024-byte alignment
    const int KC = p.K >> 8;                                      // 256-k boxes per row
    const int srow = p.K >> 4;                                    // scale bytes per row
    const int IR = p.item_rows, S = p.stages;
    const uint32_t box_bytes = (uint32_t)IR * 128;
    const uint32_t slot_bytes = ((uint32_t)KC * box_bytes + (uint32_t)IR * srow + 1023u) & ~1023u;
    const uint32_t ring = base;
    const uint32_t xs = ring + (uint32_t)S * slot_bytes;              // [tok_pass][x_pitch] f16 x 2^-8
    const uint32_t x_pitch = (uint32_t)p.K * 2 + 64;
    const uint32_t scratch = xs + (uint32_t)p.tok_pass * x_pitch;     // [2][kMmaWarps][2 groups][32 lanes][4] fp32
    const int items_per_expert = (p.N + IR - 1) / IR;
    const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[kMoeMaxStages]);

    // ---- active experts (every CTA derives the same list) and this CTA's items
    if (warp == 0) {
        int cnt = 0;
        bool bad_off = false;
        for (int e0 = 0; e0 < p.E; e0 += 32) {
            const int e = e0 + lane;
            bool on = false;
            if (e < p.E) {
                const int a0 = __ldg(p.off + e), a1 = __ldg(p.off + e + 1);
                if (a0 < 0 || a1 < a0 || a1 > p.A) bad_off = true;
                else on = a1 > a0;
            }
            const unsigned m = __ballot_sync(0xffffffffu, on);
            if (on) act[cnt + __popc(m & ((1u << lane) - 1u))] = e;
            cnt += __popc(m);
        }
        if (lane == 0) act[kMoeMaxExperts] = cnt;
        if (__any_sync(0xffffffffu, bad_off) && lane == 0 && blockIdx.x == 0) atomicOr(p.err, kDevErrRoutingMma);
    }
    if (threadIdx.x == 32) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, kMmaWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    const long long total = (long long)act[kMoeMaxExperts] * items_per_expert;
    const long long i0 = total * blockIdx.x / gridDim.x, i1 = total * (blockIdx.x + 1) / gridDim.x;
    const int count = (int)(i1 - i0);

    if (warp == kMmaWarps) {
        // --------------------------------------------------------- producer
        if (lane == 0 && count > 0) {
            prefetch_tensormap(&tmap_w);
            const uint64_t policy = l2_policy_evict_first();  // each expert block is read once
            int issued = 0;
            for (; issued < count; ++issued) {
                const int slot = issued % S;
                if (issued >= S && !mbar_wait_bounded(empty0 + 8 * slot, ((issued / S) - 1) & 1)) {
                    atomicOr(p.err, kDevErrTimeoutEmpty);
                    break;
                }
                const long long it = i0 + issued;
                const int e = act[(int)(it / items_per_expert)];
                const int wr0 = (int)(it % items_per_expert) * IR;
                const int rows = min(p.N - wr0, IR);
                const uint32_t dst = ring + (uint32_t)slot * slot_bytes;
                const uint32_t full = full0 + 8 * slot;
                // the boxes always move IR rows (past this expert: the next one's rows or zeros)
                mbar_arrive_expect_tx(full, (uint32_t)KC * box_bytes + (uint32_t)rows * srow);
                const int grow = e * p.N + wr0;  // row of the [E * N][K/2] tensor
                for (int b = 0; b < KC; ++b) tma_load_2d(dst + b * box_bytes, &tmap_w, b * 128, grow, full, policy);
                bulk_g2s(dst + KC * box_bytes, p.s + (size_t)grow * srow, (uint32_t)rows * srow, full, policy);
            }
            // wait (bounded) for the copies in flight before the warp leaves
            for (int i = issued > S ? issued - S : 0; i < issued; ++i)
                if (!mbar_wait_bounded(full0 + 8 * (i % S), (i / S) & 1)) {
                    atomicOr(p.err, kDevErrTimeoutDrain);
                    break;
                }
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const int ngroups = IR >> 4, kparts = kMmaWarps / ngroups;
    const int gi = warp % ngroups, kp = warp / ngroups;
    const int b0 = kp * KC / kparts, b1 = (kp + 1) * KC / kparts;  // this warp's 256-k boxes
    const int g = lane >> 2, q = lane & 3;
    const int r0 = gi * 16 + g;  // this lane's rows r0 and r0 + 8 of the item
    uint32_t bad = 0;
    bool ok = true;  // false after a timeout: no more waits or compute, same barrier steps
    int staged_e = -1, staged_j0 = -1, red = 0;
    for (int k = 0; k < count; ++k) {
        const long long it = i0 + k;
        const int e = act[(int)(it / items_per_expert)];
        const int wr0 = (int)(it % items_per_expert) * IR;
        const int rows = min(p.N - wr0, IR);
        const int a0 = __ldg(p.off + e), a1 = __ldg(p.off + e + 1);
        const float gs = __ldg(p.gs + e) * 256.0f;  // undoes the 2^-8 prescale of X
        const int slot = k % S;
        const uint32_t wsm = ring + (uint32_t)slot * slot_bytes;
        const uint32_t ssm = wsm + (uint32_t)KC * box_bytes;
        if (ok && __any_sync(0xffffffffu, !mbar_wait_bounded(full0 + 8 * slot, (k / S) & 1))) {
            if (lane == 0) atomicOr(p.err, kDevErrTimeoutFull);
            ok = false;
        }
        for (int j0 = a0; j0 < a1; j0 += p.tok_pass) {
            const int c = min(p.tok_pass, a1 - j0);
            if (staged_e != e || staged_j0 != j0) {
                // stage the pass's token rows of X as f16 x 2^-8 (16-byte chunks)
                named_barrier(1, kMmaConsumerThreads);  // every consumer is done with the previous rows
                const int row_chunks = p.K >> 3;
                for (int i = threadIdx.x; i < c * row_chunks; i += kMmaConsumerThreads) {
                    const int t = i / row_chunks, chk = i - t * row_chunks;
                    const int tok = __ldg(p.tok + j0 + t);
                    uint4 o = make_uint4(0, 0, 0, 0);
                    if (tok >= 0 && tok < p.ntok) {
                        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)tok * p.K) + chk);
                        o = make_uint4(bf16x2_to_f16x2_scaled_moe(v.x, bad), bf16x2_to_f16x2_scaled_moe(v.y, bad),
                                       bf16x2_to_f16x2_scaled_moe(v.z, bad), bf16x2_to_f16x2_scaled_moe(v.w, bad));
                    } else if (chk == 0) {
                        atomicOr(p.err, kDevErrRoutingMma);
                    }
                    sts128(xs + (uint32_t)t * x_pitch + (uint32_t)chk * 16, o);
                }
                named_barrier(1, kMmaConsumerThreads);
                staged_e = e;
                staged_j0 = j0;
            }
            const int ntg = (c + 7) >> 3;  // token groups of 8 (1 or 2)
            float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            if (ok) {
                // token rows this lane feeds to the MMA (rows past c are never stored)
                const int n0 = min(g, p.tok_pass - 1), n1 = min(8 + g, p.tok_pass - 1);
                const uint32_t xr0 = xs + (uint32_t)n0 * x_pitch + (uint32_t)q * 16;
                const uint32_t xr1 = xs + (uint32_t)n1 * x_pitch + (uint32_t)q * 16;
                const uint32_t sw = (uint32_t)(r0 & 7);  // 128-byte swizzle phase of rows r0 and r0 + 8
                const int hq = q >> 1;                   // lane quad q covers 16-k block 2 cb + hq of chunk cb
                for (int b = b0; b < b1; ++b) {
                    // the box's 16 scales of rows r0 and r0 + 8, shifted so that byte 2j + 16m of word m is block
                    // 2 (2m + j) + hq, i.e. the scale of chunk cb = 2m + j
                    uint4 sa = lds128(ssm + (uint32_t)r0 * srow + b * 16);
                    uint4 sb = lds128(ssm + (uint32_t)(r0 + 8) * srow + b * 16);
                    const uint32_t shv = 8u * (uint32_t)hq;
                    sa.x >>= shv; sa.y >>= shv; sa.z >>= shv; sa.w >>= shv;
                    sb.x >>= shv; sb.y >>= shv; sb.z >>= shv; sb.w >>= shv;
                    const uint32_t wbox = wsm + (uint32_t)b * box_bytes + q * 4;
                    const uint32_t xo0 = xr0 + (uint32_t)b * 512, xo1 = xr1 + (uint32_t)b * 512;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const uint32_t s2a = scales02_to_f16x2(m == 0 ? sa.x : m == 1 ? sa.y : m == 2 ? sa.z : sa.w);
                        const uint32_t s2b = scales02_to_f16x2(m == 0 ? sb.x : m == 1 ? sb.y : m == 2 ? sb.z : sb.w);
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const int cb = 2 * m + j;
                            const uint32_t woff = wbox + (((uint32_t)cb ^ sw) << 4);
                            const uint32_t wa = lds32(woff + (uint32_t)r0 * 128);
                            const uint32_t wb = lds32(woff + (uint32_t)(r0 + 8) * 128);
                            uint32_t aa[4], ab[4];
                            dequant_word(wa, j ? dup_hi(s2a) : dup_lo(s2a), aa);  // k 8q..8q+7: one scale block
                            dequant_word(wb, j ? dup_hi(s2b) : dup_lo(s2b), ab);
                            const uint4 x0 = lds128(xo0 + cb * 64);
                            mma_16816(d[0], aa[0], ab[0], aa[1], ab[1], x0.x, x0.y);
                            mma_16816(d[0], aa[2], ab[2], aa[3], ab[3], x0.z, x0.w);
                            if (ntg > 1) {
                                const uint4 x1 = lds128(xo1 + cb * 64);
                                mma_16816(d[1], aa[0], ab[0], aa[1], ab[1], x1.x, x1.y);
                                mma_16816(d[1], aa[2], ab[2], aa[3], ab[3], x1.z, x1.w);
                            }
                        }
                    }
                }
            }
            if (kparts > 1) {  // k parts summed in order by the kp = 0 warp of the group
                const uint32_t mine = scratch + ((uint32_t)((red & 1) * kMmaWarps + warp) * 2) * 512 + lane * 16;
                if (kp > 0) {
                    sts128(mine, make_uint4(__float_as_uint(d[0][0]), __float_as_uint(d[0][1]),
                                            __float_as_uint(d[0][2]), __float_as_uint(d[0][3])));
                    sts128(mine + 512, make_uint4(__float_as_uint(d[1][0]), __float_as_uint(d[1][1]),
                                                  __float_as_uint(d[1][2]), __float_as_uint(d[1][3])));
                }
                named_barrier(2, kMmaConsumerThreads);
                if (kp == 0) {
                    for (int o = 1; o < kparts; ++o) {
                        const uint32_t src =
                            scratch + ((uint32_t)((red & 1) * kMmaWarps + gi + o * ngroups) * 2) * 512 + lane * 16;
                        const uint4 v0 = lds128(src), v1 = lds128(src + 512);
                        d[0][0] += __uint_as_float(v0.x); d[0][1] += __uint_as_float(v0.y);
                        d[0][2] += __uint_as_float(v0.z); d[0][3] += __uint_as_float(v0.w);
                        d[1][0] += __uint_as_float(v1.x); d[1][1] += __uint_as_float(v1.y);
                        d[1][2] += __uint_as_float(v1.z); d[1][3] += __uint_as_float(v1.w);
                    }
                }
                ++red;
            }
            if (kp == 0 && ok) {
                // fragment: d[tg][0..1] = rows r0, tokens 8tg + 2q, +1; d[tg][2..3] = row r0 + 8
#pragma unroll
                for (int tg = 0; tg < 2; ++tg) {
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const int r = r0 + (h >> 1) * 8, t = 8 * tg + 2 * q + (h & 1);
                        const float v = d[tg][h] * gs;
                        if (!SWIGLU) {
                            if (t < c && r < rows) {
                                __nv_bfloat16 hv = __float2bfloat16_rn(v);
                                p.y[(size_t)(j0 + t) * p.N + wr0 + r] = *reinterpret_cast<uint16_t *>(&hv);
                            }
                        } else {
                            const float up = __shfl_down_sync(0xffffffffu, v, 4);  // row r + 1 sits in lane + 4
                            if ((g & 1) == 0 && t < c && r < rows) {
                                __nv_bfloat16 hv = __float2bfloat16_rn(v / (1.0f + expf(-v)) * up);
                                p.y[(size_t)(j0 + t) * (p.N / 2) + (wr0 + r) / 2] = *reinterpret_cast<uint16_t *>(&hv);
                            }
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * slot);  // this warp is done with the item's rows
    }
    if (bad) atomicOr(p.err, kDevErrXRangeMma);
}

}  // namespace

// Items of 128, 64, 32 or 16 W rows (16-row groups times k parts = 8 warps):
// the largest that leaves two ring slots beside 16 (else 8) staged tokens --
// fewer k parts mean fewer partial sums to exchange per item (measured on the
// 1536 x 2048 gate/up experts: 64 rows, 2 slots, 8 tokens 77 us per layer;
// 32 rows, 3-4 slots 90 us; 16 rows, 7 slots 122 us) -- else fewer staged
// tokens (deep K); false if even that does not fit.
bool moe_mma_plan(int N, int K, int smem_optin, int *item_rows, int *stages, int *tok_pass) {
    if (K % 256 != 0) return false;
    const int budget = smem_optin - kMoeMmaStaticSmem - 1024 - 2 * kMmaWarps * 2 * 512;
    auto fits = [&](int rows, int tok) {
        if (rows > N && rows > 16) return false;
        const int slot = ((K / 256) * rows * 128 + rows * (K / 16) + 1023) & ~1023;
        int st = (budget - tok * (K * 2 + 64)) / slot;
        if (st > kMoeMaxStages) st = kMoeMaxStages;
        if (st < 2) return false;
        *item_rows = rows;
        *stages = st;
        *tok_pass = tok;
        return true;
    };
    for (int rows = 128; rows >= 16; rows /= 2)
        for (int tok = 16; tok >= 8; tok /= 2)
            if (fits(rows, tok)) return true;
    for (int tok = 4; tok >= 1; tok /= 2)
        for (int rows = 128; rows >= 16; rows /= 2)
            if (fits(rows, tok)) return true;
    return false;
}

int moe_mma_smem_bytes(const MoeParams &p) {
    const int slot = ((p.K / 256) * p.item_rows * 128 + p.item_rows * (p.K / 16) + 1023) & ~1023;
    return 1024 + p.stages * slot + p.tok_pass * (p.K * 2 + 64) + 2 * kMmaWarps * 2 * 512;
}

cudaError_t moe_mma_set_smem_limit(int smem_optin) {
    const int dyn = smem_optin - kMoeMmaStaticSmem;
    cudaError_t e = cudaFuncSetAttribute(moe_mma_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(moe_mma_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
}

cudaError_t launch_moe_mma(const CUtensorMap &tw, const MoeParams &p, cudaStream_t stream) {
    const int smem = moe_mma_smem_bytes(p);
    if (p.swiglu)
        moe_mma_kernel<true><<<(unsigned)p.ctas, kMmaThreads, smem, stream>>>(tw, p);
    else
        moe_mma_kernel<false><<<(unsigned)p.ctas, kMmaThreads, smem, stream>>>(tw, p);
    return cudaGetLastError();
}

}  // namespace nvfp4
