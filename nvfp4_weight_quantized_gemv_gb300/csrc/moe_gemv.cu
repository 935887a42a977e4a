// moe_gemv.cu -- grouped read-once NVFP4 GEMV over routed experts (MoE decode).
//
// The grouped-GEMM MoE decode arm of the pages (rustdoc of
// spark_model/layers/mod.rs, moe_grouped_decode_min_rows: "reads each routed
// expert ONCE instead of once per token", with the tokens sorted by expert):
// for every expert e and every assignment j in [off[e], off[e+1]) of a token
// to that expert,
//
//     Y[j, r] = bf16( g_e * sum_k X[tok[j], k] * E2M1(W_e[r, k]) * E4M3(S_e[r, k/16]) )
//
// (or, with the SwiGLU option, h[j, f] = bf16(silu(Y[j, 2f]) * Y[j, 2f+1]) from
// the unrounded values, as nvfp4_gemv_swiglu).  Each CTA owns one expert and a
// block of its output rows: the block's packed rows and scales are contiguous
// and arrive in shared memory with two bulk copies (read once from HBM);
// meanwhile the expert's token rows of X are staged (f16 times 2^-8, as the
// tcgen05 path), up to 16 (8 with SwiGLU) per pass.  A warp per row: E2M1 ->
// f16 cvt times the E4M3 scale (exact), mixed f16 x f16 + f32 FMAs.  Each assignment's sum runs in a fixed order that does
// not depend on the other tokens routed to the expert, so a token's result is
// the same whether it shares its expert or not.
//
// Bad routing data (an offset outside [0, A] or decreasing, a token index
// outside [0, n)) cannot be checked before launch: the kernel skips it and
// sets bit 32 of the device error word.
#include "internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace nvfp4 {

namespace {

constexpr unsigned kDevErrRouting = 32u;  // bad expert offset or token index
constexpr unsigned kDevErrXRangeMoe = 8u;  // some |x| >= 2^24 (f16 overflow after the 2^-8 prescale)
constexpr int kMoeThreads = 256;          // 8 warps
constexpr int kMoeWarps = kMoeThreads / 32;
constexpr float kMoeXScale = 1.0f / 256.0f;

// f32 += f16 * f16 for both halves of two f16x2 registers (lo first).
__device__ __forceinline__ float fma2_f16(uint32_t w2, uint32_t x2, float acc) {
    float d;
    asm("{\n .reg .f16 wl, wh, xl, xh;\n .reg .f32 t;\n"
        " mov.b32 {wl, wh}, %1;\n mov.b32 {xl, xh}, %2;\n"
        " fma.rn.f32.f16 t, wl, xl, %3;\n fma.rn.f32.f16 %0, wh, xh, t;\n}\n"
        : "=f"(d)
        : "r"(w2), "r"(x2), "f"(acc));
    return d;
}

// Plain bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint32_t x_to_f16x2(uint32_t w, uint32_t &bad) {
    const uint32_t m = w & 0x7FFF7FFFu;
    bad |= (m + 0x34803480u) & ~(m + 0x00800080u) & 0x80008000u;  // finite |x| >= 2^24
    __half2 h = __floats2half2_rn(__uint_as_float(w << 16) * kMoeXScale, __uint_as_float(w & 0xFFFF0000u) * kMoeXScale);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Dot products of one W row held in shared memory with the staged tokens:
// lane covers 32 k per 16-byte chunk of the packed row, c <= TOK tokens;
// returns the warp-reduced sums (every lane holds all of them).  The order of
// the sum (lane-strided chunks, then a butterfly) does not depend on c.
template <int TOK>
__device__ __forceinline__ void moe_row(const uint8_t *wrow, const uint8_t *srow, const uint32_t *xs, int K, int c,
                                        int lane, float (&acc)[TOK]) {
#pragma unroll
    for (int t = 0; t < TOK; ++t) acc[t] = 0.f;
    const int chunks = K >> 5;
    const int xrow_words = K >> 1;
    for (int q = lane; q < chunks; q += 32) {
        const uint4 wv = *reinterpret_cast<const uint4 *>(wrow + q * 16);
        const uint32_t s01 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t *>(srow + q * 2));
        const uint32_t sc[2] = {dup_lo(s01), dup_hi(s01)};
        const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t w2[16];  // pair i: k = 32 q + 2i, 2i+1
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            uint32_t f;
            switch (i & 3) {
                case 0: f = e2m1x2_to_f16x2<0>(words[i >> 2]); break;
                case 1: f = e2m1x2_to_f16x2<1>(words[i >> 2]); break;
                case 2: f = e2m1x2_to_f16x2<2>(words[i >> 2]); break;
                default: f = e2m1x2_to_f16x2<3>(words[i >> 2]); break;
            }
            w2[i] = hmul2_u32(f, sc[i >> 3]);  // 8 pairs per 16-k scale block
        }
#pragma unroll
        for (int t = 0; t < TOK; ++t) {
            if (t < c) {
                const uint4 *xr = reinterpret_cast<const uint4 *>(xs + (size_t)t * xrow_words + q * 16);
                float a = acc[t];
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const uint4 xv = xr[v];
                    a = fma2_f16(w2[4 * v], xv.x, a);
                    a = fma2_f16(w2[4 * v + 1], xv.y, a);
                    a = fma2_f16(w2[4 * v + 2], xv.z, a);
                    a = fma2_f16(w2[4 * v + 3], xv.w, a);
                }
                acc[t] = a;
            }
        }
    }
#pragma unroll
    for (int t = 0; t < TOK; ++t) {
        float a = acc[t];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
        acc[t] = a;
    }
}

// This warp's rows of the block for the pass's c <= CB tokens (CB a
// compile-time bound on c): plain projection or gate/up with SwiGLU.
template <bool SWIGLU, int CB>
__device__ __forceinline__ void moe_rows(const MoeParams &p, const uint8_t *wsm, const uint8_t *ssm,
                                         const uint32_t *xs, int c, int j0, int orow0, int orows, float gs, int warp,
                                         int lane) {
    const int wrow_bytes = p.K / 2, srow_bytes = p.K / 16;
    const int out_rows = SWIGLU ? p.N / 2 : p.N;
    for (int r = warp; r < orows; r += kMoeWarps) {
        if (!SWIGLU) {
            float acc[CB];
            moe_row<CB>(wsm + (size_t)r * wrow_bytes, ssm + (size_t)r * srow_bytes, xs, p.K, c, lane, acc);
#pragma unroll
            for (int t = 0; t < CB; ++t) {
                if (t < c && lane == t) {
                    __nv_bfloat16 hv = __float2bfloat16_rn(acc[t] * gs);
                    p.y[(size_t)(j0 + t) * p.N + orow0 + r] = *reinterpret_cast<uint16_t *>(&hv);
                }
            }
        } else {
            float gate[CB], up[CB];
            moe_row<CB>(wsm + (size_t)(2 * r) * wrow_bytes, ssm + (size_t)(2 * r) * srow_bytes, xs, p.K, c, lane, gate);
            moe_row<CB>(wsm + (size_t)(2 * r + 1) * wrow_bytes, ssm + (size_t)(2 * r + 1) * srow_bytes, xs, p.K, c,
                        lane, up);
#pragma unroll
            for (int t = 0; t < CB; ++t) {
                if (t < c && lane == t) {
                    const float a = gate[t] * gs, u = up[t] * gs;
                    __nv_bfloat16 hv = __float2bfloat16_rn(a / (1.0f + expf(-a)) * u);
                    p.y[(size_t)(j0 + t) * out_rows + orow0 + r] = *reinterpret_cast<uint16_t *>(&hv);
                }
            }
        }
    }
}

// One CTA: expert e, a block of rows_per_cta output rows (W rows: twice as many
// with SwiGLU).  The block's packed rows and scales are contiguous in memory
// and arrive with two bulk copies, read once from HBM whatever the number of
// tokens; the tokens are staged TOK at a time.
template <bool SWIGLU>
__global__ void __launch_bounds__(kMoeThreads, 2) moe_gemv_kernel(const MoeParams p) {
    constexpr int TOK = SWIGLU ? 8 : 16;  // tokens per pass (register budget)
    extern __shared__ __align__(128) uint8_t sm[];
    __shared__ __align__(8) unsigned long long wbar;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int e = blockIdx.x / p.row_groups, rg = blockIdx.x % p.row_groups;
    const int a0 = __ldg(p.off + e), a1 = __ldg(p.off + e + 1);
    if (a0 < 0 || a1 < a0 || a1 > p.A) {
        if (threadIdx.x == 0) atomicOr(p.err, kDevErrRouting);
        return;
    }
    if (a0 == a1) return;  // no token routed to this expert
    const int wrows_per_cta = SWIGLU ? 2 * p.rows_per_cta : p.rows_per_cta;
    const int wr0 = rg * wrows_per_cta;                        // first W row of the block
    const int wrows = min(p.N - wr0, wrows_per_cta);           // W rows present (multiple of 16)
    const int wrow_bytes = p.K / 2, srow_bytes = p.K / 16;
    uint32_t *const xs = reinterpret_cast<uint32_t *>(sm);    // [TOK][K/2] f16x2
    uint8_t *const wsm = sm + (size_t)TOK * p.K * 2;          // [wrows][K/2]
    uint8_t *const ssm = wsm + (size_t)wrows_per_cta * wrow_bytes;  // [wrows][K/16]
    const uint32_t bar = smem_u32(&wbar);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
        const uint32_t wbytes = (uint32_t)wrows * wrow_bytes, sbytes = (uint32_t)wrows * srow_bytes;
        const uint64_t policy = l2_policy_evict_first();
        mbar_arrive_expect_tx(bar, wbytes + sbytes);
        bulk_copy_g2s(smem_u32(wsm), p.w + ((size_t)e * p.N + wr0) * wrow_bytes, wbytes, bar, policy);
        bulk_copy_g2s(smem_u32(ssm), p.s + ((size_t)e * p.N + wr0) * srow_bytes, sbytes, bar, policy);
    }
    const int out_rows = SWIGLU ? p.N / 2 : p.N;
    const int orow0 = rg * p.rows_per_cta;
    const int orows = min(out_rows - orow0, p.rows_per_cta);
    const float gs = __ldg(p.gs + e) * 256.0f;  // undoes the 2^-8 prescale of X
    uint32_t bad = 0;
    bool landed = false;
    for (int j0 = a0; j0 < a1; j0 += TOK) {
        const int c = min(TOK, a1 - j0);
        // stage the pass's token rows of X as f16 x 2^-8 (16-byte chunks)
        const int row_chunks = p.K >> 3;
        for (int i = threadIdx.x; i < c * row_chunks; i += kMoeThreads) {
            const int t = i / row_chunks, ch = i - t * row_chunks;
            const int tok = __ldg(p.tok + j0 + t);
            uint4 o = make_uint4(0, 0, 0, 0);
            if (tok >= 0 && tok < p.ntok) {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)tok * p.K) + ch);
                o = make_uint4(x_to_f16x2(v.x, bad), x_to_f16x2(v.y, bad), x_to_f16x2(v.z, bad), x_to_f16x2(v.w, bad));
            } else if (ch == 0) {
                atomicOr(p.err, kDevErrRouting);
            }
            reinterpret_cast<uint4 *>(xs)[(size_t)t * row_chunks + ch] = o;
        }
        __syncthreads();
        if (!landed) {  // the weight block (requested at entry) must be in shared memory
            if (!mbar_wait_bounded(bar, 0)) {
                if (threadIdx.x == 0) atomicOr(p.err, kDevErrTimeoutFull);
                return;
            }
            landed = true;
        }
        // the pass's token count, rounded up to a compile-time bound
        if (c <= 1) moe_rows<SWIGLU, 1>(p, wsm, ssm, xs, c, j0, orow0, orows, gs, warp, lane);
        else if (c <= 2) moe_rows<SWIGLU, 2>(p, wsm, ssm, xs, c, j0, orow0, orows, gs, warp, lane);
        else if (c <= 4) moe_rows<SWIGLU, 4>(p, wsm, ssm, xs, c, j0, orow0, orows, gs, warp, lane);
        else if (c <= 8) moe_rows<SWIGLU, 8>(p, wsm, ssm, xs, c, j0, orow0, orows, gs, warp, lane);
        else moe_rows<SWIGLU, SWIGLU ? 8 : 16>(p, wsm, ssm, xs, c, j0, orow0, orows, gs, warp, lane);
        __syncthreads();  // the next pass overwrites the staged rows
    }
    if (bad) atomicOr(p.err, kDevErrXRangeMoe);
}

}  // namespace

// Shared memory of one CTA: the staged tokens and the weight block.
int moe_smem_bytes(int K, int rows_per_cta, bool swiglu) {
    const int tok = swiglu ? 8 : 16, wrows = swiglu ? 2 * rows_per_cta : rows_per_cta;
    return tok * K * 2 + wrows * (K / 2 + K / 16);
}

// Output rows per CTA for K (multiple of 16, at most 128): preferably a block
// small enough for two CTAs per SM (one loads while the other computes) if
// that still holds 32 rows, else as many as fit one CTA; 0 if even 16 do not.
int moe_rows_per_cta(int K, bool swiglu, int smem_optin) {
    const int half = (smem_optin - 2048) / 2;
    for (int rows = 128; rows >= 32; rows -= 16)
        if (moe_smem_bytes(K, rows, swiglu) <= half) return rows;
    for (int rows = 128; rows >= 16; rows -= 16)
        if (moe_smem_bytes(K, rows, swiglu) <= smem_optin - 1024) return rows;
    return 0;
}

// The kernels also hold a little static shared memory (the barrier): leave
// 1 KB of the opt-in limit for it, as moe_rows_per_cta does.
cudaError_t moe_set_smem_limit(int smem_optin) {
    const int dyn = smem_optin - 1024;
    cudaError_t e = cudaFuncSetAttribute(moe_gemv_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(moe_gemv_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
}

cudaError_t launch_moe(const MoeParams &p, cudaStream_t stream) {
    const long long blocks = (long long)p.E * p.row_groups;
    const int smem = moe_smem_bytes(p.K, p.rows_per_cta, p.swiglu != 0);
    if (p.swiglu)
        moe_gemv_kernel<true><<<(unsigned)blocks, kMoeThreads, smem, stream>>>(p);
    else
        moe_gemv_kernel<false><<<(unsigned)blocks, kMoeThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace nvfp4
