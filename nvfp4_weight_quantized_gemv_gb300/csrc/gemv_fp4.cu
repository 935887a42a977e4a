// gemv_fp4.cu -- the block-scaled FP4 tensor-core path of the NVFP4 batched
// GEMV: the weights go from HBM to the tensor core as they are stored (E2M1
// codes plus one E4M3 scale per 16 k), with no dequantisation on CUDA cores.
//
// Computes Y[t, r] = g * sum_k X[t, k] * E2M1(W[r, k]) * E4M3(S[r, k/16]) for
// n <= 16 tokens from ONE pass over W (atlas pull request #266, "What it
// does": a tile of decode tokens reads the projection weight once; here the
// tile is all n tokens).
//
// The tensor core's block-scaled FP4 MMA (tcgen05.mma kind::mxf4nvf4,
// scale_vec::4X) multiplies E2M1 operands that each carry an E4M3 scale per
// 16 k -- exactly NVFP4 -- so the weight operand is the stored W tile and the
// weight scales are the stored S bytes.  The other operand must be NVFP4 too,
// so each bf16 activation row is written as a sum of J = 8 NVFP4 terms
// (fp4_xprep_kernel):
//
//     x[k] ~= sum_j s_j * b[k/16] * q_j[k],
//     s_0 = max|x| / (6 * 2^8),  s_j = s_{j-1} / 6,
//     b[i] = 2^e, the smallest power of two (2^-9 <= b <= 2^8, so UE4M3
//            holds it exactly) with 6 * s_0 * b >= max |x| over block i,
//
// q_j the E2M1 code (nearest, ties to even) of what the earlier terms left,
// r_j / (s_j b).  The grid's largest gap (4 to 6) is 2, so |r_{j+1}| <= s_j b
// = 6 s_{j+1} b: no term saturates, and after eight terms a block's residual
// is at most its own largest entry / 6^8 (1.5e-7 of it) -- relative to the
// block, not the row, for blocks down to 2^-17 of the row's largest; below
// that, at most 2^-17 max|x| / 6^8.  The tensor core applies b as the
// activation operand's block scale (the same byte for the token's eight
// terms); each term occupies its own MMA column (token t, term j -> column
// 8t + j) and the epilogue applies the s_j and sums a token's terms in a
// fixed order (the smallest first), multiplies by g and rounds to bf16.
// Every token's arithmetic is the same whatever n (the columns of an MMA are
// independent, the expansion is per token), so a batched call equals n
// single-token calls bit for bit.
//
// Work split.  Units of 128 rows x 256 k (one 16 KB W tile, 128-byte swizzle,
// plus the rows' 16 scale bytes); the persistent grid (one CTA per SM) takes
// equal contiguous ranges of the row-block-major unit order (stream-K over all
// of K).  A row block held whole by one CTA is finished there.  When the grid
// gives every row block p equal parts, the p CTAs of a row block run as one
// thread-block cluster and sum the parts through distributed shared memory
// after a cluster barrier, in CTA order.  Otherwise the parts of a split row
// block are written as fp32 tiles and the CTA that adds the last part (an
// atomic count per row block, or a look at it when the others are known to
// be in) sums them in CTA order and stores the row -- fixed order, no second
// launch, no waiting on other CTAs.  A CTA processes the partial row block at
// the end of its range first, so that its part is published early.
//
// Warp roles (384 threads):
//   warp 0     weight producer: TMA of the unit's W and S tiles into a ring of S
//              stages, at most `inflight` stages requested and not yet landed
//              (HBM stays busy without queueing in front of latency-bound
//              loads); the ring fills before the wait for the kernel ahead.
//   warp 10    X loader: after that wait, the X codes -- all unit columns
//              at once when they fit in shared memory, else one unit column
//              per stage.
//   warps 1,11 MMA issuers, units alternating (one issuer above 64 columns):
//              per unit four MMAs (K = 64 each, M = 128 weight rows, N = 8n
//              rounded up to 16 columns, fp32 in tensor memory) into the
//              issuer's accumulator of the row-block segment; the whole warp
//              runs the loop and one elected lane issues.
//   warps 2-5  scale-factor warps, one per tensor-memory lane quarter: the MMA
//              reads row m's four scale bytes of a K = 64 step from lane m,
//              column base + m / 32, and column n's from lane 32 q + n % 32,
//              column base + n / 32 in every quarter q (measured on sm_103a);
//              per unit a warp copies its rows' 16 S bytes and the unit
//              column's activation block scales with two tcgen05.st.
//   warps 6-9  epilogue: per finished row-block segment, tcgen05.ld of the
//              accumulators, the per-token sum of terms, then the bf16 store or
//              the split-row protocol above.
//
// Programmatic dependent launch: the X-prep kernel lets this grid launch at
// once; this grid streams weights before its griddepcontrol.wait and lets the
// next kernel (the next call's X prep) launch right after its setup.  X codes,
// the term scales, g, the workspace and Y are touched only after the wait.
// Every wait is bounded (2 s of %globaltimer); a timeout sets the device error
// word, skips the remaining work, waits (bounded) for the CTA's own copies and
// MMAs, and frees the tensor memory.
#include "internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

#include <cuda_bf16.h>

namespace nvfp4 {

namespace {

constexpr int kF4WBytes = kUnitRows * 128;      // 128 rows x 256 packed k
constexpr int kF4SBytes = kUnitRows * 16;       // 128 rows x 16 scale bytes
constexpr int kF4WarpProducer = 0;
constexpr int kF4WarpIssuer = 1;
constexpr int kF4WarpSf0 = 2;                   // warps 2..5
constexpr int kF4WarpEpi0 = 6;                  // warps 6..9
constexpr int kF4WarpXLoad = 10;                // X loader
constexpr int kF4WarpIssuer1 = 11;              // second MMA issuer (f4_issuers(cols) == 2)
constexpr int kF4Threads = 12 * 32;
constexpr uint32_t kF4TmemCols = 512;
constexpr int kF4SfCols = 32;                   // tensor-memory columns per stage: W scales 16, X scales 16
constexpr int kF4XprepThreads = 256;
constexpr int kF4XprepElems = kF4XprepThreads * 8;  // activations per X-prep CTA
constexpr unsigned kF4ErrSmemBase = 64u;            // dynamic shared memory not 1024-byte aligned

__device__ __forceinline__ void mma_fp4(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                        uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(
            d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// Instruction descriptor of kind::mxf4nvf4: A and B E2M1 (format 1 in bits
// [7,10) and [10,13)), both K-major, N >> 3 in [17,23), scale type E4M3 (bit
// 23 = 0), M >> 4 in [24,29), scale-factor ids 0, K = 64 (bit 31 = 0).
__host__ __device__ constexpr uint32_t idesc_fp4(int M, int N) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void bulk_load_f4(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                             uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// True in one lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n .reg .b32 r;\n .reg .pred p;\n elect.sync r|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(pred));
    return pred != 0;
}

__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier over `threads` threads that also ORs `v` over them: every
// participant gets the same answer (so a bounded wait that gave up in one warp
// makes all of them leave together and no named barrier is left unmatched).
__device__ __forceinline__ bool named_sync_or(int id, int threads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
        " bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

// Progress counters in shared memory, written with release and read with
// acquire semantics (CTA scope): cheaper than an mbarrier wait when the
// producer side is known to be ahead.
__device__ __forceinline__ void st_release_smem(uint32_t addr, uint32_t v) {
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_smem(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Count one published part: release (the CTA's partial-tile stores, ordered
// before by the named barrier) and acquire (the other parts, for the CTA that
// adds the last one) in one atomic.
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Non-blocking check of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint32_t bar, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// One row's outputs for all n tokens (v[t] = token t's sum of terms, before
// g): y = bf16(v g), or with swiglu the gated form of rows 2f / 2f + 1 held by
// lanes 2i / 2i + 1 (every lane of the warp must call it).
// The output side of the parameters (F4Params, or F4Out by value).
struct F4Out {
    uint16_t *y;
    int N, n, swiglu;
};
template <typename P>
__device__ __forceinline__ void f4_store_row(const P &p, const float (&v)[16], int row, float g) {
    const int lane = threadIdx.x & 31;
    if (!p.swiglu) {
        if (row < p.N) {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                if (t < p.n) {
                    __nv_bfloat16 h = __float2bfloat16_rn(v[t] * g);
                    p.y[(size_t)t * p.N + row] = *reinterpret_cast<uint16_t *>(&h);
                }
            }
        }
        return;
    }
    const int F = p.N >> 1;
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        const float a = v[t] * g;
        const float up = __shfl_down_sync(0xffffffffu, a, 1);
        if (t < p.n && (lane & 1) == 0 && row < p.N) {
            const float h = a / (1.0f + expf(-a)) * up;
            __nv_bfloat16 hv = __float2bfloat16_rn(h);
            p.y[(size_t)t * F + (row >> 1)] = *reinterpret_cast<uint16_t *>(&hv);
        }
    }
}

// Part c (a CTA) of split row block rb for this thread's row r.  A CTA's
// range of units splits at most its first and its last row block, so each CTA
// has two partial tiles: slot 0 for its first row block, slot 1 for its last.
__device__ __forceinline__ void f4_load_part(const F4Params &p, float (&part)[16], int c, int rb, int r,
                                             long long U, int KC) {
    const long long cu0 = (long long)c * U / p.ctas;
    const int crb0 = (int)(cu0 / KC);
    const float4 *src = reinterpret_cast<const float4 *>(p.partials + ((size_t)c * 2 + (rb == crb0 ? 0 : 1)) *
                                                                         (kUnitRows * 16) + (size_t)r * 16);
    const bool in = nvfp4_in_bounds(c >= 0 && c < p.ctas && r >= 0 && r < kUnitRows, p.err);
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
        if (in && 4 * qd < p.n) f = __ldcg(src + qd);
        part[4 * qd] = f.x;
        part[4 * qd + 1] = f.y;
        part[4 * qd + 2] = f.z;
        part[4 * qd + 3] = f.w;
    }
}

// Sum of the parts of split row block rb for this thread's row r, in CTA
// order ca..cb (fixed, so the result does not depend on which CTA adds it);
// part `self` is `own`, the others come from the partial tiles.  KQ float4 a
// row hold the call's tokens; the loads of up to 8 / KQ parts are in flight
// together (one memory round trip per batch).
template <int KQ>
__device__ __forceinline__ void f4_sum_parts(const F4Params &p, float (&sum)[16], int ca, int cb, int self,
                                             const float (&own)[16], int rb, int r, long long U, int KC) {
    constexpr int B = 8 / KQ;
    for (int c0 = ca; c0 <= cb; c0 += B) {
        float4 f[B][KQ];
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int c = c0 + j;
            if (c <= cb && c != self && nvfp4_in_bounds(c >= 0 && c < p.ctas, p.err)) {
                const long long cu0 = (long long)c * U / p.ctas;
                const int crb0 = (int)(cu0 / KC);
                const float4 *src = reinterpret_cast<const float4 *>(
                    p.partials + ((size_t)c * 2 + (rb == crb0 ? 0 : 1)) * (kUnitRows * 16) + (size_t)r * 16);
#pragma unroll
                for (int qd = 0; qd < KQ; ++qd) f[j][qd] = __ldcg(src + qd);
            }
        }
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int c = c0 + j;
            if (c > cb) break;
#pragma unroll
            for (int qd = 0; qd < KQ; ++qd) {
                const float4 v = c == self ? make_float4(own[4 * qd], own[4 * qd + 1], own[4 * qd + 2], own[4 * qd + 3])
                                           : f[j][qd];
                if (c == ca) {
                    sum[4 * qd] = v.x;
                    sum[4 * qd + 1] = v.y;
                    sum[4 * qd + 2] = v.z;
                    sum[4 * qd + 3] = v.w;
                } else {
                    sum[4 * qd] += v.x;
                    sum[4 * qd + 1] += v.y;
                    sum[4 * qd + 2] += v.z;
                    sum[4 * qd + 3] += v.w;
                }
            }
        }
    }
#pragma unroll
    for (int t = 4 * KQ; t < 16; ++t) sum[t] = 0.f;
}

// The cluster's sum of this thread's row over its `cl` parts, in rank order
// (the same order, and so the same rounding, as the workspace path's CTA
// order), stored: part `rank` (this CTA's own) at `own` in ring stage 0, the
// peers' parts in this CTA's receive area at `recv` + slot * `slot_stride`
// (slot = sender rank, less one above this CTA's rank).  Local shared-memory
// loads only: the peers pushed their parts before the cluster barrier.
template <int KQ>
__device__ __forceinline__ void f4_cluster_finish(const F4Out p, uint32_t own, uint32_t recv, uint32_t slot_stride,
                                                  int rank, int cl, int row, float g) {
    float sum[16];
    for (int k = 0; k < cl; ++k) {
        const uint32_t src = k == rank ? own : recv + (uint32_t)(k < rank ? k : k - 1) * slot_stride;
#pragma unroll
        for (int qd = 0; qd < KQ; ++qd) {
            const uint4 u = lds128(src + 16 * qd);
            const float4 v = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                                         __uint_as_float(u.w));
            if (k == 0) {
                sum[4 * qd] = v.x;
                sum[4 * qd + 1] = v.y;
                sum[4 * qd + 2] = v.z;
                sum[4 * qd + 3] = v.w;
            } else {
                sum[4 * qd] += v.x;
                sum[4 * qd + 1] += v.y;
                sum[4 * qd + 2] += v.z;
                sum[4 * qd + 3] += v.w;
            }
        }
    }
#pragma unroll
    for (int t = 4 * KQ; t < 16; ++t) sum[t] = 0.f;
    f4_store_row(p, sum, row, g);
}

// Eight fp32 values -> eight E2M1 codes, value j in nibble j (the hardware
// conversion puts its first operand in the high nibble).
__device__ __forceinline__ uint32_t f4_cvt_e2m1x8(const float (&q)[8]) {
    uint32_t out;
    asm("{\n"
        " .reg .b8 c0, c1, c2, c3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 c0, %2, %1;\n"
        " cvt.rn.satfinite.e2m1x2.f32 c1, %4, %3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 c2, %6, %5;\n"
        " cvt.rn.satfinite.e2m1x2.f32 c3, %8, %7;\n"
        " mov.b32 %0, {c0, c1, c2, c3};\n"
        "}\n"
        : "=r"(out)
        : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
    return out;
}

}  // namespace

// Shared memory: the ring (W + S tiles, plus the unit column's X codes when
// they are streamed), the resident X codes (all K / 256 unit columns) when not,
// the X block scales of all unit columns, the barriers, then flags and the
// term scales.
int f4_smem_bytes(int stages, int cols, bool x_resident, int KC, int cluster) {
    const int slot = f4_slot_bytes(cols), groups = (KC + kF4XGroup - 1) / kF4XGroup;
    const int xbars = x_resident ? (groups > stages ? groups : stages) : stages;
    const int tabs = (KC * f4_tab_bytes(cols) + 15) & ~15;
    return stages * (kF4XOffHost + (x_resident ? 0 : slot)) + (x_resident ? KC * slot : 0) + tabs +
           8 * (3 * stages + xbars + 9) + kF4MiscBytes + f4_red_bytes(cluster);
}

// TMEM: accumulators [issuer][segment buffer 2][f4_dstride(cols)] from column
// 0, then kF4SfCols per stage (W scales, then X block scales).
int f4_max_stages(int cols, int smem_limit, bool x_resident, int KC, int cluster) {
    const int tmem_stages = ((int)kF4TmemCols - 2 * f4_issuers(cols) * f4_dstride(cols)) / kF4SfCols;
    int s = 2;
    while (s + 1 <= tmem_stages && s + 1 <= kF4MaxStages &&
           f4_smem_bytes(s + 1, cols, x_resident, KC, cluster) <= smem_limit)
        ++s;
    return f4_smem_bytes(s, cols, x_resident, KC, cluster) <= smem_limit ? s : 0;
}

// ------------------------------------------------------------------ X prep
// The expansion of one token's activations, shared by the X-prep kernel and
// the GEMV's own prep (small n): the same arithmetic in both, so a token's
// codes and scales do not depend on which of them wrote them.

// Max |x| of bf16 values as bf16 magnitude bits (a uint32 max of the two halves).
__device__ __forceinline__ uint32_t f4_absmax_bits(const uint4 &v, uint32_t m) {
    m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.w & 0x7FFF7FFFu);
    return m;
}

// Term scales from the row's max |x| (bf16 magnitude bits; >= 0x7F80 is inf
// or NaN, and the token's outputs become NaN): s_0 = max|x| / (6 * 2^8),
// s_j = s_{j-1} / 6 (zero for an all-zero row); with them the reciprocals the
// expansion multiplies by, inv_j = (1 / s_0) 6^j (6^j is exact in fp32; inv_j
// is 1 / s_j to within a few ulp, which only moves the rare tie between two
// codes -- the residual is always taken with the exact s_j), and inv6 =
// (1 / s_0) / 6 for the block exponents.  Computed once per token.
struct F4TokenScales {
    float sc[kF4Terms], inv[kF4Terms], inv6;
};
__device__ __forceinline__ void f4_token_scales(uint32_t m, F4TokenScales &t) {
    t.sc[0] = m < 0x7F80u ? __fdiv_rn(__uint_as_float(m << 16), 6.0f * kF4BlockHeadroom) : __int_as_float(0x7FC00000);
#pragma unroll
    for (int j = 1; j < kF4Terms; ++j) t.sc[j] = __fdiv_rn(t.sc[j - 1], 6.0f);
    const float inv0 = t.sc[0] > 0.f ? __frcp_rn(t.sc[0]) : 0.f;
    float p6 = 1.0f;
#pragma unroll
    for (int j = 0; j < kF4Terms; ++j, p6 *= 6.0f) t.inv[j] = inv0 * p6;
    t.inv6 = inv0 * (1.0f / 6.0f);
}

// Eight consecutive activations (this lane) of a 16-element block whose other
// half the neighbouring lane (lane ^ 1) holds: the block exponent e and the
// eight terms' E2M1 codes (code word j = term j, value i in nibble i).  Every
// lane of the warp calls it.  The block scale b = 2^e is the smallest power of
// two with 6 s_0 b >= the block's max |x|, within UE4M3's powers of two 2^-9
// .. 2^8; rounding in the ratio can only pick the neighbouring power: a first
// code clamped at 6 (the later terms take the excess) or one bit of the first
// term unused.
__device__ __forceinline__ int f4_expand8(const uint4 &raw, const F4TokenScales &ts, bool finite,
                                          uint32_t (&codes)[kF4Terms]) {
    float r[8];
    {
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            r[2 * i] = __uint_as_float(w[i] << 16);
            r[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    float bmax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) bmax = fmaxf(bmax, fabsf(r[i]));
    bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 1));
    int e = -9;
    if (finite && ts.sc[0] > 0.f) {
        const float ratio = bmax * ts.inv6;
        const uint32_t u = __float_as_uint(ratio);
        const int E = (int)(u >> 23) - 127;  // ratio >= 0 and finite here; 0 or subnormal give E = -127
        if (ratio > 0.f) e = E + ((u & 0x7FFFFFu) != 0u ? 1 : 0);
        e = min(max(e, -9), 8);
    }
    const float b = __int_as_float((e + 127) << 23), binv = __int_as_float((127 - e) << 23);  // 2^e, 2^-e
#pragma unroll
    for (int j = 0; j < kF4Terms; ++j) {
        codes[j] = 0;
        const float sj = ts.sc[j] * b;  // exact: a power-of-two multiple
        if (finite && sj >= 1.17549435e-38f) {  // a subnormal scale's term is below any output's rounding
            const float inv = ts.sc[j] >= 1.17549435e-38f ? ts.inv[j] * binv : __frcp_rn(sj);
            float q[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) q[i] = r[i] * inv;
            codes[j] = f4_cvt_e2m1x8(q);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t h2 = e2m1x2_to_f16x2_rt(codes[j], i);
                const float2 d = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
                r[2 * i] = fmaf(-d.x, sj, r[2 * i]);
                r[2 * i + 1] = fmaf(-d.y, sj, r[2 * i + 1]);
            }
        }
    }
    return e;
}

// UE4M3 byte of 2^e (-9 <= e <= 8): subnormal below 2^-6.
__device__ __forceinline__ uint8_t f4_ue4m3_pow2(int e) { return (uint8_t)(e >= -6 ? (e + 7) << 3 : 1 << (e + 9)); }

// Byte offset of code word (column c, activations k0 .. k0 + 7) in a unit
// column's code tile: row c of 128 bytes, 16-byte chunks swizzled by c % 8.
__device__ __forceinline__ uint32_t f4_code_offset(int c, int k0) {
    const int bo = (k0 & 255) >> 1;
    return (uint32_t)(c * 128 + ((((bo >> 4) ^ (c & 7)) << 4) | (bo & 15)));
}

// Token t = blockIdx.y; this CTA expands activations [blockIdx.x * 2048,
// + 2048) of it.  Every CTA of a token reads the whole row once (all loads in
// flight together, one memory round trip) to find max |x| itself, so all of
// them derive the same term scales without exchanging anything.
template <int L>  // 16-byte loads per thread that cover a whole row: ceil(K / 2048) rounded up to 1, 2, 4, 8, 16
__global__ void __maxnreg__(64) fp4_xprep_kernel(const uint16_t *__restrict__ x, uint8_t *__restrict__ xq,
                                                 uint8_t *__restrict__ xtab, float *__restrict__ xs, int K,
                                                 int cols) {
    griddep_launch_dependents();  // the GEMV may launch and start streaming its weights
    griddep_wait();               // X may be the output of the kernel ahead of this one
    const int t = blockIdx.y, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)t * K);
    const int nvec = K / 8;  // <= L * 256
    const int own = blockIdx.x * kF4XprepThreads + tid;  // this thread's vector of this CTA's slice
    uint4 v[L];
#pragma unroll
    for (int j = 0; j < L; ++j) {
        const int i = tid + j * kF4XprepThreads;
        v[j] = i < nvec ? ld_dep_v4(xr + i) : make_uint4(0, 0, 0, 0);
    }
    const uint4 mine = own < nvec ? ld_dep_v4(xr + own) : make_uint4(0, 0, 0, 0);  // one of the above: same line
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < L; ++j) m = f4_absmax_bits(v[j], m);
    m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ uint32_t wmax[kF4XprepThreads / 32];
    if (lane == 0) wmax[wid] = m;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kF4XprepThreads / 32; ++w) m = max(m, wmax[w]);
    const bool finite = m < 0x7F80u;
    __shared__ F4TokenScales tok;  // the token's scales, computed once
    if (tid == 0) {
        f4_token_scales(m, tok);
        if (blockIdx.x == 0) {
#pragma unroll
            for (int j = 0; j < kF4Terms; ++j) xs[t * kF4Terms + j] = tok.sc[j];
        }
    }
    __syncthreads();
    const int k0 = own * 8;
    if (k0 >= K) return;  // whole warps: K / 8 is a multiple of 32
    uint32_t codes[kF4Terms];
    const int e = f4_expand8(mine, tok, finite, codes);
    const int kc = k0 >> 8;
    uint8_t *const tile = xq + (size_t)kc * f4_slot_bytes(cols);
#pragma unroll
    for (int j = 0; j < kF4Terms; ++j)  // MMA column of (token, term): row 8t + j of the unit column's code tile
        *reinterpret_cast<uint32_t *>(tile + f4_code_offset(t * kF4Terms + j, k0)) = codes[j];
    if ((own & 1) == 0) xtab[(size_t)kc * f4_tab_bytes(cols) + t * 16 + ((k0 & 255) >> 4)] = f4_ue4m3_pow2(e);
}

// Processing order of a CTA's units.  The CTA's range [u0, u0 + count) of the
// row-block-major order falls into `nseg` row-block segments (natural order);
// when the last one is partial (a split row block continued by the next CTA)
// it is processed first, so that this CTA's contribution to it is published
// early and whichever CTA completes that row block does not wait on it.
struct F4Order {
    int rb0, kc0, count, KC, nseg;
    bool rot;
    __device__ void init(long long u0, int cnt, int kc) {
        KC = kc;
        count = cnt;
        rb0 = (int)(u0 / KC);
        kc0 = (int)(u0 - (long long)rb0 * KC);
        nseg = cnt > 0 ? (int)((u0 + cnt - 1) / KC - u0 / KC + 1) : 0;
        rot = nseg >= 2 && seg_len(nseg - 1) < KC;
    }
    __device__ int nat(int s) const { return rot ? (s == 0 ? nseg - 1 : s - 1) : s; }   // natural index
    __device__ int seg_kc(int ns) const { return ns == 0 ? kc0 : 0; }                    // first unit column
    __device__ int seg_len(int ns) const {
        if (ns == 0) return min(KC - kc0, count);
        const int before = (KC - kc0) + (ns - 1) * KC;
        return min(KC, count - before);
    }
};

// Walks the units in processing order (row block, unit column) together with
// their ring stage and its phase parity; everything held in registers (no
// pointer to the order, no division per unit).
struct F4Walk {
    F4Order o;
    int s, ns, rb, kc, left;
    int st, S;          // ring stage of the current unit, ring size
    unsigned ph;        // parity of the stage's current phase
    __device__ void begin(const F4Order &ord, int stages) {
        o = ord;
        S = stages;
        s = 0;
        st = 0;
        ph = 0;
        if (o.nseg > 0) enter();
    }
    __device__ void enter() {
        ns = o.nat(s);
        rb = o.rb0 + ns;
        kc = o.seg_kc(ns);
        left = o.seg_len(ns);
    }
    __device__ void next() {  // advance by one unit
        ++kc;
        if (++st == S) {
            st = 0;
            ph ^= 1u;
        }
        if (--left == 0 && ++s < o.nseg) enter();
    }
};

// ------------------------------------------------------------------- GEMV
template <int NC>  // MMA columns: 16 * ceil(8 n / 16)
__global__ void __maxnreg__(128)
    gemv_fp4_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_s,
                    const F4Params p) {
    static_assert(NC % 16 == 0 && NC >= 16 && NC <= kF4MaxCols, "columns");
    constexpr int kDStride = NC <= 32 ? 32 : NC <= 64 ? 64 : 128;
    constexpr int kIssuers = NC <= 64 ? 2 : 1;  // units alternate between the issuers (own accumulators)
    constexpr uint32_t kSlot = 128u * NC;       // one unit column's X codes
    constexpr uint32_t kTab = 2u * NC;          // its block scales: NC / 8 tokens x 16 blocks
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t sbase = smem_u32(smem_raw);
    if (sbase & 1023u) {  // the swizzled tiles need a 1024-byte aligned base; never expected
        griddep_wait();
        if (threadIdx.x == 0) atomicOr(p.err, kF4ErrSmemBase);
        if (p.cluster) {  // every CTA of the cluster takes this path (same layout): the cluster phase
            __syncwarp();
            cluster_arrive();
            cluster_wait();
        }
        return;
    }
    const int S = p.stages;
    const int KC = p.KC;
    const bool xres = p.x_resident != 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- this CTA's unit range and the order it processes them in
    const long long U = (long long)p.row_blocks * KC;
    const long long u0 = (long long)blockIdx.x * U / p.ctas;
    const int count = (int)((long long)(blockIdx.x + 1) * U / p.ctas - u0);
    F4Order ord;
    ord.init(u0, count, KC);

    // ---- shared memory: ring stages [W 16 KB][S 2 KB]([X slot] when streamed),
    // resident X slots [KC] when not, the X block scales ([S] or [KC]), then
    // the barriers
    const uint32_t kStage = kF4XOffHost + (xres ? 0u : kSlot);
    const uint32_t sX = sbase + S * kStage;                  // resident X codes
    const uint32_t sTab = sX + (xres ? KC * kSlot : 0u);     // X block scales of every unit column
    const int xgroups = (KC + kF4XGroup - 1) / kF4XGroup;    // bulk copies of resident X codes
    const int xbars = xres ? (xgroups > S ? xgroups : S) : S;
    const uint32_t sFull = sTab + ((KC * kTab + 15u) & ~15u);  // [S] W + S landed (TMA)
    const uint32_t sXFull = sFull + 8 * S;      // [S] X codes of the stage landed / [xgroups] resident groups landed
    const uint32_t sSf = sXFull + 8 * xbars;    // [S] weight scales in tensor memory, count 4
    const uint32_t sEmpty = sSf + 8 * S;        // [S] MMAs done with the stage (commit)
    const uint32_t sDFull = sEmpty + 8 * S;     // [issuer][2] segment accumulated (commit)
    const uint32_t sDEmpty = sDFull + 32;       // [2] accumulators read, count 4
    const uint32_t sFinal = sDEmpty + 16;       // [issuer] every MMA done (commit)
    const uint32_t sTabFull = sFinal + 16;      // the X block scales landed
    const uint32_t sMisc = sTabFull + 8;        // [0] tensor-memory base, [1] last-part flag, [2] preload flag,
                                                // [4 + q] units whose weight scales quarter q has stored
    uint32_t *const misc = reinterpret_cast<uint32_t *>(smem_raw + (sMisc - sbase));
    const uint32_t sSfDone = sMisc + 16;
    float *const tscale = reinterpret_cast<float *>(misc + 8);  // [16][kF4Terms] the tokens' term scales
    // X codes of the unit with unit column kc in stage st
    auto x_addr = [&](int st, int kc) -> uint32_t {
        return xres ? sX + (uint32_t)kc * kSlot : sbase + (uint32_t)st * kStage + kF4XOffHost;
    };

    // Weights are read once per call: evict-first, unless another pass over
    // the same weights follows (n > 16), which keeps them in L2.
    const uint64_t w_policy = p.w_keep ? l2_policy_evict_last() : l2_policy_evict_first();
    F4Walk wk{};  // the producer's walk
    auto issue_w = [&]() {
        const uint32_t stage = sbase + wk.st * kStage, full = sFull + 8 * wk.st;
        mbar_arrive_expect_tx(full, kF4WBytes + kF4SBytes);
        tma_load_2d(stage, &tmap_w, wk.kc * 128, wk.rb * kUnitRows, full, w_policy);
        tma_load_2d(stage + kF4WBytes, &tmap_s, wk.kc * 16, wk.rb * kUnitRows, full, w_policy);
        wk.next();
    };
    // The weight stream: at most `inflight` stages requested and not yet
    // landed, so that HBM stays busy without queueing so much in front of the
    // latency-bound loads (X, partial tiles) that they wait microseconds.
    const int inflight = p.inflight < S ? p.inflight : S;
    const int pre = count < inflight ? count : inflight;
    int issued = 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(sFull + 8 * s, 1);
            mbar_init(sSf + 8 * s, 4);
            mbar_init(sEmpty + 8 * s, 1);
        }
        for (int s = 0; s < xbars; ++s) mbar_init(sXFull + 8 * s, 1);
        for (int b = 0; b < 4; ++b) mbar_init(sDFull + 8 * b, 1);
        for (int b = 0; b < 2; ++b) mbar_init(sDEmpty + 8 * b, 4);
        for (int b = 0; b < 2; ++b) mbar_init(sFinal + 8 * b, 1);
        mbar_init(sTabFull, 1);
        for (int q = 0; q < 4; ++q) misc[4 + q] = 0;
        fence_barrier_init();
        if (count > 0) wk.begin(ord, S);
        for (; issued < pre; ++issued) issue_w();
    }
    if (warp == kF4WarpIssuer) {
        tc::tmem_alloc(sMisc, kF4TmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = misc[0];
    // the next kernel on the stream (the next call's X prep) may launch now
    if (threadIdx.x == 0) griddep_launch_dependents();
    // per stage kF4SfCols columns: the W scales (16), then the X block scales (16)
    const uint32_t sf_base = tbase + 2 * kIssuers * kDStride;

    // Split row blocks summed in a cluster (p.cluster = p CTAs per row block,
    // one segment each): the rows of epilogue warp q are summed by the CTA of
    // rank q % p.  Each CTA's epilogue leaves its part of its own rows in
    // ring stage 0 (free once the segment's MMAs are done) and pushes its part
    // of the other rows into their CTA's receive area (distributed shared
    // memory stores); after one cluster barrier every CTA sums its rows over
    // the p parts in rank (= CTA) order from its own shared memory and stores
    // them.  (Measured on GB300: the hardware cluster barrier beat remote
    // mbarrier arrivals here by ~1.2 us per call.)
    const int cl = p.cluster;
    const uint32_t sRed = sbase;  // [128 rows][16] fp32, a row's tokens in 64 bytes
    const uint32_t sRecv = (sMisc + kF4MiscBytes + 15u) & ~15u;  // the peers' parts ([cl - 1][red_rows][16] fp32)
    const int red_rows = cl ? 32 * ((4 + cl - 1) / cl) : 0;
    bool red_pending = false;
    int red_row = 0;
    float g_ep = 0.f;

    if (warp == kF4WarpProducer) {
        // ---------------------------------------------------- weight producer
        if (lane == 0) {
            int lst = 0;       // stage of unit issued - inflight, whose landing paces the stream
            unsigned lph = 0;  // and its parity
            for (; issued < count; ++issued) {
                if ((issued >= S && !mbar_wait_bounded(sEmpty + 8 * wk.st, wk.ph ^ 1u)) ||
                    !mbar_wait_bounded(sFull + 8 * lst, lph)) {
                    atomicOr(p.err, kDevErrTimeoutEmpty);
                    break;
                }
                issue_w();
                if (++lst == S) {
                    lst = 0;
                    lph ^= 1u;
                }
            }
            // wait (bounded) for the most recent copies into every stage before exiting
            const int lo = issued > S ? issued - S : 0;
            for (int i = lo; i < issued; ++i) {
                if (!mbar_wait_bounded(sFull + 8 * (i % S), (i / S) & 1)) {
                    atomicOr(p.err, kDevErrTimeoutDrain);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp == kF4WarpXLoad) {
        // ----------------------------------------------------------- X loader
        if (lane == 0 && count > 0) {
            griddep_wait();  // the X codes are the output of the X-prep kernel ahead
            const uint64_t x_policy = l2_policy_evict_last();  // every CTA reads the same X codes
            // every unit column's block scales first: the scale-factor warps need only these
            mbar_arrive_expect_tx(sTabFull, KC * kTab);
            bulk_load_f4(sTab, p.xtab, KC * kTab, sTabFull, x_policy);
            if (xres) {
                // every unit column's X codes, kF4XGroup columns per bulk copy
                for (int g = 0; g < xgroups; ++g) {
                    const int c0 = g * kF4XGroup, nc = KC - c0 < kF4XGroup ? KC - c0 : kF4XGroup;
                    const uint32_t bytes = (uint32_t)nc * kSlot, bar = sXFull + 8 * g;
                    mbar_arrive_expect_tx(bar, bytes);
                    bulk_load_f4(sX + (uint32_t)c0 * kSlot, p.xq + (size_t)c0 * kSlot, bytes, bar, x_policy);
                }
                for (int g = 0; g < xgroups; ++g) {
                    if (!mbar_wait_bounded(sXFull + 8 * g, 0)) {
                        atomicOr(p.err, kDevErrTimeoutDrain);
                        break;
                    }
                }
            } else {
                F4Walk xw;
                xw.begin(ord, S);
                int loaded = 0;
                for (; loaded < count; ++loaded) {
                    if (loaded >= S && !mbar_wait_bounded(sEmpty + 8 * xw.st, xw.ph ^ 1u)) {
                        atomicOr(p.err, kDevErrTimeoutEmpty);
                        break;
                    }
                    const uint32_t bar = sXFull + 8 * xw.st;
                    mbar_arrive_expect_tx(bar, kSlot);
                    bulk_load_f4(sbase + xw.st * kStage + kF4XOffHost, p.xq + (size_t)xw.kc * kSlot, kSlot, bar,
                                 x_policy);
                    xw.next();
                }
                const int lo = loaded > S ? loaded - S : 0;
                for (int i = lo; i < loaded; ++i) {
                    if (!mbar_wait_bounded(sXFull + 8 * (i % S), (i / S) & 1)) {
                        atomicOr(p.err, kDevErrTimeoutDrain);
                        break;
                    }
                }
            }
            if (!mbar_wait_bounded(sTabFull, 0)) atomicOr(p.err, kDevErrTimeoutDrain);
        }
        __syncwarp();
    } else if (warp == kF4WarpIssuer || (kIssuers == 2 && warp == kF4WarpIssuer1)) {
        // ------------------------------------------------------------- issuers
        // Issuer j takes the units i with i % kIssuers == j, into its own
        // accumulator per segment buffer.  The whole warp runs the loop (the
        // descriptors stay warp-uniform) and one elected lane issues: much
        // cheaper per MMA than a single lane on its own.
        const int j = warp == kF4WarpIssuer ? 0 : 1;
        constexpr uint32_t idesc = idesc_fp4(kUnitRows, NC);
        // descriptors at shared address 0; the operand's address goes into the
        // start field (bits [0, 14), 16-byte units; no carry below 256 KB)
        const uint64_t desc0 = tc::smem_desc_sw128(0, 1024);
        bool ok = true;
        int mine = 0;          // the current unit's issuer (units alternate)
        int i = 0;             // the current unit's index in processing order
        int sf_known = 0;      // units whose weight scales are known to be in tensor memory
        uint32_t xg_ready = 0; // resident X code groups known to have landed (bit per group)
        F4Walk iw;
        if (count > 0) iw.begin(ord, S);
        for (int s = 0; s < ord.nseg && ok; ++s) {
            const int len = iw.left;
            const int sb = s & 1;
            if (s >= 2 && __any_sync(0xffffffffu, !mbar_wait_bounded(sDEmpty + 8 * sb, ((s >> 1) - 1) & 1))) {
                ok = false;
                break;
            }
            const uint32_t d_tmem = tbase + (j * 2 + sb) * kDStride;
            bool first = true;
            for (int u = 0; u < len; ++u, ++i, iw.next(), mine = kIssuers == 2 ? mine ^ 1 : 0) {
                if (mine != j) continue;
                const int st = iw.st;
                // the unit's weight scales: the scale-factor warps run ahead, so
                // their progress counters usually say so without a wait
                bool good = true;
                if (sf_known <= i) {
                    uint32_t lo = ld_acquire_smem(sSfDone);
#pragma unroll
                    for (int q = 1; q < 4; ++q) lo = min(lo, ld_acquire_smem(sSfDone + 4 * q));
                    sf_known = (int)lo;
                    if (sf_known <= i) good = mbar_wait_bounded(sSf + 8 * st, iw.ph);
                }
                // the unit's X codes: resident ones are waited for once per group
                if (xres) {
                    const int xg = iw.kc / kF4XGroup;
                    if (!((xg_ready >> xg) & 1u)) {
                        good = good && mbar_wait_bounded(sXFull + 8 * xg, 0);
                        xg_ready |= 1u << xg;
                    }
                } else {
                    good = good && mbar_wait_bounded(sXFull + 8 * st, iw.ph);
                }
                if (__any_sync(0xffffffffu, !good)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint64_t ad = desc0 + ((sbase + st * kStage) >> 4), bd = desc0 + (x_addr(st, iw.kc) >> 4);
                const uint32_t sfa = sf_base + st * kF4SfCols, sfb = sfa + 16;
                __syncwarp();
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_fp4(d_tmem, ad + 2 * k, bd + 2 * k, idesc, sfa + 4 * k, sfb + 4 * k,
                                (!first || k > 0) ? 1u : 0u);
                    tc::commit(sEmpty + 8 * st);
                }
                __syncwarp();
                first = false;
            }
            // every segment is closed by both issuers, so the epilogue sees each phase
            if (elect_one()) tc::commit(sDFull + 8 * (j * 2 + sb));
            __syncwarp();
        }
        if (lane == 0) {
            if (!ok) atomicOr(p.err, kDevErrTimeoutFull);
            tc::commit(sFinal + 8 * j);
            if (!mbar_wait_bounded(sFinal + 8 * j, 0)) atomicOr(p.err, kDevErrTimeoutDrain);
        }
        __syncwarp();
    } else if (warp >= kF4WarpSf0 && warp < kF4WarpEpi0) {
        // ------------------------------------------------- scale-factor warps
        // Lane quarter q: rows 32q + lane.  Per stage, kF4SfCols columns.  W
        // scales: the MMA of step s reads column 4s + q for its quarter-q rows,
        // so every column of the group gets the word.  X block scales: the MMA
        // of step s reads column 16 + 4s + n / 32 at lane n % 32 of every
        // quarter for token-term column n; the word is the four block bytes of
        // the step for the column's token (the same for its eight terms).
        const int q = warp & 3;
        const uint32_t lane_bits = (uint32_t)(32 * q) << 16;
        const int r = 32 * q + lane;
        bool ok = true;
        if (count > 0)  // every unit column's block scales, once
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(sTabFull, 0));
        // one unit's two stores: the W scales of stage st, the X block scales of unit column kc
        auto store_unit = [&](int st, int kc) {
            const uint32_t sfa = sf_base + st * kF4SfCols;
            const uint4 a = lds128(sbase + st * kStage + kF4WBytes + 16 * r);
            const uint32_t v[16] = {a.x, a.x, a.x, a.x, a.y, a.y, a.y, a.y, a.z, a.z, a.z, a.z, a.w, a.w, a.w, a.w};
            tc::st_32x32b_x16(sfa + lane_bits, v);
            const uint32_t tab = sTab + (uint32_t)kc * kTab;
            uint32_t w[16];
#pragma unroll
            for (int c32 = 0; c32 < 4; ++c32) {
                const int n = 32 * c32 + lane;  // token-term column; token n / 8
                uint4 b = make_uint4(0, 0, 0, 0);
                if (n < NC) b = lds128(tab + 16 * (n >> 3));
                w[c32] = b.x;
                w[4 + c32] = b.y;
                w[8 + c32] = b.z;
                w[12 + c32] = b.w;
            }
            tc::st_32x32b_x16(sfa + 16 + lane_bits, w);
        };
        // Units in pairs when the next stage has landed too: one hand-off
        // (store wait, fence, arrivals) for both.
        F4Walk sw;
        if (count > 0) sw.begin(ord, S);
        for (int i = 0; i < count && ok;) {
            const int st0 = sw.st;
            if (__any_sync(0xffffffffu, !mbar_wait_bounded(sFull + 8 * st0, sw.ph))) {
                ok = false;
                break;
            }
            store_unit(st0, sw.kc);
            sw.next();
            int done = 1;
            if (i + 1 < count && __all_sync(0xffffffffu, mbar_test(sFull + 8 * sw.st, sw.ph))) {
                store_unit(sw.st, sw.kc);
                done = 2;
            }
            const int st1 = sw.st;
            if (done == 2) sw.next();
            tc::wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(sSf + 8 * st0);
                if (done == 2) mbar_arrive(sSf + 8 * st1);
                st_release_smem(sSfDone + 4 * q, (uint32_t)(i + done));
            }
            i += done;
        }
        tc::wait_st();
        if (!ok && lane == 0) atomicOr(p.err, kDevErrTimeoutFull);
    } else if (warp >= kF4WarpEpi0 && warp < kF4WarpEpi0 + 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const uint32_t lane_bits = (uint32_t)(32 * q) << 16;
        const int r = 32 * q + lane;
        griddep_wait();  // the term scales, g, the workspace and Y belong to this call from here on
        const float g = ld_dep_f32(p.gscale);
        g_ep = g;
        for (int i = (int)threadIdx.x - kF4WarpEpi0 * 32; i < 16 * kF4Terms; i += 128)
            tscale[i] = i < p.n * kF4Terms ? ld_dep_f32(p.xs + i) : 0.f;
        named_sync(1, 128);
        // the other part of a two-part row block, loaded ahead of time
        float pre_part[16];
        int pre_rb = -1;
        int seg_i0 = 0;  // processing-order index of the segment's first unit
        for (int s = 0; s < ord.nseg; seg_i0 += ord.seg_len(ord.nat(s)), ++s) {
            const int ns = ord.nat(s);
            const int rb = ord.rb0 + ns;
            const int len = ord.seg_len(ns);
            const bool whole = len == KC;
            // the row block's counter, partial tiles and rows (the same for the four warps)
            if (!nvfp4_in_bounds(rb >= 0 && rb < p.row_blocks, p.err)) break;
            const long long ub = (long long)rb * KC;
            const int ca = (int)(((ub + 1) * p.ctas - 1) / U), cb = (int)(((ub + KC) * p.ctas - 1) / U);
            const int sb = s & 1;
            // While the last segment's MMAs run: if it is one of the two parts
            // of a split row block, watch for the other part to be published
            // and load it then; this CTA then adds the last part and needs no
            // count (a two-part sum is the same in either order).  The watch
            // ends when the accumulators are ready (bounded like every wait).
            if (!cl && s == ord.nseg - 1 && !whole && cb == ca + 1) {
                const unsigned long long t0 = globaltimer_ns();
                for (;;) {
                    if (warp == kF4WarpEpi0 && lane == 0) {
                        unsigned v = ld_acquire_u32(p.counters + rb) == 1u ? 1u : 0u;
                        if (!v) {
                            bool ready = true;
#pragma unroll
                            for (int j = 0; j < kIssuers; ++j)
                                ready = ready && mbar_test(sDFull + 8 * (j * 2 + sb), (s >> 1) & 1);
                            v = ready || globaltimer_ns() - t0 > kWaitLimitNs ? 2u : 0u;
                        }
                        misc[2] = v;
                    }
                    named_sync(1, 128);
                    const unsigned v = misc[2];
                    named_sync(1, 128);  // misc[2] is written again in the next round
                    if (v == 1u) {
                        pre_rb = rb;
                        f4_load_part(p, pre_part, (int)blockIdx.x == ca ? cb : ca, rb, r, U, KC);
                    }
                    if (v != 0u) break;
                    __nanosleep(200);
                }
            }
            bool waited = true;
#pragma unroll
            for (int j = 0; j < kIssuers; ++j)
                waited = waited && mbar_wait_bounded(sDFull + 8 * (j * 2 + sb), (s >> 1) & 1);
            // all four epilogue warps leave together if any of them gave up
            if (named_sync_or(1, 128, !waited)) {
                if (lane == 0) atomicOr(p.err, kDevErrTimeoutFull);
                break;
            }
            tc::fence_after_sync();
            // issuer j contributed to this segment if one of its units lies in it
            const bool from1 = kIssuers == 2 && (len >= 2 || (seg_i0 & 1) == 1);
            const bool from0 = kIssuers == 1 || len >= 2 || (seg_i0 & 1) == 0;
            float acc[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) acc[t] = 0.f;
            // columns in chunks of 32 (four tokens' eight terms)
#pragma unroll
            for (int c0 = 0; c0 < NC; c0 += 32) {
                uint32_t d[32];
                // the issuers' accumulators, summed in issuer order
#pragma unroll
                for (int c = 0; c < 32; c += 16) {
                    if (c0 + c < NC) {
                        uint32_t part[16];
                        tc::ld_32x32b_x16(tbase + lane_bits + ((from0 ? 0 : 2) + sb) * kDStride + c0 + c, part);
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) d[c + jj] = part[jj];
                    }
                }
                tc::wait_ld();
                if (kIssuers == 2 && from0 && from1) {
#pragma unroll
                    for (int c = 0; c < 32; c += 16) {
                        if (c0 + c < NC) {
                            uint32_t part[16];
                            tc::ld_32x32b_x16(tbase + lane_bits + (2 + sb) * kDStride + c0 + c, part);
                            tc::wait_ld();
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj)
                                d[c + jj] = __float_as_uint(__uint_as_float(d[c + jj]) + __uint_as_float(part[jj]));
                        }
                    }
                }
#pragma unroll
                for (int tl = 0; tl < 4; ++tl) {
                    const int t = c0 / kF4Terms + tl;
                    if (t < 16 && c0 + kF4Terms * tl + kF4Terms - 1 < NC) {
                        // the terms times their scales, the smallest first
                        float sum = __uint_as_float(d[kF4Terms * tl + kF4Terms - 1]) *
                                    tscale[t * kF4Terms + kF4Terms - 1];
#pragma unroll
                        for (int jj = kF4Terms - 2; jj >= 0; --jj)
                            sum = sum + __uint_as_float(d[kF4Terms * tl + jj]) * tscale[t * kF4Terms + jj];
                        acc[t] = sum;
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(sDEmpty + 8 * sb);
            const int row = rb * kUnitRows + r;
            if (whole) {
                f4_store_row(p, acc, row, g);
                continue;
            }
            if (cl) {  // the cluster sums the parts after the loop
                // the rows of warp q are summed by the CTA of rank q % cl: its
                // own part stays in its ring stage 0, the others are pushed
                // into its receive area (slot = sender rank, less one above it)
                const int rank = (int)cluster_ctarank(), k = q % cl;
                if (k == rank) {
#pragma unroll
                    for (int qd = 0; qd < 4; ++qd)
                        if (4 * qd < p.n)
                            sts128(sRed + (uint32_t)r * 64 + 16 * qd,
                                   make_uint4(__float_as_uint(acc[4 * qd]), __float_as_uint(acc[4 * qd + 1]),
                                              __float_as_uint(acc[4 * qd + 2]), __float_as_uint(acc[4 * qd + 3])));
                } else {
                    const uint32_t slot = (uint32_t)(rank < k ? rank : rank - 1);
                    const uint32_t dst = cluster_map(
                        sRecv + (slot * (uint32_t)red_rows + (uint32_t)((q / cl) * 32 + lane)) * 64, (uint32_t)k);
#pragma unroll
                    for (int qd = 0; qd < 4; ++qd)
                        if (4 * qd < p.n)
                            st_cluster_f4(dst + 16 * qd, acc[4 * qd], acc[4 * qd + 1], acc[4 * qd + 2],
                                          acc[4 * qd + 3]);
                }
                red_pending = true;
                red_row = row;
                continue;
            }
            // A split row block.  This CTA adds the last part when the other
            // parts are in already -- found before the segment (and loaded
            // ahead, two-part rows) or now (loaded now) -- or when its count
            // arrives last; it then sums the parts in CTA order.  Otherwise it
            // publishes its part and counts it.
            bool last = pre_rb == rb, loaded = last;
            if (!last) {
                if (warp == kF4WarpEpi0 && lane == 0)
                    misc[2] = ld_acquire_u32(p.counters + rb) + 1 == (unsigned)(cb - ca + 1) ? 1u : 0u;
                named_sync(1, 128);
                last = misc[2] != 0;
            }
            if (!last) {
                float *const part_out =
                    p.partials + ((size_t)blockIdx.x * 2 + (ns == 0 ? 0 : 1)) * (kUnitRows * 16) + (size_t)r * 16;
#pragma unroll
                for (int qd = 0; qd < 4; ++qd)
                    if (4 * qd < p.n)
                        __stcg(reinterpret_cast<float4 *>(part_out) + qd,
                               make_float4(acc[4 * qd], acc[4 * qd + 1], acc[4 * qd + 2], acc[4 * qd + 3]));
                named_sync(1, 128);  // every row's part is stored: one release covers them
                if (warp == kF4WarpEpi0 && lane == 0) {
                    const unsigned old = atom_add_acq_rel(p.counters + rb, 1u);
                    misc[1] = (old + 1 == (unsigned)(cb - ca + 1)) ? 1u : 0u;
                }
                named_sync(1, 128);
                last = misc[1] != 0;
            }
            if (!last) continue;
            float sum[16];
            if (loaded) {
                // the two parts of the row block; either order gives the same sum
#pragma unroll
                for (int t = 0; t < 16; ++t) sum[t] = acc[t] + pre_part[t];
            } else {
                f4_sum_parts<(NC / kF4Terms + 3) / 4>(p, sum, ca, cb, (int)blockIdx.x, acc, rb, r, U, KC);
            }
            f4_store_row(p, sum, row, g);
            if (warp == kF4WarpEpi0 && lane == 0) p.counters[rb] = 0;  // ready for the next call
        }
    }

    if (cl) {
        // every CTA's parts are in the shared memory of the CTAs that sum them
        // (the hardware cluster barrier: every thread of the cluster arrives,
        // and every CTA gets here, since all its own waits are bounded; after
        // it no CTA touches another's shared memory, so none waits to leave)
        __syncwarp();
        cluster_arrive();
        cluster_wait();
        const int q = warp & 3, rank = (int)cluster_ctarank();
        if (warp >= kF4WarpEpi0 && warp < kF4WarpEpi0 + 4 && q % cl == rank && red_pending)
            f4_cluster_finish<(NC / kF4Terms + 3) / 4>(
                F4Out{p.y, p.N, p.n, p.swiglu}, sRed + (uint32_t)(32 * q + lane) * 64,
                sRecv + (uint32_t)((q / cl) * 32 + lane) * 64, (uint32_t)red_rows * 64, rank, cl, red_row, g_ep);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kF4WarpIssuer) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tbase, kF4TmemCols);
    }
}

cudaError_t f4_set_smem_limit(int smem_optin) {
    cudaError_t e;
#define NVFP4_F4_SET(NCV)                                                                                     \
    if ((e = cudaFuncSetAttribute(gemv_fp4_kernel<NCV>, cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                                  smem_optin)) != cudaSuccess)                                                \
        return e;
    NVFP4_F4_SET(16)
    NVFP4_F4_SET(32)
    NVFP4_F4_SET(48)
    NVFP4_F4_SET(64)
    NVFP4_F4_SET(80)
    NVFP4_F4_SET(96)
    NVFP4_F4_SET(112)
    NVFP4_F4_SET(128)
#undef NVFP4_F4_SET
    return cudaSuccess;
}

static const void *f4_kernel(int cols) {
    switch (cols) {
        case 16: return reinterpret_cast<const void *>(gemv_fp4_kernel<16>);
        case 32: return reinterpret_cast<const void *>(gemv_fp4_kernel<32>);
        case 48: return reinterpret_cast<const void *>(gemv_fp4_kernel<48>);
        case 64: return reinterpret_cast<const void *>(gemv_fp4_kernel<64>);
        case 80: return reinterpret_cast<const void *>(gemv_fp4_kernel<80>);
        case 96: return reinterpret_cast<const void *>(gemv_fp4_kernel<96>);
        case 112: return reinterpret_cast<const void *>(gemv_fp4_kernel<112>);
        case 128: return reinterpret_cast<const void *>(gemv_fp4_kernel<128>);
        default: return nullptr;
    }
}

// Whether `ctas` CTAs in clusters of `cs` can all be resident at once (the
// CTAs of a cluster share a GPC, so not every grid of one CTA per SM divides
// into co-resident clusters).  Cached per (device, columns, shared memory,
// cluster size).
static bool f4_clusters_fit(int cols, int smem, int cs, int ctas) {
    struct Entry {
        int dev, cols, smem, cs, clusters;
    };
    static thread_local Entry cache[16];
    static thread_local int used = 0, next = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    for (int i = 0; i < used; ++i)
        if (cache[i].dev == dev && cache[i].cols == cols && cache[i].smem == smem && cache[i].cs == cs)
            return cache[i].clusters * cs >= ctas;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kF4Threads);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, f4_kernel(cols), &cfg) != cudaSuccess) {
        cudaGetLastError();  // not fatal: the split rows go through the workspace then
        clusters = 0;
    }
    cache[next] = Entry{dev, cols, smem, cs, clusters};
    next = (next + 1) % 16;
    if (used < 16) ++used;
    return clusters * cs >= ctas;
}

cudaError_t launch_fp4(const CUtensorMap &tw, const CUtensorMap &ts, const uint16_t *x, const F4Params &p_in,
                       int smem, cudaStream_t stream) {
    F4Params p = p_in;
    // clusters only when they can all be resident at once (one CTA per SM)
    if (p.cluster && (p.ctas % p.cluster != 0 || !f4_clusters_fit(p.cols, smem, p.cluster, p.ctas))) p.cluster = 0;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = p.cluster ? (unsigned)p.cluster : 1u;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t xc = {};
    xc.gridDim = dim3((unsigned)((p.K + kF4XprepElems - 1) / kF4XprepElems), (unsigned)p.n);
    xc.blockDim = dim3(kF4XprepThreads);
    xc.stream = stream;
    xc.attrs = attr;
    xc.numAttrs = 1;
    const int loads = (p.K + kF4XprepElems - 1) / kF4XprepElems;
    cudaError_t e;
    if (loads <= 1) e = cudaLaunchKernelEx(&xc, fp4_xprep_kernel<1>, x, p.xq, p.xtab, p.xs, p.K, p.cols);
    else if (loads <= 2) e = cudaLaunchKernelEx(&xc, fp4_xprep_kernel<2>, x, p.xq, p.xtab, p.xs, p.K, p.cols);
    else if (loads <= 4) e = cudaLaunchKernelEx(&xc, fp4_xprep_kernel<4>, x, p.xq, p.xtab, p.xs, p.K, p.cols);
    else if (loads <= 8) e = cudaLaunchKernelEx(&xc, fp4_xprep_kernel<8>, x, p.xq, p.xtab, p.xs, p.K, p.cols);
    else e = cudaLaunchKernelEx(&xc, fp4_xprep_kernel<16>, x, p.xq, p.xtab, p.xs, p.K, p.cols);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ctas);
    cfg.blockDim = dim3(kF4Threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = p.cluster ? 2 : 1;
    switch (p.cols) {
        case 16: return cudaLaunchKernelEx(&cfg, gemv_fp4_kernel<16>, tw, ts, p);
        case 32: return cudaLaunchKernelEx(&cfg, gemv_fp4_kernel<32>, tw, ts, p);
        case 48: return cudaLaunchKernelEx(&cfg, gemv_fp4_kernel<48>, tw, ts, p);
        case 64: return cudaLaunchKernelEx(&cfg, gemv_fp4_kernel<64>, tw, ts, p);
        case 80: return cudaLaunchKernelEx(&cfg, gemv_fp4_kernel<80>, tw, ts, p);
        case 96: return cudaLaunchKernelEx(&cfg, gemv_fp4_kernel<96>, tw, ts, p);
        case 112: return cudaLaunchKernelEx(&cfg, gemv_fp4_kernel<112>, tw, ts, p);
        case 128: return cudaLaunchKernelEx(&cfg, gemv_fp4_kernel<128>, tw, ts, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace nvfp4
