// gemv_stream.cu -- the streaming NVFP4 batched-decode GEMV kernels for sm_103a.
//
// Y[t, r] = g * sum_k X[t, k] * E2M1(W[r, k]) * E4M3(S[r, k/16]) for all n <= 16
// tokens from ONE pass over W (atlas pull request #266, "What it does": each
// tile of tokens reads the projection weight once; here the tile is all n).
//
// Structure of one launch (persistent grid, one CTA per SM):
//   * The weight matrix is cut into units of 128 rows x 128 k.  Units are
//     ordered row-block-major and CTA c owns the contiguous range
//     [c*U/C, (c+1)*U/C), so every SM streams the same number of bytes
//     whatever N and K are ("stream-K" partition).
//   * Warp 4 is the producer: one lane issues 2D TMA loads (packed W tile
//     128 x 64 B and its 128 x 16 B scale tile) into a ring of up to 8
//     shared-memory stages, each guarded by a full and an empty mbarrier.
//   * Warps 0-3 are consumers: warp w owns rows 32w..32w+31 of every unit.
//     X (n x K bf16) is converted to f16 once per CTA into shared memory in a
//     fragment-native order; weights are dequantised in registers (E2M1 ->
//     f16 with cvt, times the E4M3 block scale, both exact) and fed to
//     mma.sync m16n8k16 (A = 16 tokens x 16 k, B = 16 k x 8 rows, fp32
//     accumulate) -- or, in the SIMT variant, to fp32 FMAs.
//   * A row block finished inside one CTA is written directly (times g,
//     rounded to bf16).  A row block split between CTAs writes fp32 partial
//     tiles to the workspace; the last CTA to arrive (atomic counter) sums
//     the partials in CTA order -- a fixed order, so results are
//     deterministic and independent of n -- and writes Y.  Nobody waits on
//     another CTA.
//   * Every mbarrier wait gives up after 2 s of wall-clock time, sets the
//     device error word and unwinds; the producer then waits (again bounded)
//     for its own copies in flight before the CTA exits.
#include "internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>

namespace nvfp4 {

__device__ unsigned g_device_error;

__device__ __forceinline__ int cta_of_unit(long long u, long long U, int C) {
    return (int)(((u + 1) * (long long)C - 1) / U);
}

// -------------------------------------------------------------- X staging
// X[t][k] -> f16 at  kc*(4*n*64) + i*(n*64) + t*64 + q*16 + e*2  bytes, where
// k = kc*128 + 32q + 8i + e.  For a fixed (kc, i) the 16-byte groups of all
// tokens and quads are contiguous, so the consumers' A-fragment loads
// (lane = 4*token + quad) are bank-conflict free.
__device__ __forceinline__ uint32_t x_slot_offset(int t, int k, int n) {
    return (uint32_t)((k >> 7) * (4 * n * 64) + ((k >> 3) & 3) * (n * 64) + t * 64 + ((k >> 5) & 3) * 16);
}

__device__ __forceinline__ uint32_t bf16pair_to_f16x2(uint32_t u, float mul, bool &ovf) {
    float lo = __uint_as_float(u << 16) * mul;
    float hi = __uint_as_float(u & 0xFFFF0000u) * mul;
    // f16 overflows to infinity at |v| >= 65520; infinities and NaNs in X are
    // passed through unchanged (they propagate, as in the definition).
    ovf |= (fabsf(lo) >= 65520.f && isfinite(lo)) || (fabsf(hi) >= 65520.f && isfinite(hi));
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ bool stage_x_pass(const StreamParams &p, uint32_t sX, float mul) {
    const int groups = p.K >> 3;
    const int total = p.n * groups;
    bool ovf = false;
    for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
        const int t = idx / groups;
        const int k = (idx - t * groups) << 3;
        const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)t * p.K + k));
        uint4 o;
        o.x = bf16pair_to_f16x2(raw.x, mul, ovf);
        o.y = bf16pair_to_f16x2(raw.y, mul, ovf);
        o.z = bf16pair_to_f16x2(raw.z, mul, ovf);
        o.w = bf16pair_to_f16x2(raw.w, mul, ovf);
        sts128(sX + x_slot_offset(t, k, p.n), o);
    }
    return ovf;
}

// Stage X; returns the power-of-two exponent e such that the staged values
// are X * 2^-e (e = 0 unless some |x| would overflow f16).  All CTAs see the
// same X and so choose the same e.
__device__ int stage_x(const StreamParams &p, uint32_t sX, unsigned *sh_word) {
    bool ovf = stage_x_pass(p, sX, 1.0f);
    if (!__syncthreads_or(ovf)) return 0;
    // Rare path: find max |x| over finite entries, rescale by a power of two.
    if (threadIdx.x == 0) *sh_word = 0u;
    __syncthreads();
    const int total = p.n * p.K;
    unsigned local = 0u;
    for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
        float v = fabsf(__uint_as_float((unsigned)p.x[idx] << 16));
        if (isfinite(v)) local = max(local, __float_as_uint(v));
    }
    atomicMax(sh_word, local);
    __syncthreads();
    const float amax = __uint_as_float(*sh_word);
    const int e = ilogbf(amax) - 14;  // amax * 2^-e < 2^15
    __syncthreads();
    stage_x_pass(p, sX, ldexpf(1.0f, -e));
    return e;
}

// --------------------------------------------------------- compute: MMA
// Thread (g = lane/4, q = lane%4) of consumer warp w, for one unit in stage
// buffers (wS, sS):
//   B fragment of row group r = W rows 32w + 8r + g, k = kc*128 + 32q + [0,32)
//   (16 packed bytes), A fragment = X[g] and X[g+8] at the same k.  MMA step
//   j (0..7) uses packed bytes 2j, 2j+1, i.e. k0 = kc*128 + 32q + 4j .. +3,
//   mapped to the MMA's k slots {2q, 2q+1} and {2q+8, 2q+9}; A uses the same
//   mapping, so the sum over slots is the sum over these 16 physical k.
struct MmaAcc {
    float d[4][4];
};

__device__ __forceinline__ void compute_unit_mma(MmaAcc &acc, uint32_t wS, uint32_t sS, uint32_t xblk, int kc,
                                                 int n, int warp, int g, int q) {
    uint4 xa[4], xb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        xa[i] = (g < n) ? lds128(xblk + i * (n * 64) + g * 64 + q * 16) : make_uint4(0, 0, 0, 0);
        xb[i] = (g + 8 < n) ? lds128(xblk + i * (n * 64) + (g + 8) * 64 + q * 16) : make_uint4(0, 0, 0, 0);
    }
    const uint32_t wrow = wS + (uint32_t)(warp * 32 + g) * 64 + q * 16;
    const uint32_t srow = sS + (uint32_t)(warp * 32 + g) * 16 + (kc & 1) * 8 + q * 2;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const uint4 wv = lds128(wrow + r * 8 * 64);
        const uint32_t s2 = e4m3x2_to_f16x2(lds16(srow + r * 8 * 16));
        const uint32_t sc[2] = {dup_lo(s2), dup_hi(s2)};
        const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t word = words[j >> 1];
            const uint32_t s = sc[j >> 2];
            uint32_t b0, b1;
            if (j & 1) {
                b0 = hmul2_u32(e2m1x2_to_f16x2<2>(word), s);
                b1 = hmul2_u32(e2m1x2_to_f16x2<3>(word), s);
            } else {
                b0 = hmul2_u32(e2m1x2_to_f16x2<0>(word), s);
                b1 = hmul2_u32(e2m1x2_to_f16x2<1>(word), s);
            }
            const uint4 a = xa[j >> 1];
            const uint4 c = xb[j >> 1];
            const uint32_t a0 = (j & 1) ? a.z : a.x;
            const uint32_t a2 = (j & 1) ? a.w : a.y;
            const uint32_t a1 = (j & 1) ? c.z : c.x;
            const uint32_t a3 = (j & 1) ? c.w : c.y;
            mma_16816(acc.d[r], a0, a1, a2, a3, b0, b1);
        }
    }
}

// Value i (0..15) of an MMA lane <-> (token, row within the warp's 32 rows):
// d[r][c] = D[token g + 8*(c>>1)][row 8r + 2q + (c&1)].
__device__ __forceinline__ void mma_coord(int lane, int i, int &tok, int &row) {
    const int r = i >> 2, c = i & 3, g = lane >> 2, q = lane & 3;
    tok = g + 8 * (c >> 1);
    row = 8 * r + 2 * q + (c & 1);
}

// -------------------------------------------------------- compute: SIMT
// Thread (g, q) keeps fp32 partial sums for rows 32w + 8r + g (r = 0..3), all
// tokens, over its own 32 k of each unit; the 4 quads are summed at flush.
struct SimtAcc {
    float d[4][kMaxTokensPerPass];
};

__device__ __forceinline__ float fma_f16x2_into(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{\n .reg .b16 al, ah, bl, bh;\n .reg .f32 t;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
        " fma.rn.f32.f16 t, al, bl, %3;\n fma.rn.f32.f16 %0, ah, bh, t;\n}\n"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
    return d;
}

__device__ __forceinline__ void compute_unit_simt(SimtAcc &acc, uint32_t wS, uint32_t sS, uint32_t xblk, int kc,
                                                  int n, int warp, int g, int q) {
    uint32_t wd[4][16];  // dequantised f16x2 pairs, pair p = k (32q + 2p, +1)
    const uint32_t wrow = wS + (uint32_t)(warp * 32 + g) * 64 + q * 16;
    const uint32_t srow = sS + (uint32_t)(warp * 32 + g) * 16 + (kc & 1) * 8 + q * 2;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const uint4 wv = lds128(wrow + r * 8 * 64);
        const uint32_t s2 = e4m3x2_to_f16x2(lds16(srow + r * 8 * 16));
        const uint32_t sc[2] = {dup_lo(s2), dup_hi(s2)};
        const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int p = 0; p < 16; ++p) {
            const uint32_t word = words[p >> 2];
            const uint32_t s = sc[p >> 3];
            uint32_t v;
            switch (p & 3) {
                case 0: v = e2m1x2_to_f16x2<0>(word); break;
                case 1: v = e2m1x2_to_f16x2<1>(word); break;
                case 2: v = e2m1x2_to_f16x2<2>(word); break;
                default: v = e2m1x2_to_f16x2<3>(word); break;
            }
            wd[r][p] = hmul2_u32(v, s);
        }
    }
#pragma unroll
    for (int t = 0; t < kMaxTokensPerPass; ++t) {
        if (t < n) {
            uint4 xv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) xv[i] = lds128(xblk + i * (n * 64) + t * 64 + q * 16);
            const uint32_t xs[16] = {xv[0].x, xv[0].y, xv[0].z, xv[0].w, xv[1].x, xv[1].y, xv[1].z, xv[1].w,
                                     xv[2].x, xv[2].y, xv[2].z, xv[2].w, xv[3].x, xv[3].y, xv[3].z, xv[3].w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float a = acc.d[r][t];
#pragma unroll
                for (int p = 0; p < 16; ++p) a = fma_f16x2_into(wd[r][p], xs[p], a);
                acc.d[r][t] = a;
            }
        }
    }
}

// Value i of a SIMT lane after the quad reduction: token q + 4*(i&3), row 8*(i>>2) + g.
__device__ __forceinline__ void simt_coord(int lane, int i, int &tok, int &row) {
    const int g = lane >> 2, q = lane & 3;
    tok = q + 4 * (i & 3);
    row = 8 * (i >> 2) + g;
}

// ------------------------------------------------------------------ flush
template <int kVariant>
__device__ __forceinline__ void epilogue(const StreamParams &p, const float (&v)[16], int row_base, int lane,
                                         float gs) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        int tok, rs;
        if constexpr (kVariant == kMma) mma_coord(lane, i, tok, rs);
        else simt_coord(lane, i, tok, rs);
        const int row = row_base + rs;
        if (tok >= p.n || row >= p.N) continue;
        if constexpr (kVariant == kMma) {
            // (i, i+1) with even i are adjacent rows of the same token
            if ((i & 1) == 0 && p.y_vec2 && row + 1 < p.N) {
                __nv_bfloat162 h = __floats2bfloat162_rn(v[i] * gs, v[i + 1] * gs);
                *reinterpret_cast<__nv_bfloat162 *>(p.y + (size_t)tok * p.N + row) = h;
                continue;
            }
            if ((i & 1) == 1 && p.y_vec2 && row < p.N) continue;  // written with its pair
        }
        __nv_bfloat16 h = __float2bfloat16_rn(v[i] * gs);
        p.y[(size_t)tok * p.N + row] = *reinterpret_cast<uint16_t *>(&h);
    }
}

template <int kVariant>
__device__ __forceinline__ void flush_tile(const StreamParams &p, float (&v)[16], int rb, int kfirst, int klast,
                                           int warp, int lane, float gs) {
    const int row_base = rb * kUnitRows + warp * 32;
    if (!(kfirst == 0 && klast == p.KC - 1)) {
        const long long ufirst = (long long)rb * p.KC;
        const int cfirst = cta_of_unit(ufirst, p.units, p.ctas);
        const int clast = cta_of_unit(ufirst + p.KC - 1, p.units, p.ctas);
        const int slot = ((int)blockIdx.x == cfirst) ? 1 : 0;
        // the tile's counter and the parts' slots
        if (!nvfp4_in_bounds(cfirst >= 0 && clast < p.ctas && cfirst <= (int)blockIdx.x &&
                                 (int)blockIdx.x <= clast, p.err))
            return;
        float4 *mine = reinterpret_cast<float4 *>(
            p.partials + (((size_t)blockIdx.x * 2 + slot) * kConsumerWarps + warp) * kSlotFloats + lane * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) mine[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        __threadfence();
        __syncwarp();
        unsigned old = 0;
        if (lane == 0) old = atomicAdd(&p.counters[cfirst * kCountersPerCta + warp], 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old != (unsigned)(clast - cfirst)) return;  // another CTA finishes this tile
        __threadfence();
        for (int c = cfirst; c <= clast; ++c) {
            const int s = (c == cfirst) ? 1 : 0;
            const float4 *src = reinterpret_cast<const float4 *>(
                p.partials + (((size_t)c * 2 + s) * kConsumerWarps + warp) * kSlotFloats + lane * 16);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 f = __ldcg(src + i);
                if (c == cfirst) {
                    v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
                } else {
                    v[4 * i] += f.x; v[4 * i + 1] += f.y; v[4 * i + 2] += f.z; v[4 * i + 3] += f.w;
                }
            }
        }
        if (lane == 0) atomicExch(&p.counters[cfirst * kCountersPerCta + warp], 0u);
    }
    epilogue<kVariant>(p, v, row_base, lane, gs);
}

// ----------------------------------------------------------------- kernel
template <int kVariant>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_stream_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_s,
                       const StreamParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t sW = (raw_addr + 1023u) & ~1023u;
    uint8_t *const base = smem_raw + (sW - raw_addr);
    const int S = p.stages;
    const uint32_t sS = sW + S * kWTileBytes;
    const uint32_t sX = sS + S * kSTileBytes;
    const uint32_t sFull = sX + (uint32_t)(p.n * p.K * 2);
    const uint32_t sEmpty = sFull + 8 * S;
    unsigned *const sh_word = reinterpret_cast<unsigned *>(base + (sEmpty + 8 * S - sW));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long u0 = (long long)blockIdx.x * p.units / p.ctas;
    const long long u1 = (long long)(blockIdx.x + 1) * p.units / p.ctas;
    const int count = (int)(u1 - u0);
    const bool producer = (warp == kConsumerWarps);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(sFull + 8 * s, 1);
            mbar_init(sEmpty + 8 * s, kConsumerWarps);
        }
        fence_barrier_init();
    }
    if (producer && lane == 0) {
        prefetch_tensormap(&tmap_w);
        prefetch_tensormap(&tmap_s);
    }
    __syncthreads();

    const uint64_t policy = l2_policy_evict_first();
    auto issue = [&](int i) {
        const long long u = u0 + i;
        const int rb = (int)(u / p.KC), kc = (int)(u - (long long)rb * p.KC);
        const int slot = i % S;
        const uint32_t full = sFull + 8 * slot;
        mbar_arrive_expect_tx(full, kStageBytes);
        tma_load_2d(sW + slot * kWTileBytes, &tmap_w, kc * (kUnitK / 2), rb * kUnitRows, full, policy);
        tma_load_2d(sS + slot * kSTileBytes, &tmap_s, (kc >> 1) * 16, rb * kUnitRows, full, policy);
    };

    // Start the weight stream before staging X so HBM latency overlaps it.
    int issued = 0;
    if (producer && lane == 0) {
        const int first = count < S ? count : S;
        for (; issued < first; ++issued) issue(issued);
    }
    const int xexp = stage_x(p, sX, sh_word);
    __syncthreads();
    const float gs = __ldg(p.gscale) * ldexpf(1.0f, xexp);

    if (producer) {
        if (lane == 0) {
            bool ok = true;
            for (; issued < count; ++issued) {
                const int slot = issued % S;
                if (!mbar_wait_bounded(sEmpty + 8 * slot, ((issued / S) - 1) & 1)) {
                    atomicOr(p.err, kDevErrTimeoutEmpty);
                    ok = false;
                    break;
                }
                issue(issued);
            }
            // Wait (bounded) for the most recent copy of every slot before the
            // CTA may exit; on the normal path these have all been consumed.
            const int lo = issued > S ? issued - S : 0;
            for (int i = lo; i < issued; ++i) {
                if (!mbar_wait_bounded(sFull + 8 * (i % S), (i / S) & 1)) {
                    atomicOr(p.err, kDevErrTimeoutDrain);
                    break;
                }
            }
            (void)ok;
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int g = lane >> 2, q = lane & 3;
    int kfirst = -1;
    if constexpr (kVariant == kMma) {
        MmaAcc acc;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc.d[r][c] = 0.f;
        for (int i = 0; i < count; ++i) {
            const long long u = u0 + i;
            const int rb = (int)(u / p.KC), kc = (int)(u - (long long)rb * p.KC);
            if (kfirst < 0) kfirst = kc;
            const int slot = i % S;
            const bool ok = mbar_wait_bounded(sFull + 8 * slot, (i / S) & 1);
            if (__any_sync(0xffffffffu, !ok)) {
                if (lane == 0) atomicOr(p.err, kDevErrTimeoutFull);
                return;
            }
            compute_unit_mma(acc, sW + slot * kWTileBytes, sS + slot * kSTileBytes,
                             sX + (uint32_t)kc * (4 * p.n * 64), kc, p.n, warp, g, q);
            __syncwarp();
            if (lane == 0) mbar_arrive(sEmpty + 8 * slot);
            if (kc == p.KC - 1 || i == count - 1) {
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = acc.d[j >> 2][j & 3];
                flush_tile<kMma>(p, v, rb, kfirst, kc, warp, lane, gs);
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc.d[r][c] = 0.f;
                kfirst = -1;
            }
        }
    } else {
        SimtAcc acc;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int t = 0; t < kMaxTokensPerPass; ++t) acc.d[r][t] = 0.f;
        for (int i = 0; i < count; ++i) {
            const long long u = u0 + i;
            const int rb = (int)(u / p.KC), kc = (int)(u - (long long)rb * p.KC);
            if (kfirst < 0) kfirst = kc;
            const int slot = i % S;
            const bool ok = mbar_wait_bounded(sFull + 8 * slot, (i / S) & 1);
            if (__any_sync(0xffffffffu, !ok)) {
                if (lane == 0) atomicOr(p.err, kDevErrTimeoutFull);
                return;
            }
            compute_unit_simt(acc, sW + slot * kWTileBytes, sS + slot * kSTileBytes,
                              sX + (uint32_t)kc * (4 * p.n * 64), kc, p.n, warp, g, q);
            __syncwarp();
            if (lane == 0) mbar_arrive(sEmpty + 8 * slot);
            if (kc == p.KC - 1 || i == count - 1) {
                // sum the four quads' partial dot products (same value on all four)
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int t = 0; t < kMaxTokensPerPass; ++t) {
                        float a = acc.d[r][t];
                        a += __shfl_xor_sync(0xffffffffu, a, 1);
                        a += __shfl_xor_sync(0xffffffffu, a, 2);
                        acc.d[r][t] = a;
                    }
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int r = j >> 2, jj = j & 3;
                    const float c0 = acc.d[r][4 * jj], c1 = acc.d[r][4 * jj + 1];
                    const float c2 = acc.d[r][4 * jj + 2], c3 = acc.d[r][4 * jj + 3];
                    v[j] = (q == 0) ? c0 : (q == 1) ? c1 : (q == 2) ? c2 : c3;
                }
                flush_tile<kSimt>(p, v, rb, kfirst, kc, warp, lane, gs);
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int t = 0; t < kMaxTokensPerPass; ++t) acc.d[r][t] = 0.f;
                kfirst = -1;
            }
        }
    }
}

// ------------------------------------------------------------------- host
cudaError_t stream_set_smem_limits(int smem_optin) {
    cudaError_t e = cudaFuncSetAttribute(gemv_stream_kernel<kMma>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_optin);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gemv_stream_kernel<kSimt>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_optin);
}

cudaError_t launch_stream(int variant, const CUtensorMap &tw, const CUtensorMap &ts, const StreamParams &p,
                          int smem, cudaStream_t stream) {
    const dim3 grid(p.ctas), block(kThreads);
    if (variant == kMma)
        gemv_stream_kernel<kMma><<<grid, block, smem, stream>>>(tw, ts, p);
    else
        gemv_stream_kernel<kSimt><<<grid, block, smem, stream>>>(tw, ts, p);
    return cudaGetLastError();
}

cudaError_t device_error_word(unsigned **ptr) {
    return cudaGetSymbolAddress(reinterpret_cast<void **>(ptr), g_device_error);
}

}  // namespace nvfp4
