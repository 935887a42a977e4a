// quantize_gpu.cu -- GPU quantizer: fp32 or bf16 weights [N][K] -> NVFP4
// (packed E2M1 codes [N][K/2], E4M3 block scales [N][K/16], fp32 global scale).
//
// This is the runtime requantization step in front of the GEMV: the pages'
// measurements turn on attention weights stored as BF16 and requantized to
// FP4 at load time (atlas pull request #266, conversation, "Tiebreaker: the
// win is the BF16→FP4 requant path").  The steps and their fp32 rounding are
// those of the library's reference quantizer (nvfp4_quantize_ref):
//   amax = max |w|;  g = amax / 2688 (1 if amax == 0);
//   per 16-block: s = E4M3_rne_sat(blockabsmax / (6 g));
//   per element: code = E2M1_rne_sat(w / (E4M3(s) g)), 0 when E4M3(s) == 0;
// every division and product correctly rounded fp32 (no fused multiply-add),
// so the bytes equal the reference's.
//
// Three launches: the amax reduction (into the global-scale slot, as the bits
// of a non-negative float), the block quantizer (one thread per 16-block,
// walking the matrix back to front so that it starts on what the amax pass
// left in L2), and a one-thread finish that turns amax into g in place.
#include "internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>

namespace nvfp4 {

namespace {

constexpr unsigned kDevErrQuantInput = 16u;  // a weight was not finite

// Weights travel as raw 16-byte vectors: 4 fp32 or 8 bf16 (bf16 -> fp32 is
// exact: the bf16 bits are the top half of the fp32 bits).
template <typename TW> struct WTraits;
template <> struct WTraits<float> {
    static constexpr int kVecPerBlock = 4;  // 16 weights = 64 bytes
    // fp32 bits of element j of the block.
    __device__ static uint32_t bits(const uint4 (&r)[4], int j) {
        const uint4 u = r[j >> 2];
        return (j & 3) == 0 ? u.x : (j & 3) == 1 ? u.y : (j & 3) == 2 ? u.z : u.w;
    }
    // fp32 bits of the block's largest |w| (non-negative floats order as integers).
    __device__ static uint32_t abs_max_bits(const uint4 (&r)[4]) {
        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) m = max(m, bits(r, j) & 0x7FFFFFFFu);
        return m;
    }
};
template <> struct WTraits<uint16_t> {
    static constexpr int kVecPerBlock = 2;  // 16 weights = 32 bytes
    __device__ static uint32_t bits(const uint4 (&r)[2], int j) {
        const uint4 u = r[j >> 3];
        const int h = (j & 7) >> 1;
        const uint32_t word = h == 0 ? u.x : h == 1 ? u.y : h == 2 ? u.z : u.w;
        return (j & 1) ? (word & 0xFFFF0000u) : (word << 16);  // element 2i in the low half
    }
    __device__ static uint32_t abs_max_bits(const uint4 (&r)[2]) {
        uint32_t m = 0;  // two 16-bit magnitudes per word, compared as unsigned halves
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            m = __vmaxu2(m, r[q].x & 0x7FFF7FFFu);
            m = __vmaxu2(m, r[q].y & 0x7FFF7FFFu);
            m = __vmaxu2(m, r[q].z & 0x7FFF7FFFu);
            m = __vmaxu2(m, r[q].w & 0x7FFF7FFFu);
        }
        return max(m & 0xFFFFu, m >> 16) << 16;
    }
};

__device__ __forceinline__ uint4 ld_vec(const uint4 *p) {
    uint4 u;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                 : "l"(p));
    return u;
}

// E4M3, round to nearest even, saturating at 448; a >= 0 and finite.
__device__ __forceinline__ unsigned e4m3_encode(float a) {
    if (a >= 448.0f) return 0x7Eu;
    if (a < 0.015625f) {  // below 2^-6: subnormal grid of 2^-9 (a * 512 is exact)
        return (unsigned)__float2int_rn(a * 512.0f);  // 8 (rounded up a binade) is also the code of 2^-6
    }
    const unsigned bits = __float_as_uint(a);
    int exp = (int)(bits >> 23) - 127;  // -6 .. 8
    unsigned mant = bits & 0x7FFFFFu;
    unsigned keep = mant >> 20, rem = mant & 0xFFFFFu;
    if (rem > 0x80000u || (rem == 0x80000u && (keep & 1u))) ++keep;
    if (keep == 8u) {
        keep = 0u;
        ++exp;
    }
    const unsigned code = ((unsigned)(exp + 7) << 3) | keep;
    return code > 0x7Eu ? 0x7Eu : code;
}

// E4M3 code -> fp32 (exact).
__device__ __forceinline__ float e4m3_decode(unsigned c) {
    const unsigned e = (c >> 3) & 15u, m = c & 7u;
    if (e == 0) return (float)m * 0.001953125f;  // m * 2^-9
    return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// E2M1, round to nearest with ties to the even mantissa, saturating at 6; a
// magnitude that rounds to zero is code 0 whatever the sign.
__device__ __forceinline__ unsigned e2m1_encode(float v) {
    const float a = fabsf(v);
    unsigned mag = (a <= 0.25f) ? 0u
                 : (a < 0.75f)  ? 1u
                 : (a <= 1.25f) ? 2u
                 : (a < 1.75f)  ? 3u
                 : (a <= 2.5f)  ? 4u
                 : (a < 3.5f)   ? 5u
                 : (a <= 5.0f)  ? 6u
                                : 7u;
    return (mag != 0u && v < 0.0f) ? (mag | 8u) : mag;
}

// Running max of |w| over one 16-byte vector; `bad` records inf or NaN.
template <typename TW>
__device__ __forceinline__ void vec_abs_max(const uint4 u, float &m, bool &bad) {
    const uint32_t words[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (sizeof(TW) == 4) {
            const float a = __uint_as_float(words[j] & 0x7FFFFFFFu);
            bad |= !(a <= 3.402823466e38f);
            m = a > m ? a : m;
        } else {
            const float a0 = __uint_as_float((words[j] << 16) & 0x7FFFFFFFu);
            const float a1 = __uint_as_float(words[j] & 0x7FFF0000u);
            bad |= !(a0 <= 3.402823466e38f) || !(a1 <= 3.402823466e38f);
            m = a0 > m ? a0 : m;
            m = a1 > m ? a1 : m;
        }
    }
}

// amax over the nvec 16-byte vectors of w, four loads in flight per thread,
// one atomicMax per CTA on the bits of the (non-negative) result.
constexpr int kAmaxThreads = 512;
template <typename TW>
__global__ void __launch_bounds__(kAmaxThreads) quant_amax_kernel(const TW *__restrict__ w, size_t nvec,
                                                                  unsigned *amax_bits, unsigned *err) {
    griddep_launch_dependents();  // the block pass may start loading weights as SMs free up
    const uint4 *p = reinterpret_cast<const uint4 *>(w);
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    float m = 0.0f;
    bool bad = false;
    for (; i + 3 * stride < nvec; i += 4 * stride) {
        const uint4 u0 = ld_vec(p + i), u1 = ld_vec(p + i + stride), u2 = ld_vec(p + i + 2 * stride),
                    u3 = ld_vec(p + i + 3 * stride);
        vec_abs_max<TW>(u0, m, bad);
        vec_abs_max<TW>(u1, m, bad);
        vec_abs_max<TW>(u2, m, bad);
        vec_abs_max<TW>(u3, m, bad);
    }
    for (; i < nvec; i += stride) vec_abs_max<TW>(ld_vec(p + i), m, bad);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float warp_max[kAmaxThreads / 32];
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
    const int any_bad = __syncthreads_or(bad ? 1 : 0);
    if (threadIdx.x < 32) {
        m = threadIdx.x < kAmaxThreads / 32 ? warp_max[threadIdx.x] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (threadIdx.x == 0) {
            atomicMax(amax_bits, __float_as_uint(m));  // non-negative floats order as integers
            if (any_bad) atomicOr(err, kDevErrQuantInput);
        }
    }
}

// Per-element quotient without a division instruction sequence per element.
// Markstein's method (P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Develop. 34(1), 1990): if
// y = RN(1/d), q is a faithful approximation of v/d (one of the two floats
// around it) and nothing underflows, then r = v - q d is exact in one fma and
// RN(q + r y) = RN(v / d).  q0 = RN(v y) may be two ulps off, so one
// correction first makes it faithful and a second one makes it exact.  The
// caller keeps d in [2^-60, 2^60]: then the only quotients that can decide a
// code (|v/d| >= 0.25) have v and r far above the fp32 normal range's floor.
__device__ __forceinline__ float div_by_markstein(float v, float d, float y) {
    float q = __fmul_rn(v, y);
    float r = __fmaf_rn(-q, d, v);
    q = __fmaf_rn(r, y, q);  // faithful
    r = __fmaf_rn(-q, d, v);  // exact
    return __fmaf_rn(r, y, q);
}

// Eight fp32 values -> eight E2M1 codes (nearest, ties to even, saturating at
// 6), value j in nibble j (the hardware conversion puts its first operand in
// the high nibble).  A negative value that rounds to zero comes out as code 8
// (-0); the caller clears those.
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float (&q)[8]) {
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

// Clear the sign bit of every nibble whose magnitude bits are 0 (-0 -> +0):
// adding 7 to a 3-bit magnitude carries into bit 3 exactly when it is nonzero.
__device__ __forceinline__ uint32_t clear_negative_zeros(uint32_t x) {
    const uint32_t nonzero = ((x & 0x77777777u) + 0x77777777u) & 0x88888888u;
    return x & (nonzero | 0x77777777u);
}

// Scale byte and 8 code bytes of one 16-block held as raw vectors.
template <typename TW>
__device__ __forceinline__ void quantize_block(const uint4 (&r)[WTraits<TW>::kVecPerBlock], float g, float six_g,
                                               uint2 &codes, unsigned &sc) {
    sc = e4m3_encode(__fdiv_rn(__uint_as_float(WTraits<TW>::abs_max_bits(r)), six_g));
    const float s_val = e4m3_decode(sc);
    const float d = __fmul_rn(s_val, g);
    uint32_t half[2] = {0u, 0u};
    if (d >= 0x1p-60f && d <= 0x1p60f) {
        const float y = __frcp_rn(d);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float q[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) q[j] = div_by_markstein(__uint_as_float(WTraits<TW>::bits(r, 8 * h + j)), d, y);
            half[h] = clear_negative_zeros(cvt_e2m1x8(q));
        }
    } else if (s_val != 0.0f) {  // scales far out of range: one correctly rounded division per element
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const unsigned q = e2m1_encode(__fdiv_rn(__uint_as_float(WTraits<TW>::bits(r, j)), d));
            half[j >> 3] |= q << (4 * (j & 7));
        }
    }
    codes = make_uint2(half[0], half[1]);  // element 2i in the low nibble of byte i
}

// One thread per 16-block, kBlocksInFlight blocks loaded per thread before
// any is processed.  Blocks are taken from the END of the matrix first: the
// amax pass read the matrix front to back, so its last part is what L2 still
// holds.
constexpr int kBlockThreads = 256, kBlockCtasPerSm = 3;  // one resident wave (launch bounds below)
template <typename TW> struct BlockPass {
    static constexpr int kBlocksInFlight = sizeof(TW) == 2 ? 4 : 2;  // 128 bytes of weights per thread
};

template <typename TW>
__global__ void __launch_bounds__(kBlockThreads, kBlockCtasPerSm) quant_blocks_kernel(const TW *__restrict__ w, long long nb,
                                                                        const unsigned *amax_bits,
                                                                        uint8_t *__restrict__ packed,
                                                                        uint8_t *__restrict__ scale) {
    constexpr int V = WTraits<TW>::kVecPerBlock, B = BlockPass<TW>::kBlocksInFlight;
    const uint4 *p = reinterpret_cast<const uint4 *>(w);  // block b = vectors [V b, V b + V)
    const long long stride = (long long)gridDim.x * blockDim.x;
    long long j = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    uint4 r[B][V];
    // Iteration j holds blocks nb - 1 - (j + i stride), i < B (those >= 0).
    auto load = [&](long long jj) {
#pragma unroll
        for (int i = 0; i < B; ++i) {
            const long long b = nb - 1 - (jj + i * stride);
            if (b >= 0) {
#pragma unroll
                for (int q = 0; q < V; ++q) r[i][q] = ld_vec(p + b * V + q);
            }
        }
    };
    // The weights are this call's input, final before the amax pass started:
    // the first blocks are requested while that pass is still running.
    if (j < nb) load(j);
    griddep_wait();  // amax is complete from here on
    const float amax = __uint_as_float(*amax_bits);
    const float g = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 2688.0f);
    const float six_g = __fmul_rn(6.0f, g);
    while (j < nb) {
#pragma unroll
        for (int i = 0; i < B; ++i) {
            const long long b = nb - 1 - (j + i * stride);
            if (b >= 0) {
                uint2 c;
                unsigned sc;
                quantize_block<TW>(r[i], g, six_g, c, sc);
                *reinterpret_cast<uint2 *>(packed + b * 8) = c;
                scale[b] = (uint8_t)sc;
            }
        }
        j += B * stride;
        if (j < nb) load(j);
    }
}

__global__ void quant_finish_kernel(float *global_scale) {
    griddep_wait();                    // every block has read amax
    if (threadIdx.x != 0) return;
    const float amax = *global_scale;  // holds the amax bits until now
    *global_scale = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 2688.0f);
}

template <typename TW>
cudaError_t launch_quantize(const TW *w, int N, int K, uint8_t *packed, uint8_t *scale, float *global_scale,
                            unsigned *err, int sms, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(global_scale, 0, sizeof(float), stream);
    if (e != cudaSuccess) return e;
    const size_t nvec = (size_t)N * K / (16 / sizeof(TW));  // K % 16 == 0: whole 16-byte vectors
    const long long want = (long long)((nvec + kAmaxThreads - 1) / kAmaxThreads);
    const int grid_a = (int)(want < 4LL * sms ? want : 4LL * sms);
    quant_amax_kernel<TW><<<grid_a, kAmaxThreads, 0, stream>>>(w, nvec, reinterpret_cast<unsigned *>(global_scale), err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const long long nb = (long long)N * (K >> 4);
    const long long want_b = (nb + kBlockThreads - 1) / kBlockThreads;
    const long long wave_b = (long long)kBlockCtasPerSm * sms;
    const int grid_b = (int)(want_b < wave_b ? want_b : wave_b);
    // The block pass and the finish launch as programmatic dependents: each
    // waits (griddepcontrol.wait) for the grid ahead of it before it reads
    // amax, and the finish triggers nothing early, so work queued after this
    // call starts only when all three are done.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_b);
    cfg.blockDim = dim3(kBlockThreads);
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, quant_blocks_kernel<TW>, w, nb, reinterpret_cast<const unsigned *>(global_scale),
                           packed, scale);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(32);
    return cudaLaunchKernelEx(&cfg, quant_finish_kernel, global_scale);
}

}  // namespace

cudaError_t launch_quantize_f32(const float *w, int N, int K, uint8_t *packed, uint8_t *scale, float *global_scale,
                                unsigned *err, int sms, cudaStream_t stream) {
    return launch_quantize<float>(w, N, K, packed, scale, global_scale, err, sms, stream);
}

cudaError_t launch_quantize_bf16(const uint16_t *w, int N, int K, uint8_t *packed, uint8_t *scale,
                                 float *global_scale, unsigned *err, int sms, cudaStream_t stream) {
    return launch_quantize<uint16_t>(w, N, K, packed, scale, global_scale, err, sms, stream);
}

}  // namespace nvfp4
