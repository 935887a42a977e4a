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
// of a non-negative float), the block quantizer (one thread per 16-block), and
// a one-thread finish that turns amax into g in place.
#include "internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>

namespace nvfp4 {

namespace {

constexpr unsigned kDevErrQuantInput = 16u;  // a weight was not finite

// The 16 weights of one scale block as fp32, in 16-byte loads (a block starts
// on a 32-byte boundary when w is 16-byte aligned); bf16 -> fp32 is exact.
__device__ __forceinline__ void load_block(const float *w, size_t base, float (&v)[16]) {
    const float4 *p = reinterpret_cast<const float4 *>(w + base);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 f = __ldg(p + q);
        v[4 * q] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
    }
}
__device__ __forceinline__ void load_block(const uint16_t *w, size_t base, float (&v)[16]) {
    const uint4 *p = reinterpret_cast<const uint4 *>(w + base);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uint4 u = __ldg(p + q);
        const uint32_t words[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // element 2j in the low half of word j
            v[8 * q + 2 * j] = __uint_as_float(words[j] << 16);
            v[8 * q + 2 * j + 1] = __uint_as_float(words[j] & 0xFFFF0000u);
        }
    }
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

// Largest |w| over the 16-byte vectors [0, nvec) of w (4 fp32 or 8 bf16 each).
__device__ __forceinline__ void vec_abs_max(const float *w, size_t i, float &m, bool &bad) {
    const float4 f = __ldg(reinterpret_cast<const float4 *>(w) + i);
    const float a[4] = {fabsf(f.x), fabsf(f.y), fabsf(f.z), fabsf(f.w)};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        bad |= !(a[j] <= 3.402823466e38f);  // inf or NaN
        m = a[j] > m ? a[j] : m;
    }
}
__device__ __forceinline__ void vec_abs_max(const uint16_t *w, size_t i, float &m, bool &bad) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(w) + i);
    const uint32_t words[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float a0 = __uint_as_float((words[j] << 16) & 0x7FFFFFFFu);
        const float a1 = __uint_as_float(words[j] & 0x7FFF0000u);
        bad |= !(a0 <= 3.402823466e38f) || !(a1 <= 3.402823466e38f);
        m = a0 > m ? a0 : m;
        m = a1 > m ? a1 : m;
    }
}

template <typename TW>
__global__ void __launch_bounds__(256) quant_amax_kernel(const TW *__restrict__ w, size_t nvec,
                                                         unsigned *amax_bits, unsigned *err) {
    float m = 0.0f;
    bool bad = false;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += (size_t)gridDim.x * blockDim.x)
        vec_abs_max(w, i, m, bad);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));  // non-negative floats order as integers
    if (bad) atomicOr(err, kDevErrQuantInput);
}

template <typename TW>
__global__ void __launch_bounds__(256) quant_blocks_kernel(const TW *__restrict__ w, int N, int K,
                                                           const unsigned *amax_bits, uint8_t *__restrict__ packed,
                                                           uint8_t *__restrict__ scale) {
    const int blocks_per_row = K >> 4;
    const long long nb = (long long)N * blocks_per_row;
    const float amax = __uint_as_float(*amax_bits);
    const float g = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 2688.0f);
    const float six_g = __fmul_rn(6.0f, g);
    for (long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x; b < nb; b += (long long)gridDim.x * blockDim.x) {
        const size_t base = (size_t)b * 16;  // row-major: block b covers elements [16 b, 16 b + 16)
        float v[16];
        load_block(w, base, v);
        float bmax = 0.0f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float a = fabsf(v[j]);
            bmax = a > bmax ? a : bmax;
        }
        const unsigned sc = e4m3_encode(__fdiv_rn(bmax, six_g));
        const float s_val = e4m3_decode(sc);
        const float denom = __fmul_rn(s_val, g);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const unsigned q = (s_val != 0.0f) ? e2m1_encode(__fdiv_rn(v[j], denom)) : 0u;
            if (j < 8) lo |= q << (4 * j);
            else hi |= q << (4 * (j - 8));
        }
        *reinterpret_cast<uint2 *>(packed + (size_t)b * 8) = make_uint2(lo, hi);  // element 2i in the low nibble
        scale[b] = (uint8_t)sc;
    }
}

__global__ void quant_finish_kernel(float *global_scale) {
    const float amax = *global_scale;  // holds the amax bits until now
    *global_scale = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 2688.0f);
}

template <typename TW>
cudaError_t launch_quantize(const TW *w, int N, int K, uint8_t *packed, uint8_t *scale, float *global_scale,
                            unsigned *err, int sms, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(global_scale, 0, sizeof(float), stream);
    if (e != cudaSuccess) return e;
    const size_t nvec = (size_t)N * K / (16 / sizeof(TW));  // K % 16 == 0: whole 16-byte vectors
    const long long want = (long long)((nvec + 255) / 256);
    const int grid_a = (int)(want < 8LL * sms ? want : 8LL * sms);
    quant_amax_kernel<TW><<<grid_a, 256, 0, stream>>>(w, nvec, reinterpret_cast<unsigned *>(global_scale), err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const long long nb = (long long)N * (K >> 4);
    const long long want_b = (nb + 255) / 256;
    const int grid_b = (int)(want_b < 16LL * sms ? want_b : 16LL * sms);
    quant_blocks_kernel<TW><<<grid_b, 256, 0, stream>>>(w, N, K, reinterpret_cast<const unsigned *>(global_scale),
                                                         packed, scale);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    quant_finish_kernel<<<1, 1, 0, stream>>>(global_scale);
    return cudaGetLastError();
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
