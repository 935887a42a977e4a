// gemv_generic.cu -- NVFP4 batched GEMV for inputs the streaming kernels do not
// take (K % 256 != 0, or pointers that are not 16-byte aligned).  Plain byte
// loads, one warp per output row, up to 16 tokens per launch, fp32 FMAs and a
// fixed-order warp reduction: deterministic, and token t's result does not
// depend on the other tokens in the call.
#include "internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>

namespace nvfp4 {

__global__ void __launch_bounds__(256) gemv_generic_kernel(const GenericParams p) {
    const int lane = threadIdx.x & 31;
    const int warps_per_block = blockDim.x >> 5;
    const int half_k = p.K >> 1;
    const float gs = __ldg(p.gscale);
    for (int row = blockIdx.x * warps_per_block + (threadIdx.x >> 5); row < p.N; row += gridDim.x * warps_per_block) {
        float acc[kMaxTokensPerPass];
#pragma unroll
        for (int t = 0; t < kMaxTokensPerPass; ++t) acc[t] = 0.f;
        const uint8_t *wrow = p.w + (size_t)row * half_k;
        const uint8_t *srow = p.s + (size_t)row * (p.K >> 4);
        for (int b = lane; b < half_k; b += 32) {
            const uint32_t byte = __ldg(wrow + b);
            const uint32_t s2 = e4m3x2_to_f16x2(__ldg(srow + (b >> 3)));
            const uint32_t w2 = hmul2_u32(e2m1x2_to_f16x2_rt(byte, 0), dup_lo(s2));
            const __half2 wh = *reinterpret_cast<const __half2 *>(&w2);
            const float w0 = __low2float(wh), w1 = __high2float(wh);
            const int k = 2 * b;
#pragma unroll
            for (int t = 0; t < kMaxTokensPerPass; ++t) {
                if (t < p.n) {
                    const uint16_t *xr = p.x + (size_t)t * p.K + k;
                    const float x0 = __uint_as_float((uint32_t)__ldg(xr) << 16);
                    const float x1 = __uint_as_float((uint32_t)__ldg(xr + 1) << 16);
                    acc[t] = fmaf(x1, w1, fmaf(x0, w0, acc[t]));
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kMaxTokensPerPass; ++t) {
            float a = acc[t];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
            acc[t] = a;
        }
        // lane t writes token t (every lane holds the same reduced values)
#pragma unroll
        for (int t = 0; t < kMaxTokensPerPass; ++t) {
            if (t < p.n && lane == t) {
                __nv_bfloat16 h = __float2bfloat16_rn(acc[t] * gs);
                p.y[(size_t)t * p.N + row] = *reinterpret_cast<uint16_t *>(&h);
            }
        }
    }
}

cudaError_t launch_generic(const GenericParams &p, cudaStream_t stream) {
    const int threads = 256;
    const int warps = threads / 32;
    int blocks = (p.N + warps - 1) / warps;
    if (blocks > 65535) blocks = 65535;
    gemv_generic_kernel<<<blocks, threads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace nvfp4
