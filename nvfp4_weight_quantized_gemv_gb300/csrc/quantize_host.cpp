// quantize_host.cpp -- host NVFP4 quantizer exported as nvfp4_quantize_ref.
//
// Produces test/bench weights in the layout the GEMV consumes.  Two-level
// NVFP4: fp32 global scale g = amax / (6 * 448), one E4M3 scale per 16 k
// (nearest-even, saturating at 448), E2M1 codes (nearest, ties to the even
// mantissa, saturating at 6).  All arithmetic is fp32; the rounding to E4M3
// is done on the fp32 bit pattern and the rounding to E2M1 by comparison
// against the midpoints of the code table.  Compiled with -ffp-contract=off.
#include "../../include/nvfp4_gemv.h"

#include <cmath>
#include <cstdint>
#include <cstring>

namespace nvfp4 {
void set_last_error(const char *msg);

namespace {

uint32_t f32_bits(float f) {
    uint32_t u;
    std::memcpy(&u, &f, sizeof u);
    return u;
}

// Non-negative finite fp32 -> E4M3 code, nearest-even, saturating at 0x7E.
uint8_t e4m3_from_f32(float a) {
    if (!(a > 0.0f)) return 0;
    if (a >= 448.0f) return 0x7E;
    const uint32_t u = f32_bits(a);
    const int exp = (int)((u >> 23) & 0xFF) - 127;
    if (exp < -6) {
        // subnormal E4M3: value = m * 2^-9; a * 512 is exact in fp32
        const float m = std::nearbyint(a * 512.0f);  // default rounding: nearest-even
        return (uint8_t)m;                            // m == 8 encodes 2^-6 (e = 1, m = 0)
    }
    const uint32_t mant = u & 0x7FFFFFu;
    uint32_t top = mant >> 20;           // 3 mantissa bits kept
    const uint32_t rest = mant & 0xFFFFFu;
    const uint32_t half = 0x80000u;
    uint32_t code = ((uint32_t)(exp + 7) << 3) | top;
    if (rest > half || (rest == half && (top & 1u))) code += 1;  // may carry into the exponent
    return code > 0x7Eu ? (uint8_t)0x7E : (uint8_t)code;
}

// E4M3 code (finite, non-negative) -> fp32 value.
float e4m3_value(uint8_t c) {
    const int e = (c >> 3) & 15, m = c & 7;
    if (e == 0) return std::ldexp((float)m, -9);
    return std::ldexp(1.0f + (float)m / 8.0f, e - 7);
}

// fp32 -> E2M1 code by the code table's midpoints.  At a midpoint the even
// mantissa wins: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2,
// 3.5 -> 4, 5 -> 4.  A zero magnitude is code 0 whatever the sign.
uint8_t e2m1_from_f32(float v) {
    const float a = std::fabs(v);
    uint8_t mag;
    if (a <= 0.25f) mag = 0;
    else if (a < 0.75f) mag = 1;
    else if (a <= 1.25f) mag = 2;
    else if (a < 1.75f) mag = 3;
    else if (a <= 2.5f) mag = 4;
    else if (a < 3.5f) mag = 5;
    else if (a <= 5.0f) mag = 6;
    else mag = 7;
    if (mag == 0) return 0;
    return (v < 0.0f) ? (uint8_t)(mag | 8) : mag;
}

}  // namespace
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_quantize_ref(const float *w, int N, int K, uint8_t *w_packed, uint8_t *w_scale,
                                           float *global_scale) {
    using namespace nvfp4;
    if (!w || !w_packed || !w_scale || !global_scale) {
        set_last_error("nvfp4_quantize_ref: null pointer");
        return NVFP4_ERR_INVALID_ARG;
    }
    if (N < 1 || K < 16 || K % 16 != 0) {
        set_last_error("nvfp4_quantize_ref: need N >= 1, K >= 16 and K % 16 == 0");
        return NVFP4_ERR_INVALID_ARG;
    }
    const size_t total = (size_t)N * (size_t)K;
    float amax = 0.0f;
    for (size_t i = 0; i < total; ++i) {
        const float a = std::fabs(w[i]);
        if (!std::isfinite(a)) {
            set_last_error("nvfp4_quantize_ref: non-finite weight");
            return NVFP4_ERR_INVALID_ARG;
        }
        amax = a > amax ? a : amax;
    }
    const float g = (amax == 0.0f) ? 1.0f : amax / 2688.0f;
    const float six_g = 6.0f * g;
    *global_scale = g;
    const int blocks = K / 16;
    for (int r = 0; r < N; ++r) {
        const float *row = w + (size_t)r * K;
        uint8_t *prow = w_packed + (size_t)r * (K / 2);
        uint8_t *srow = w_scale + (size_t)r * blocks;
        for (int b = 0; b < blocks; ++b) {
            const float *blk = row + b * 16;
            float bmax = 0.0f;
            for (int j = 0; j < 16; ++j) {
                const float a = std::fabs(blk[j]);
                bmax = a > bmax ? a : bmax;
            }
            const uint8_t sc = e4m3_from_f32(bmax / six_g);
            srow[b] = sc;
            const float s_val = e4m3_value(sc);
            const float denom = s_val * g;
            for (int j = 0; j < 16; j += 2) {
                uint8_t lo = 0, hi = 0;
                if (s_val != 0.0f) {
                    lo = e2m1_from_f32(blk[j] / denom);
                    hi = e2m1_from_f32(blk[j + 1] / denom);
                }
                prow[(b * 16 + j) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
    return NVFP4_OK;
}
