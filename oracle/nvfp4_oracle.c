/*
 * nvfp4_oracle.c -- plain, slow CPU oracle for the NVFP4 batched decode GEMV.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/, __graft_entry__.smoke()
 * and bench.py's cpu_baseline / reference leg may load or run anything under
 * oracle/.  It shares no code, header, table or constant with the CUDA library
 * and includes none of it.
 *
 * What it computes (the method's definition, written out):
 *
 *   Y[t, r] = bf16_rne( g * sum_{k<K} x[t, k] * E2M1(nib(r, k)) * E4M3(S[r, k/16]) )
 *
 * for tokens t < n and output rows r < N, with the sum and the product by g in
 * fp64.  This is the projection "Y = X W^T" that the atlas pull request #266
 * ("perf(decode): n>=4 tiled QKV + o_proj GEMV for NVFP4 batched decode"),
 * section "What it does", runs for a tile of decode tokens while reading the
 * projection weight once; its section "Correctness argument" and the review
 * thread's "Numeric identity" caveat fix that a batched call must agree with
 * n separate single-token (n == 1) calls, which holds here by construction
 * because every (t, r) is computed on its own.
 *
 * Encodings (the pages name NVFP4 but do not define it; these are the public
 * definitions the format is built from):
 *   - E2M1 element: 1 sign, 2 exponent, 1 mantissa bit, exponent bias 1, no
 *     inf/NaN (OCP Microscaling Formats v1.0, FP4 E2M1).  Magnitudes
 *     {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 *   - E4M3 block scale: 1 sign, 4 exponent, 3 mantissa bits, bias 7, max 448,
 *     no inf, S.1111.111 is NaN (OCP 8-bit floating point, E4M3).
 *   - One E4M3 scale per 16 consecutive elements along K, one fp32 global scale.
 *   - Layout: packed W is row-major [N][K/2] bytes, element 2i in the low
 *     nibble and element 2i+1 in the high nibble of byte i; scales row-major
 *     [N][K/16]; X row-major [n][K] bf16; Y row-major [n][N] bf16.
 *
 * Quantizer (test-data producer, see oracle_quantize): amax over the whole
 * matrix, g = amax / (6 * 448) in fp32 (1 if amax == 0), per 16-block scale
 * s = blockabsmax / (6 * g) rounded to E4M3 (nearest, ties to even, saturating
 * at 448), element code = E2M1 rounding (nearest, ties to even mantissa,
 * saturating at 6) of w / (E4M3(s) * g).  All quantizer arithmetic is fp32
 * with IEEE round-to-nearest, because the codes it emits are integers decided
 * by floating point and the product-side quantizers decide them in fp32 too.
 *
 * Build with -ffp-contract=off (no fused multiply-add contraction) so that the
 * fp32 quantizer steps and the fp64 sums round the same way on every host.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ---------------------------------------------------------------- decoding */

/* E2M1 nibble -> value.  Closed form: sign = bit 3, e = bits 2..1, m = bit 0;
 * e == 0 is the subnormal 0.5 * m, otherwise (1 + m/2) * 2^(e-1). */
double oracle_e2m1_decode(unsigned nib)
{
    nib &= 15u;
    unsigned s = (nib >> 3) & 1u, e = (nib >> 1) & 3u, m = nib & 1u;
    double mag = (e == 0) ? 0.5 * (double)m : (1.0 + 0.5 * (double)m) * ldexp(1.0, (int)e - 1);
    return s ? -mag : mag;
}

/* E4M3 byte -> value.  sign = bit 7, e = bits 6..3, m = bits 2..0;
 * e == 0 is subnormal m * 2^-9, S.1111.111 is NaN, else (1 + m/8) * 2^(e-7). */
double oracle_e4m3_decode(unsigned b)
{
    b &= 255u;
    unsigned s = (b >> 7) & 1u, e = (b >> 3) & 15u, m = b & 7u;
    double mag;
    if (e == 15u && m == 7u)
        return NAN;
    if (e == 0)
        mag = (double)m * ldexp(1.0, -9);
    else
        mag = (1.0 + (double)m / 8.0) * ldexp(1.0, (int)e - 7);
    return s ? -mag : mag;
}

/* bf16 bits -> value (bf16 is the upper half of an IEEE binary32). */
double oracle_bf16_decode(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round half to even of a non-negative double (callers pass a value divided
 * by a power of two, which is exact). */
static double round_half_even(double m)
{
    double fl = floor(m);
    double frac = m - fl;
    if (frac > 0.5)
        return fl + 1.0;
    if (frac < 0.5)
        return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* fp64 -> bf16 bits, round to nearest even, directly from the fp64 value (no
 * intermediate fp32 rounding).  bf16: 8 exponent bits (bias 127), 7 stored
 * mantissa bits; subnormal spacing 2^-133; overflow to infinity. */
uint16_t oracle_bf16_encode(double v)
{
    uint16_t sign = (signbit(v) != 0) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(v))
        return 0x7FC0u;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);          /* a = f * 2^e with f in [0.5, 1) */
    int ex = e - 1;        /* a in [2^ex, 2^(ex+1)) */
    if (ex < -126)
        ex = -126;         /* the subnormal range shares the spacing of 2^-126 */
    double spacing = ldexp(1.0, ex - 7);
    double m = round_half_even(a / spacing);
    double r = m * spacing;
    if (r >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80u);
    float rf = (float)r;   /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &rf, sizeof u);
    return (uint16_t)(sign | (uint16_t)((u >> 16) & 0x7FFFu));
}

/* ---------------------------------------------------------------- encoding */

/* Non-negative value -> E4M3 code, nearest with ties to even mantissa,
 * saturating at 448 (0x7E); never emits NaN.  Binade [2^e, 2^(e+1)) has
 * spacing 2^(e-3) for e >= -6; below 2^-6 the subnormal spacing is 2^-9. */
unsigned oracle_e4m3_encode(double a)
{
    if (!(a > 0.0))
        return 0u;         /* zero or negative zero: scales are never negative */
    if (a >= 448.0)
        return 0x7Eu;
    int e;
    frexp(a, &e);
    int ex = e - 1;
    if (ex < -6)
        ex = -6;
    double spacing = ldexp(1.0, ex - 3);
    double r = round_half_even(a / spacing) * spacing;
    if (r >= 448.0)
        return 0x7Eu;
    if (r == 0.0)
        return 0u;
    /* encode the representable value r (it may have rounded up a binade) */
    frexp(r, &e);
    int rex = e - 1;
    if (rex < -6) {        /* subnormal: r = m * 2^-9 */
        unsigned m = (unsigned)(r / ldexp(1.0, -9));
        return m & 7u;
    }
    unsigned m = (unsigned)((r / ldexp(1.0, rex) - 1.0) * 8.0);
    return ((unsigned)(rex + 7) << 3) | (m & 7u);
}

/* Value -> E2M1 nibble, nearest with ties to even mantissa, saturating at 6.
 * Spacing 0.5 below 2, 1 in [2, 4), 2 in [4, 6].  A magnitude that rounds to
 * zero gives code 0 (positive zero) whatever the sign. */
unsigned oracle_e2m1_encode(double v)
{
    double a = fabs(v);
    double r;
    if (a >= 6.0) {
        r = 6.0;
    } else {
        double spacing = (a < 2.0) ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
        r = round_half_even(a / spacing) * spacing;
    }
    unsigned mag;
    if (r == 0.0)
        return 0u;
    else if (r == 0.5)
        mag = 1u;
    else if (r == 1.0)
        mag = 2u;
    else if (r == 1.5)
        mag = 3u;
    else if (r == 2.0)
        mag = 4u;
    else if (r == 3.0)
        mag = 5u;
    else if (r == 4.0)
        mag = 6u;
    else
        mag = 7u;          /* 6.0 */
    return (v < 0.0) ? (mag | 8u) : mag;
}

/* -------------------------------------------------------------- quantizer */

/* fp32 W[N][K] -> packed [N][K/2], scales [N][K/16], global scale.
 * Returns 0 on success, 1 on bad sizes, 2 on a non-finite input. */
int oracle_quantize(const float *w, int N, int K, uint8_t *packed, uint8_t *scale, float *global_scale)
{
    if (N < 1 || K < 16 || (K % 16) != 0)
        return 1;
    float amax = 0.0f;
    for (long i = 0; i < (long)N * K; ++i) {
        float a = fabsf(w[i]);
        if (!isfinite(a))
            return 2;
        if (a > amax)
            amax = a;
    }
    float g = (amax == 0.0f) ? 1.0f : amax / 2688.0f;   /* 2688 = 6 * 448 */
    float six_g = 6.0f * g;
    *global_scale = g;
    for (int r = 0; r < N; ++r) {
        const float *row = w + (long)r * K;
        for (int b = 0; b < K / 16; ++b) {
            float bmax = 0.0f;
            for (int j = 0; j < 16; ++j) {
                float a = fabsf(row[b * 16 + j]);
                if (a > bmax)
                    bmax = a;
            }
            float s_f = bmax / six_g;
            unsigned sc = oracle_e4m3_encode((double)s_f);
            scale[(long)r * (K / 16) + b] = (uint8_t)sc;
            float s_val = (float)oracle_e4m3_decode(sc);
            float denom = s_val * g;
            for (int j = 0; j < 16; ++j) {
                int k = b * 16 + j;
                unsigned q = 0u;
                if (s_val != 0.0f) {
                    float v = row[k] / denom;
                    q = oracle_e2m1_encode((double)v);
                }
                uint8_t *byte = packed + (long)r * (K / 2) + k / 2;
                if ((k & 1) == 0)
                    *byte = (uint8_t)((*byte & 0xF0u) | q);
                else
                    *byte = (uint8_t)((*byte & 0x0Fu) | (q << 4));
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------- GEMV */

/* One output: token t, row r, as the fp64 sum times g. */
static double dot_row(const uint8_t *packed, const uint8_t *scale, float global_scale,
                      const uint16_t *x, int N, int K, int t, int r)
{
    (void)N;
    double acc = 0.0;
    for (int k = 0; k < K; ++k) {
        uint8_t byte = packed[(long)r * (K / 2) + k / 2];
        unsigned nib = (k & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 15u);
        double w = oracle_e2m1_decode(nib) * oracle_e4m3_decode(scale[(long)r * (K / 16) + k / 16]);
        acc += oracle_bf16_decode(x[(long)t * K + k]) * w;
    }
    return acc * (double)global_scale;
}

/* Y for output rows [row_begin, row_end) and all n tokens.  y64 and y16 are
 * full [n][N] arrays (either may be NULL); only the selected rows are written.
 * Returns 0 on success, 1 on bad sizes. */
int oracle_gemv_rows(const uint8_t *packed, const uint8_t *scale, float global_scale,
                     const uint16_t *x, int n, int N, int K, int row_begin, int row_end,
                     double *y64, uint16_t *y16)
{
    if (n < 0 || N < 1 || K < 16 || (K % 16) != 0 || row_begin < 0 || row_end > N || row_begin > row_end)
        return 1;
    for (int t = 0; t < n; ++t) {
        for (int r = row_begin; r < row_end; ++r) {
            double y = dot_row(packed, scale, global_scale, x, N, K, t, r);
            if (y64)
                y64[(long)t * N + r] = y;
            if (y16)
                y16[(long)t * N + r] = oracle_bf16_encode(y);
        }
    }
    return 0;
}

int oracle_gemv(const uint8_t *packed, const uint8_t *scale, float global_scale, const uint16_t *x,
                int n, int N, int K, double *y64, uint16_t *y16)
{
    return oracle_gemv_rows(packed, scale, global_scale, x, n, N, K, 0, N, y64, y16);
}

/* Y at an explicit list of (token, row) pairs; y64/y16 have `count` entries. */
int oracle_gemv_points(const uint8_t *packed, const uint8_t *scale, float global_scale,
                       const uint16_t *x, int n, int N, int K, const int *tok, const int *row,
                       int count, double *y64, uint16_t *y16)
{
    if (n < 1 || N < 1 || K < 16 || (K % 16) != 0 || count < 0)
        return 1;
    for (int i = 0; i < count; ++i) {
        if (tok[i] < 0 || tok[i] >= n || row[i] < 0 || row[i] >= N)
            return 1;
    }
    for (int i = 0; i < count; ++i) {
        double y = dot_row(packed, scale, global_scale, x, N, K, tok[i], row[i]);
        if (y64)
            y64[i] = y;
        if (y16)
            y16[i] = oracle_bf16_encode(y);
    }
    return 0;
}

/* ------------------------------------------------------------------ SwiGLU */

/* Dense SwiGLU activation of the verify FFN (rustdoc of spark_model/layers/
 * mod.rs, FfnComponent: "dense SwiGLU"; the pages give no formula, this is
 * the standard one):  h[t, f] = silu(G[t, f]) * U[t, f],  silu(a) = a / (1 +
 * exp(-a)).  gu64 holds the unrounded projection results of rows laid out
 * gate/up interleaved: column 2f of token t is G[t, f], column 2f+1 is
 * U[t, f] ([n][2F]).  h64 (may be NULL) gets the fp64 value, h16 (may be NULL)
 * its bf16 rounding (nearest even, straight from fp64).  Returns 0, or 1 on
 * bad sizes. */
int oracle_swiglu(const double *gu64, int n, int F, double *h64, uint16_t *h16)
{
    if (n < 0 || F < 1)
        return 1;
    for (int t = 0; t < n; ++t) {
        for (int f = 0; f < F; ++f) {
            double g = gu64[(long)t * 2 * F + 2 * f];
            double u = gu64[(long)t * 2 * F + 2 * f + 1];
            double h = g / (1.0 + exp(-g)) * u;
            if (h64)
                h64[(long)t * F + f] = h;
            if (h16)
                h16[(long)t * F + f] = oracle_bf16_encode(h);
        }
    }
    return 0;
}

