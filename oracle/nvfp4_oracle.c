/*
 * NVFP4 oracle: a plain, slow, CPU-only statement of what the NVFP4 hot path
 * computes.  TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke()
 * and bench.py's cpu_baseline / reference leg may load or call this library.
 * It shares no code, header, table or helper with the CUDA path, and the CUDA
 * path never calls it.
 *
 * Sources (page title, then section or item):
 *  [TRT] "NVIDIA Ships TensorRT-LLM 0.16: Native FP4 Quantization for
 *        Blackwell B200", section "The Mathematical Breakthrough of
 *        Microscopic FP4 Scaling": the E2M1 bit split (1 sign, 2 exponent,
 *        1 mantissa bit), item 2 "Two-Level Block Scaling" (16-element
 *        micro-vectors with an FP8 scale each; groups of 16 micro-vectors
 *        share an FP16 macro-scale), item 3 "Hardware-Fused Dequantization"
 *        (scales are applied before the dot products, so the product is the
 *        plain dot product of the dequantised operands).
 *  [LCP] "llama.cpp Put Precision Policy Inside the Model. That Matters More
 *        Than W4A4", section "One model can need more than one precision"
 *        (W4A8 route for marked tensors, dense and mixture-of-experts).
 *
 * Readings where the pages are silent:
 *  - E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}; the FP8 micro-scale is E4M3;
 *    the default second level is one FP32 tensor scale amax / (6 * 448).
 *  - Rounding is to the nearest representable value, ties to the even code,
 *    saturating at the largest finite value (6 for E2M1, 448 for E4M3,
 *    65504 for FP16).  The sign of a value that rounds to zero is kept.
 *  - Encode order, all in IEEE binary32 (no contraction, no fast math):
 *        s    = amax / 2688                 (tensor scale, or per 256-group
 *                                            FP16 macro-scale, see below)
 *        t    = amax_block / 6
 *        u    = t / s
 *        e    = E4M3(u)                     (0 when s == 0)
 *        d    = value(e) * s
 *        r    = 1 / d   (0 when d == 0; clamped to the largest finite float)
 *        code = E2M1(x * r)
 *  - Codes pack two per byte, the even element in the low nibble; scales are
 *    stored row-major [rows][K/16].
 *
 * Every floating-point number here is a C float or double evaluated by the
 * host's IEEE units; build with -ffp-contract=off and without -ffast-math.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_NONFINITE 3

/* ---------------------------------------------------------------------- */
/* Element formats                                                         */
/* ---------------------------------------------------------------------- */

/* E2M1 magnitude by the three low bits of a code: exponent field (bits 2..1,
 * bias 1, field 0 is subnormal) and mantissa bit (bit 0).  [TRT] bit split. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(uint32_t code)
{
    double m = E2M1_MAG[code & 7u];
    return (code & 8u) ? -m : m;
}

/* Nearest of the 8 magnitudes by exhaustive search; on a tie the even index
 * wins (the even mantissa bit); values past 6 saturate to 6. */
uint32_t orc_e2m1_encode(float q)
{
    uint32_t sign = signbit(q) ? 8u : 0u;
    double a = fabs((double)q);
    uint32_t best = 0;
    double bestd = INFINITY;
    if (a >= 6.0)
        return sign | 7u;
    for (uint32_t i = 0; i < 8; ++i) {
        double dd = fabs(a - E2M1_MAG[i]);
        if (dd < bestd || (dd == bestd && (i & 1u) == 0)) {
            best = i;
            bestd = dd;
        }
    }
    return sign | best;
}

/* E4M3: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0;
 * exponent field 0 is subnormal m * 2^-9; S.1111.111 is NaN; no infinity. */
double orc_e4m3_value(uint32_t code)
{
    uint32_t s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    double v;
    if (e == 15u && m == 7u)
        return NAN;
    if (e == 0u)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -v : v;
}

/* Values of the 127 non-negative finite E4M3 codes 0x00..0x7E, filled once
 * from orc_e4m3_value when the library loads; they increase with the code. */
static double E4M3_POS[127];

__attribute__((constructor)) static void fill_e4m3_table(void)
{
    for (uint32_t c = 0; c <= 0x7Eu; ++c)
        E4M3_POS[c] = orc_e4m3_value(c);
}

/* Nearest finite E4M3 value, ties to the even code, saturating at 448.  The
 * non-negative codes increase with their value, so a bisection over the
 * table finds the two neighbours of |u|; the nearer one wins. */
uint32_t orc_e4m3_encode(float u)
{
    uint32_t sign = signbit(u) ? 0x80u : 0u;
    double a = fabs((double)u);
    if (a >= 448.0)
        return sign | 0x7Eu;
    uint32_t lo = 0, hi = 0x7Eu;
    while (hi - lo > 1u) { /* invariant: E4M3_POS[lo] <= a < E4M3_POS[hi] */
        uint32_t mid = (lo + hi) / 2u;
        if (E4M3_POS[mid] <= a)
            lo = mid;
        else
            hi = mid;
    }
    double dl = a - E4M3_POS[lo], dh = E4M3_POS[hi] - a;
    if (dl < dh)
        return sign | lo;
    if (dh < dl)
        return sign | hi;
    return sign | ((lo & 1u) ? hi : lo);
}

/* Element-wise encoders over arrays (same functions, OpenMP over i). */
void orc_e2m1_encode_array(const float *in, int64_t n, uint8_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = (uint8_t)orc_e2m1_encode(in[i]);
}

void orc_e4m3_encode_array(const float *in, int64_t n, uint8_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = (uint8_t)orc_e4m3_encode(in[i]);
}

/* IEEE binary16: sign bit 15, exponent bits 14..10 (bias 15), mantissa 9..0. */
double orc_fp16_value(uint32_t h)
{
    uint32_t s = (h >> 15) & 1u, e = (h >> 10) & 31u, m = h & 1023u;
    double v;
    if (e == 31u)
        return m ? NAN : (s ? -INFINITY : INFINITY);
    if (e == 0u)
        v = ldexp((double)m, -24);
    else
        v = ldexp(1.0 + (double)m / 1024.0, (int)e - 15);
    return s ? -v : v;
}

/* Nearest finite binary16 value, ties to the even code, saturating at 65504.
 * Finite non-negative codes 0x0000..0x7BFF increase with their value, so a
 * bisection finds the two neighbours of |v|. */
uint32_t orc_fp16_encode(float v)
{
    uint32_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs((double)v);
    uint32_t lo = 0, hi = 0x7BFFu;
    if (a >= orc_fp16_value(hi))
        return sign | hi;
    while (hi - lo > 1u) { /* invariant: value(lo) <= a < value(hi) */
        uint32_t mid = (lo + hi) / 2u;
        if (orc_fp16_value(mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    double dl = a - orc_fp16_value(lo), dh = orc_fp16_value(hi) - a;
    if (dl < dh)
        return sign | lo;
    if (dh < dl)
        return sign | hi;
    return sign | ((lo & 1u) ? hi : lo);
}

/* BF16 is the top half of a binary32. */
float orc_bf16_value(uint32_t b)
{
    union { uint32_t u; float f; } c;
    c.u = (b & 0xFFFFu) << 16;
    return c.f;
}

static int bf16_finite(uint16_t b) { return (b & 0x7F80u) != 0x7F80u; }

/* ---------------------------------------------------------------------- */
/* NVFP4 encode                                                            */
/* ---------------------------------------------------------------------- */

/* Reciprocal of a dequantisation step, as the encode order above states. */
static float recip_step(float d)
{
    if (d == 0.0f)
        return 0.0f;
    float r = 1.0f / d;
    if (r > FLT_MAX)
        r = FLT_MAX;
    return r;
}

/* Encode one 16-element block with second-level scale s (a float).  Writes
 * 8 packed code bytes and returns the E4M3 scale code. */
static uint32_t encode_block(const uint16_t *x, float s, uint8_t *out8)
{
    float amax_b = 0.0f;
    for (int i = 0; i < 16; ++i) {
        float a = fabsf(orc_bf16_value(x[i]));
        if (a > amax_b)
            amax_b = a;
    }
    uint32_t e = 0;
    if (s != 0.0f) {
        float t = amax_b / 6.0f;
        float u = t / s;
        e = orc_e4m3_encode(u);
    }
    float d = (float)orc_e4m3_value(e) * s;
    float r = recip_step(d);
    for (int i = 0; i < 16; i += 2) {
        uint32_t c0 = orc_e2m1_encode(orc_bf16_value(x[i]) * r);
        uint32_t c1 = orc_e2m1_encode(orc_bf16_value(x[i + 1]) * r);
        out8[i / 2] = (uint8_t)(c0 | (c1 << 4));
    }
    return e;
}

/* Per-tensor mode.  x: bf16 bits [R][ld] (first K used).  codes [R][K/2],
 * scales [R][K/16] row-major, s_g_out one float.  [TRT] item 2; the FP32
 * tensor scale amax / (6 * 448) is the task's second-level reading. */
int orc_nvfp4_encode(const uint16_t *x, int64_t R, int64_t K, int64_t ld,
                     uint8_t *codes, uint8_t *scales, float *s_g_out)
{
    if (R < 0 || K < 0 || K % 16 != 0 || ld < K)
        return ORC_ERR_ARG;
    float amax = 0.0f;
    int bad = 0;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k) {
            uint16_t b = x[r * ld + k];
            if (!bf16_finite(b))
                bad = 1;
            float a = fabsf(orc_bf16_value(b));
            if (a > amax)
                amax = a;
        }
    if (bad)
        return ORC_ERR_NONFINITE;
    float s_g = amax / 2688.0f;
    *s_g_out = s_g;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
        for (int64_t b = 0; b < K / 16; ++b)
            scales[r * (K / 16) + b] = (uint8_t)encode_block(
                x + r * ld + b * 16, s_g, codes + r * (K / 2) + b * 8);
    return ORC_OK;
}

/* The same block encode for binary32 inputs (a GEMM output, say). */
static uint32_t encode_block_f32(const float *x, float s, uint8_t *out8)
{
    float amax_b = 0.0f;
    for (int i = 0; i < 16; ++i) {
        float a = fabsf(x[i]);
        if (a > amax_b)
            amax_b = a;
    }
    uint32_t e = 0;
    if (s != 0.0f) {
        float t = amax_b / 6.0f;
        float u = t / s;
        e = orc_e4m3_encode(u);
    }
    float d = (float)orc_e4m3_value(e) * s;
    float r = recip_step(d);
    for (int i = 0; i < 16; i += 2) {
        uint32_t c0 = orc_e2m1_encode(x[i] * r);
        uint32_t c1 = orc_e2m1_encode(x[i + 1] * r);
        out8[i / 2] = (uint8_t)(c0 | (c1 << 4));
    }
    return e;
}

/* Per-tensor mode with a GIVEN second-level scale s_g (a calibrated or
 * previous-step tensor scale instead of this tensor's amax / 2688), on
 * binary32 inputs x [R][ld].  The block steps are those of
 * orc_nvfp4_encode; values beyond 6 * 448 * s_g saturate (E4M3 at 448, E2M1
 * at 6).  [TRT] item 2; the fused next-layer quantiser reading. */
int orc_nvfp4_encode_f32_scaled(const float *x, int64_t R, int64_t K, int64_t ld, float s_g,
                                uint8_t *codes, uint8_t *scales)
{
    if (R < 0 || K < 0 || K % 16 != 0 || ld < K || !(s_g >= 0.0f) || isinf(s_g))
        return ORC_ERR_ARG;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k)
            if (!isfinite(x[r * ld + k]))
                return ORC_ERR_NONFINITE;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
        for (int64_t b = 0; b < K / 16; ++b)
            scales[r * (K / 16) + b] = (uint8_t)encode_block_f32(
                x + r * ld + b * 16, s_g, codes + r * (K / 2) + b * 8);
    return ORC_OK;
}

/* Macro mode: every 256 consecutive elements of a row (16 micro-blocks) share
 * an FP16 macro-scale S = FP16(amax_256 / 2688) that replaces the tensor
 * scale.  [TRT] item 2.  macro [R][K/256] holds binary16 bits. */
int orc_nvfp4_encode_macro(const uint16_t *x, int64_t R, int64_t K, int64_t ld,
                           uint8_t *codes, uint8_t *scales, uint16_t *macro)
{
    if (R < 0 || K < 0 || K % 256 != 0 || ld < K)
        return ORC_ERR_ARG;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k)
            if (!bf16_finite(x[r * ld + k]))
                return ORC_ERR_NONFINITE;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
        for (int64_t g = 0; g < K / 256; ++g) {
            const uint16_t *xg = x + r * ld + g * 256;
            float amax = 0.0f;
            for (int i = 0; i < 256; ++i) {
                float a = fabsf(orc_bf16_value(xg[i]));
                if (a > amax)
                    amax = a;
            }
            uint32_t h = orc_fp16_encode(amax / 2688.0f);
            macro[r * (K / 256) + g] = (uint16_t)h;
            float S = (float)orc_fp16_value(h);
            for (int b = 0; b < 16; ++b)
                scales[r * (K / 16) + g * 16 + b] = (uint8_t)encode_block(
                    xg + b * 16, S, codes + r * (K / 2) + g * 128 + b * 8);
        }
    return ORC_OK;
}

/* Per-token FP8 activations for the W4A8 route: s_t = amax_row / 448, then
 * a = E4M3(x * (1 / s_t)).  [LCP] "One model can need more than one
 * precision"; per-token FP32 scale is the task's reading. */
int orc_fp8_token_encode(const uint16_t *x, int64_t R, int64_t K, int64_t ld,
                         uint8_t *a, float *s_t)
{
    if (R < 0 || K < 0 || ld < K)
        return ORC_ERR_ARG;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k)
            if (!bf16_finite(x[r * ld + k]))
                return ORC_ERR_NONFINITE;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float v = fabsf(orc_bf16_value(x[r * ld + k]));
            if (v > amax)
                amax = v;
        }
        float s = amax / 448.0f;
        s_t[r] = s;
        float rc = recip_step(s);
        for (int64_t k = 0; k < K; ++k)
            a[r * K + k] = (uint8_t)orc_e4m3_encode(orc_bf16_value(x[r * ld + k]) * rc);
    }
    return ORC_OK;
}

/* ---------------------------------------------------------------------- */
/* Dequantisation and the FP64 contraction                                 */
/* ---------------------------------------------------------------------- */

/* x_hat[r][k] = E2M1(code) * E4M3(scale) * s_g, exact in double. */
void orc_nvfp4_dequant(const uint8_t *codes, const uint8_t *scales, float s_g,
                       int64_t R, int64_t K, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k) {
            uint32_t byte = codes[r * (K / 2) + k / 2];
            uint32_t c = (k & 1) ? (byte >> 4) : (byte & 15u);
            out[r * K + k] = orc_e2m1_value(c) * orc_e4m3_value(scales[r * (K / 16) + k / 16]) * (double)s_g;
        }
}

/* Macro-mode dequantisation: the FP16 macro-scale of the element's 256-group
 * replaces the tensor scale. */
void orc_nvfp4_dequant_macro(const uint8_t *codes, const uint8_t *scales,
                             const uint16_t *macro, int64_t R, int64_t K, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k) {
            uint32_t byte = codes[r * (K / 2) + k / 2];
            uint32_t c = (k & 1) ? (byte >> 4) : (byte & 15u);
            out[r * K + k] = orc_e2m1_value(c) * orc_e4m3_value(scales[r * (K / 16) + k / 16]) *
                             orc_fp16_value(macro[r * (K / 256) + k / 256]);
        }
}

/* Unscaled value of one stored NVFP4 element: E2M1(code) * E4M3(scale). */
static double elem_cs(const uint8_t *codes, const uint8_t *scales, int64_t K, int64_t r, int64_t k)
{
    uint32_t byte = codes[r * (K / 2) + k / 2];
    uint32_t c = (k & 1) ? (byte >> 4) : (byte & 15u);
    return orc_e2m1_value(c) * orc_e4m3_value(scales[r * (K / 16) + k / 16]);
}

/* W4A4 contraction, [TRT] item 3: Y[m][n] = sum_k x_hatA[m][k] * x_hatW[n][k]
 * in double, with the two tensor scales taken out of the sum as their exact
 * double product.  rows[i] selects the output rows (all M when rows == NULL,
 * nrows == M).  Y is [nrows][N]. */
void orc_gemm_w4a4(const uint8_t *a_codes, const uint8_t *a_scales, float s_a,
                   const uint8_t *w_codes, const uint8_t *w_scales, float s_w,
                   int64_t M, int64_t N, int64_t K,
                   const int64_t *rows, int64_t nrows, double *Y)
{
    double alpha = (double)s_a * (double)s_w;
    double *arow = (double *)malloc(sizeof(double) * (size_t)(nrows * K));
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        for (int64_t k = 0; k < K; ++k)
            arow[i * K + k] = elem_cs(a_codes, a_scales, K, m, k);
    }
    (void)M;
#pragma omp parallel
    {
        double *wrow = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t k = 0; k < K; ++k)
                wrow[k] = elem_cs(w_codes, w_scales, K, n, k);
            for (int64_t i = 0; i < nrows; ++i) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += arow[i * K + k] * wrow[k];
                Y[i * N + n] = alpha * acc;
            }
        }
        free(wrow);
    }
    free(arow);
}

/* Macro-mode contraction: the same dot product with each element carrying
 * its own 256-group FP16 macro-scale. */
void orc_gemm_w4a4_macro(const uint8_t *a_codes, const uint8_t *a_scales, const uint16_t *a_macro,
                         const uint8_t *w_codes, const uint8_t *w_scales, const uint16_t *w_macro,
                         int64_t M, int64_t N, int64_t K,
                         const int64_t *rows, int64_t nrows, double *Y)
{
    double *arow = (double *)malloc(sizeof(double) * (size_t)(nrows * K));
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        for (int64_t k = 0; k < K; ++k)
            arow[i * K + k] = elem_cs(a_codes, a_scales, K, m, k) *
                              orc_fp16_value(a_macro[m * (K / 256) + k / 256]);
    }
    (void)M;
#pragma omp parallel
    {
        double *wrow = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t k = 0; k < K; ++k)
                wrow[k] = elem_cs(w_codes, w_scales, K, n, k) *
                          orc_fp16_value(w_macro[n * (K / 256) + k / 256]);
            for (int64_t i = 0; i < nrows; ++i) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += arow[i * K + k] * wrow[k];
                Y[i * N + n] = acc;
            }
        }
        free(wrow);
    }
    free(arow);
}

/* W4A8 contraction, [LCP]: Y[m][n] = sum_k (E4M3(a[m][k]) * s_t[m]) *
 * x_hatW[n][k], in double. */
void orc_gemm_w4a8(const uint8_t *a_fp8, const float *s_t,
                   const uint8_t *w_codes, const uint8_t *w_scales, float s_w,
                   int64_t M, int64_t N, int64_t K,
                   const int64_t *rows, int64_t nrows, double *Y)
{
    double *arow = (double *)malloc(sizeof(double) * (size_t)(nrows * K));
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        for (int64_t k = 0; k < K; ++k)
            arow[i * K + k] = orc_e4m3_value(a_fp8[m * K + k]) * (double)s_t[m];
    }
    (void)M;
#pragma omp parallel
    {
        double *wrow = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t k = 0; k < K; ++k)
                wrow[k] = elem_cs(w_codes, w_scales, K, n, k) * (double)s_w;
            for (int64_t i = 0; i < nrows; ++i) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += arow[i * K + k] * wrow[k];
                Y[i * N + n] = acc;
            }
        }
        free(wrow);
    }
    free(arow);
}

/* Grouped (mixture-of-experts) W4A4, [LCP]: expert e owns output rows
 * offsets[e] .. offsets[e+1]-1; output row j reads activation row
 * row_idx[j] (or j when row_idx is NULL) and expert e's weights
 * w_codes + e*N*K/2, w_scales + e*N*K/16, tensor scale s_w[e].
 * Y is [offsets[E]][N]. */
void orc_gemm_grouped_w4a4(const uint8_t *a_codes, const uint8_t *a_scales, float s_a,
                           const int32_t *row_idx, const int64_t *offsets, int64_t E,
                           const uint8_t *w_codes, const uint8_t *w_scales, const float *s_w,
                           int64_t N, int64_t K, double *Y)
{
#pragma omp parallel
    {
        double *wdec = (double *)malloc(sizeof(double) * (size_t)(N * K));
        double *arow = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(dynamic, 1)
        for (int64_t e = 0; e < E; ++e) {
            if (offsets[e + 1] <= offsets[e])
                continue;
            const uint8_t *wc = w_codes + e * N * (K / 2);
            const uint8_t *ws = w_scales + e * N * (K / 16);
            for (int64_t n = 0; n < N; ++n)
                for (int64_t k = 0; k < K; ++k)
                    wdec[n * K + k] = elem_cs(wc, ws, K, n, k);
            double alpha = (double)s_a * (double)s_w[e];
            for (int64_t j = offsets[e]; j < offsets[e + 1]; ++j) {
                int64_t m = row_idx ? (int64_t)row_idx[j] : j;
                for (int64_t k = 0; k < K; ++k)
                    arow[k] = elem_cs(a_codes, a_scales, K, m, k);
                for (int64_t n = 0; n < N; ++n) {
                    double acc = 0.0;
                    for (int64_t k = 0; k < K; ++k)
                        acc += arow[k] * wdec[n * K + k];
                    Y[j * N + n] = alpha * acc;
                }
            }
        }
        free(arow);
        free(wdec);
    }
}

/* OpenMP threads of the parallel loops (timing only: results do not depend
 * on it, every loop writes disjoint outputs). */
void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
