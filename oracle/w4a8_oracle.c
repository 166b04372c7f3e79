/*
 * w4a8_oracle.c -- plain, slow CPU reference of the W4A8 block-32 linear.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.  It shares no
 * code with the CUDA library.  Build flags: -O2 -ffp-contract=off, no fast
 * math, so every fp32 operation below is one IEEE binary32 operation with
 * round-to-nearest-even, in the order written.
 *
 * Sources (pages on ML Drift, Google's on-device GPU inference engine):
 *   [P1] "Що змінює ML Drift для on-device AI-інференсу на вашому телефоні?"
 *        (tech.dede.sh), section "Stage-aware оптимізація для великих мовних
 *        моделей": LLM benchmarks use 4-bit weights with block size 32;
 *        decoding quantises activations inside the kernel to avoid moving
 *        data through memory.
 *   [P2] "谷歌突然开源！端侧 AI 的 GPU 底座，要变了" (m.x-techcon.com),
 *        section "对大模型，重点已经从“算得快”变成“数据少搬”": in-kernel
 *        activation quantisation during decode.
 * The pages give no formula for the quantiser or the accumulation.  The
 * reading implemented here (symmetric int8 per token and per 32-block,
 * scale amax/127 in fp32, amax 0 -> scale 1, round half to even, clamp to
 * +-127; int32 dot per block times s_w*s_x, summed in fp32 in ascending
 * block order; fp16 output rounded to nearest even) is the plainest one the
 * pages support.
 *
 * Pinned by tests/test_oracle_pins.py (closed forms, hand vectors, brute
 * force, fp64 bound, invariants).
 */
#include "w4a8_oracle.h"

#include <fenv.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define BLOCK 32

/* ---- IEEE binary16 (sign 1, exponent 5 with bias 15, fraction 10) ---- */

float oracle_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    float v;
    if (e == 0) {
        v = ldexpf((float)m, -24);                 /* zero or subnormal: m * 2^-24 */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexpf((float)(m | 0x400), e - 25);    /* (1024+m) * 2^(e-15-10) */
    }
    return sign ? -v : v;
}

uint16_t oracle_float_to_half(float f)
{
    uint16_t sign = signbit(f) ? 0x8000u : 0u;
    if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
    float a = fabsf(f);
    /* 65520 is halfway between 65504 (largest finite, odd fraction) and
     * 2^16; the tie goes to the even neighbour, which is infinity. */
    if (a >= 65520.0f) return (uint16_t)(sign | 0x7c00u);
    if (a < 0x1p-14f) {
        /* subnormal range: a = m * 2^-24 with m rounded half to even.
         * m == 1024 is the smallest normal, whose encoding is also 1024. */
        float m = nearbyintf(a * 0x1p24f);
        return (uint16_t)(sign | (uint16_t)m);
    }
    int ex;
    (void)frexpf(a, &ex);            /* a = fr * 2^ex, fr in [0.5, 1) */
    int E = ex - 1;                  /* a in [2^E, 2^(E+1)) */
    float t = nearbyintf(ldexpf(a, 10 - E));   /* in [1024, 2048] */
    if (t == 2048.0f) { t = 1024.0f; E += 1; }
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)((int)t - 1024));
}

/* ---- activation quantisation (steps a1-a3) ---- */

/* One token, one 32-wide block: amax, scale, codes.  Returns -2 if the block
 * holds a non-finite value (outside the operator's domain). */
static int quantize_block(const uint16_t *xb, int8_t *qb, float *s_out)
{
    float xf[BLOCK];
    float amax = 0.0f;
    for (int k = 0; k < BLOCK; ++k) {
        xf[k] = oracle_half_to_float(xb[k]);
        if (!isfinite(xf[k])) return -2;
        float a = fabsf(xf[k]);
        if (a > amax) amax = a;
    }
    float s = (amax == 0.0f) ? 1.0f : amax / 127.0f;
    for (int k = 0; k < BLOCK; ++k) {
        float v = xf[k] / s;              /* one fp32 division, rounded to nearest even */
        float r = nearbyintf(v);          /* ties to even in the default rounding mode */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        qb[k] = (int8_t)(int)r;
    }
    *s_out = s;
    return 0;
}

int oracle_quantize_act(const uint16_t *x, int M, int K, int8_t *q, float *sx)
{
    if (M < 0 || K <= 0 || K % BLOCK != 0) return -1;
    if (fegetround() != FE_TONEAREST) return -3;
    int nb = K / BLOCK;
    for (int m = 0; m < M; ++m)
        for (int b = 0; b < nb; ++b) {
            int rc = quantize_block(x + (size_t)m * K + (size_t)b * BLOCK,
                                    q + (size_t)m * K + (size_t)b * BLOCK,
                                    sx + (size_t)m * nb + b);
            if (rc) return rc;
        }
    return 0;
}

/* ---- per-block integer dot (step a5) ---- */

int oracle_block_dots(const int8_t *q, const int8_t *w, int M, int N, int K,
                      int32_t *d)
{
    if (M < 0 || N < 0 || K <= 0 || K % BLOCK != 0) return -1;
    int nb = K / BLOCK;
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n)
            for (int b = 0; b < nb; ++b) {
                int32_t acc = 0;
                for (int k = b * BLOCK; k < (b + 1) * BLOCK; ++k)
                    acc += (int32_t)w[(size_t)n * K + k] * (int32_t)q[(size_t)m * K + k];
                d[((size_t)m * N + n) * nb + b] = acc;
            }
    return 0;
}

/* ---- the whole linear (steps a1-a8) ---- */

int oracle_linear(const uint16_t *x, const int8_t *w, const uint16_t *sw,
                  int M, int N, int K, uint16_t *y, float *acc_out)
{
    if (M < 0 || N < 0 || K <= 0 || K % BLOCK != 0) return -1;
    int nb = K / BLOCK;
    int8_t *q = (int8_t *)malloc((size_t)K);
    float *sx = (float *)malloc(sizeof(float) * (size_t)nb);
    if (!q || !sx) { free(q); free(sx); return -4; }
    int rc = 0;
    for (int m = 0; m < M && rc == 0; ++m) {
        rc = oracle_quantize_act(x + (size_t)m * K, 1, K, q, sx);
        if (rc) break;
        for (int n = 0; n < N; ++n) {
            const int8_t *wr = w + (size_t)n * K;
            float acc = 0.0f;
            for (int b = 0; b < nb; ++b) {
                int32_t d = 0;
                for (int k = b * BLOCK; k < (b + 1) * BLOCK; ++k)
                    d += (int32_t)wr[k] * (int32_t)q[k];
                float p = oracle_half_to_float(sw[(size_t)n * nb + b]) * sx[b];
                float t = (float)d * p;   /* exact conversion: |d| <= 32*8*127 < 2^24 */
                acc = acc + t;
            }
            if (acc_out) acc_out[(size_t)m * N + n] = acc;
            y[(size_t)m * N + n] = oracle_float_to_half(acc);
        }
    }
    free(q);
    free(sx);
    return rc;
}

/* ---- gated pair (gate rows over up rows), element-wise epilogue ---- */

static double activation(int act, double g)
{
    if (act == 1) return g / (1.0 + exp(-g));
    /* tanh form of GELU; sqrt(2/pi) written out from its definition */
    const double c = sqrt(2.0 / 3.14159265358979323846);
    return 0.5 * g * (1.0 + tanh(c * (g + 0.044715 * g * g * g)));
}

int oracle_linear_gated(const uint16_t *x, const int8_t *w, const uint16_t *sw,
                        int M, int N, int K, int act, uint16_t *y)
{
    if (M < 0 || N < 0 || K <= 0 || K % BLOCK != 0 || (act != 1 && act != 2)) return -1;
    size_t cells = (size_t)M * (size_t)(2 * N);
    uint16_t *y2 = (uint16_t *)malloc(sizeof(uint16_t) * (cells ? cells : 1));
    float *acc = (float *)malloc(sizeof(float) * (cells ? cells : 1));
    if (!y2 || !acc) { free(y2); free(acc); return -4; }
    int rc = oracle_linear(x, w, sw, M, 2 * N, K, y2, acc);
    for (int m = 0; m < M && rc == 0; ++m)
        for (int n = 0; n < N; ++n) {
            double g = (double)acc[(size_t)m * 2 * N + n];
            double u = (double)acc[(size_t)m * 2 * N + N + n];
            y[(size_t)m * N + n] = oracle_float_to_half((float)(activation(act, g) * u));
        }
    free(y2);
    free(acc);
    return rc;
}

/* ---- RMS normalisation (+ residual) emitting activation codes ---- */

int oracle_rmsnorm_quant(const uint16_t *x, const uint16_t *res, const uint16_t *gamma, float eps,
                         int M, int K, uint16_t *res_out, uint16_t *y, int8_t *q, float *sx)
{
    if (M < 0 || K <= 0 || K % BLOCK != 0 || !(eps >= 0.0f)) return -1;
    uint16_t *yr = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)K);
    float *r = (float *)malloc(sizeof(float) * (size_t)K);
    if (!yr || !r) { free(yr); free(r); return -4; }
    int rc = 0;
    for (int m = 0; m < M && rc == 0; ++m) {
        double ms = 0.0;
        for (int k = 0; k < K; ++k) {
            float h = oracle_half_to_float(x[(size_t)m * K + k]);
            if (res) h = h + oracle_half_to_float(res[(size_t)m * K + k]);
            uint16_t rb = oracle_float_to_half(h);
            if (res_out) res_out[(size_t)m * K + k] = rb;
            r[k] = oracle_half_to_float(rb);
            ms += (double)r[k] * (double)r[k];
        }
        ms /= (double)K;
        double inv = 1.0 / sqrt(ms + (double)eps);
        for (int k = 0; k < K; ++k) {
            double v = (double)r[k] * inv * (double)oracle_half_to_float(gamma[k]);
            yr[k] = oracle_float_to_half((float)v);
            if (y) y[(size_t)m * K + k] = yr[k];
        }
        rc = oracle_quantize_act(yr, 1, K, q + (size_t)m * K, sx + (size_t)m * (K / BLOCK));
    }
    free(yr);
    free(r);
    return rc;
}

/* ---- decode attention (softmax(q K^T / sqrt(D)) V, grouped heads) ---- */

int oracle_decode_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *lens,
                            int B, int Hq, int Hkv, int D, int Lmax, uint16_t *out)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || Lmax <= 0) return -1;
    for (int b = 0; b < B; ++b)
        if (lens[b] < 1 || lens[b] > Lmax) return -2;
    int G = Hq / Hkv;
    double scale = 1.0 / sqrt((double)D);
    double *s = (double *)malloc(sizeof(double) * (size_t)Lmax);
    double *o = (double *)malloc(sizeof(double) * (size_t)D);
    if (!s || !o) { free(s); free(o); return -4; }
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hq; ++h) {
            int g = h / G, L = lens[b];
            const uint16_t *qh = q + ((size_t)b * Hq + h) * D;
            const uint16_t *kb = k + ((size_t)b * Hkv + g) * (size_t)Lmax * D;
            const uint16_t *vb = v + ((size_t)b * Hkv + g) * (size_t)Lmax * D;
            double m = -INFINITY;
            for (int t = 0; t < L; ++t) {
                double acc = 0.0;
                for (int d = 0; d < D; ++d)
                    acc += (double)oracle_half_to_float(qh[d]) * (double)oracle_half_to_float(kb[(size_t)t * D + d]);
                s[t] = acc * scale;
                if (s[t] > m) m = s[t];
            }
            double den = 0.0;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            for (int t = 0; t < L; ++t) {
                double p = exp(s[t] - m);
                den += p;
                for (int d = 0; d < D; ++d) o[d] += p * (double)oracle_half_to_float(vb[(size_t)t * D + d]);
            }
            for (int d = 0; d < D; ++d)
                out[((size_t)b * Hq + h) * D + d] = oracle_float_to_half((float)(o[d] / den));
        }
    free(s);
    free(o);
    return 0;
}

int oracle_linear_f64(const uint16_t *x, const int8_t *w, const uint16_t *sw,
                      int M, int N, int K, double *ref)
{
    if (M < 0 || N < 0 || K <= 0 || K % BLOCK != 0) return -1;
    int nb = K / BLOCK;
    int8_t *q = (int8_t *)malloc((size_t)K);
    float *sx = (float *)malloc(sizeof(float) * (size_t)nb);
    if (!q || !sx) { free(q); free(sx); return -4; }
    int rc = 0;
    for (int m = 0; m < M && rc == 0; ++m) {
        rc = oracle_quantize_act(x + (size_t)m * K, 1, K, q, sx);
        if (rc) break;
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int b = 0; b < nb; ++b) {
                double swd = (double)oracle_half_to_float(sw[(size_t)n * nb + b]);
                double sxd = (double)sx[b];
                for (int k = b * BLOCK; k < (b + 1) * BLOCK; ++k)
                    acc += (swd * (double)w[(size_t)n * K + k]) * (sxd * (double)q[k]);
            }
            ref[(size_t)m * N + n] = acc;
        }
    }
    free(q);
    free(sx);
    return rc;
}

/* ---- packed-weight reader ---- */

int oracle_unpack_weights(const uint8_t *packed, int N, int K, int8_t *w)
{
    if (N < 0 || K <= 0 || K % BLOCK != 0) return -1;
    size_t row_bytes = (size_t)K / 2;
    for (int n = 0; n < N; ++n)
        for (size_t j = 0; j < row_bytes; ++j) {
            uint8_t byte = packed[(size_t)n * row_bytes + j];
            w[(size_t)n * K + 2 * j] = (int8_t)((int)(byte & 0x0f) - 8);
            w[(size_t)n * K + 2 * j + 1] = (int8_t)((int)(byte >> 4) - 8);
        }
    return 0;
}
