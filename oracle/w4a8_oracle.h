/*
 * w4a8_oracle.h -- plain, slow CPU reference of the W4A8 block-32 linear.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link or call this code; only the
 * tests, the smoke check and the benchmark's CPU-baseline leg do.  It shares
 * no source, header, table or helper with the CUDA path.
 *
 * What the method computes, and where it comes from:
 *   - 4-bit weights grouped in blocks of 32 along K, fp16 block scales, and
 *     activations quantised inside the kernel while decoding
 *     ("Що змінює ML Drift для on-device AI-інференсу на вашому телефоні?",
 *      tech.dede.sh, section "Stage-aware оптимізація для великих мовних
 *      моделей"; "谷歌突然开源！端侧 AI 的 GPU 底座，要变了", m.x-techcon.com,
 *      section "对大模型，重点已经从“算得快”变成“数据少搬”").
 *   - The pages leave the quantiser's arithmetic open.  Reading taken here:
 *     symmetric int8 per token and per 32-wide block of K, scale amax/127 in
 *     fp32 (amax 0 gives scale 1), round half to even, clamp to [-127,127];
 *     each block's integer dot is multiplied by s_w*s_x and summed in fp32;
 *     the result is written as fp16 with round-to-nearest-even.
 *
 * All fp16 values cross this interface as their IEEE binary16 bit patterns
 * (uint16_t).  All arrays are dense row-major.  Functions return 0 on
 * success and a negative number on a bad argument.
 */
#ifndef W4A8_ORACLE_H
#define W4A8_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* IEEE binary16 <-> binary32, written from the format definition. */
float    oracle_half_to_float(uint16_t h);
uint16_t oracle_float_to_half(float f);

/* Activation quantisation: x [M][K] fp16 -> codes q [M][K] int8 and scales
 * sx [M][K/32] fp32.  K must be a positive multiple of 32. */
int oracle_quantize_act(const uint16_t *x, int M, int K, int8_t *q, float *sx);

/* Per-block integer dots: d[m][n][b] = sum_{k in block b} w[n][k]*q[m][k].
 * w [N][K] int8 weight codes, q [M][K] int8 activation codes. */
int oracle_block_dots(const int8_t *q, const int8_t *w, int M, int N, int K,
                      int32_t *d);

/* The whole linear: y [M][N] fp16 = sum_b float(d_b) * (s_w * s_x) in fp32.
 * w [N][K] int8 codes in [-8,7]; sw [N][K/32] fp16.  acc (may be NULL)
 * receives the fp32 sums before the fp16 rounding. */
int oracle_linear(const uint16_t *x, const int8_t *w, const uint16_t *sw,
                  int M, int N, int K, uint16_t *y, float *acc);

/* Gated pair of linears ("Scaling On-Device GPU Inference for Large
 * Generative Models", sciencestack.ai, Figure 4 left: element-wise operators
 * of two branches fused with a fully connected operator).  w [2N][K] and
 * sw [2N][K/32] stack the gate rows (0..N-1) over the up rows (N..2N-1);
 * g and u are the fp32 sums oracle_linear computes for rows n and N+n, and
 *   y[m][n] = fp16( act(g) * u ),   act evaluated and multiplied in fp64,
 *   rounded to fp32, then to fp16 (both round to nearest even).
 * act 1 = SiLU:            g / (1 + exp(-g))
 * act 2 = GELU, tanh form: 0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) */
int oracle_linear_gated(const uint16_t *x, const int8_t *w, const uint16_t *sw,
                        int M, int N, int K, int act, uint16_t *y);

/* RMS normalisation with the residual add, emitting the linear's activation
 * codes ("Scaling On-Device GPU Inference for Large Generative Models",
 * sciencestack.ai, Figure 4 right: the residual connection and element-wise
 * operations merged into the RMS normalisation operator; producer-side
 * quantisation of the normalised activations).  Per token row m:
 *   r[k]  = fp16( float(x[k]) + float(res[k]) )   (res may be NULL: r = x)
 *   ms    = (1/K) sum_k r[k]^2                    (fp64)
 *   y[k]  = fp16( float( r[k] / sqrt(ms + eps) * gamma[k] ) )   (fp64, then fp32, then fp16)
 *   q, sx = oracle_quantize_act(y)
 * res_out (may be NULL) receives r, the updated residual stream; y (may be
 * NULL) the normalised fp16 row.  gamma [K] fp16; eps >= 0. */
int oracle_rmsnorm_quant(const uint16_t *x, const uint16_t *res, const uint16_t *gamma, float eps,
                         int M, int K, uint16_t *res_out, uint16_t *y, int8_t *q, float *sx);

/* Decode attention over an fp16 KV cache (one new token per sequence), the
 * other decode hot spot beside the linears ("Що змінює ML Drift для
 * on-device AI-інференсу на вашому телефоні?", tech.dede.sh, section
 * "Stage-aware оптимізація для великих мовних моделей": KV cache in decode).
 * Grouped query heads: query head h reads KV head h / (Hq / Hkv).
 *   q   [B][Hq][D] fp16        k, v [B][Hkv][Lmax][D] fp16 (rows t >= lens[b] unused)
 *   lens [B], 1 <= lens[b] <= Lmax
 *   s_t = (q . k_t) / sqrt(D),  out = sum_t softmax(s)_t v_t   (all in fp64)
 *   out [B][Hq][D] fp16, rounded from fp64 through fp32. */
int oracle_decode_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *lens,
                            int B, int Hq, int Hkv, int D, int Lmax, uint16_t *out);

/* Checker: the same dequantised product in fp64,
 * ref[m][n] = sum_b sum_k (double)sw*w * (double)sx*q, with the codes and
 * activation scales of oracle_quantize_act. */
int oracle_linear_f64(const uint16_t *x, const int8_t *w, const uint16_t *sw,
                      int M, int N, int K, double *ref);

/* Reads the packed weight layout of the library's public header from its
 * written definition: row n occupies K/2 bytes; byte j holds weight k=2j in
 * its low nibble and k=2j+1 in its high nibble, each stored as w+8. */
int oracle_unpack_weights(const uint8_t *packed, int N, int K, int8_t *w);

#ifdef __cplusplus
}
#endif

#endif
