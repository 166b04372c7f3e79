/*
 * w4a8.h -- C ABI of the GB300 (sm_103a) W4A8 block-32 linear.
 *
 * The operator: y = x * W^T for a linear layer whose weights are 4-bit
 * integers in blocks of 32 along K with one fp16 scale per block, and whose
 * fp16 activations are quantised to int8 inside the kernel, per token and per
 * 32-wide block.  The pages that describe it (Google's ML Drift engine):
 *   "Що змінює ML Drift для on-device AI-інференсу на вашому телефоні?"
 *   (tech.dede.sh), section "Stage-aware оптимізація для великих мовних
 *   моделей": 4-bit weights with block size 32; prefill is compute-bound and
 *   decode memory-bound; kernels and layouts switch with the phase; decode
 *   quantises activations inside the kernel to avoid extra memory traffic.
 *   "谷歌突然开源！端侧 AI 的 GPU 底座，要变了" (m.x-techcon.com), section
 *   "对大模型，重点已经从“算得快”变成“数据少搬”": the same stage-aware
 *   kernel choice and in-kernel activation quantisation.
 * The pages leave the arithmetic open; this library implements the plainest
 * reading they support:
 *   s_x[m,b] = amax_{k in b} |x[m,k]| / 127 in fp32 (amax 0 gives 1),
 *   q[m,k]   = clamp(round_half_even(x[m,k] / s_x[m,b]), -127, 127),
 *   d[m,n,b] = sum_{k in b} w[n,k] * q[m,k]            (exact integer),
 *   y[m,n]   = fp16_rne( sum_b d[m,n,b] * (s_w[n,b] * s_x[m,b]) )  in fp32.
 * Codes and block dots are exact; the fp32 sum's order and fusion are the
 * kernel's, so y matches a sequential fp32 sum to within rounding.
 *
 * Conventions for every entry point:
 *   - fp16 tensors are passed as IEEE binary16 bit patterns (uint16_t).
 *   - Every tensor is dense row-major device memory, allocated and owned by
 *     the caller; pointers must be 16-byte aligned.
 *   - Calls are asynchronous and ordered on `stream` unless stated otherwise;
 *     nothing is allocated per call except by w4a8_linear on the prefill path
 *     (stream-ordered, see there).  Distinct streams may be used from
 *     distinct host threads.
 *   - Errors are returned, never raised: no entry point aborts, exits or
 *     traps the GPU.  Argument errors are detected before anything is
 *     launched.  W4A8_ERR_CUDA means a CUDA call or launch failed; the
 *     pending CUDA error is consumed (cudaGetLastError) when it is reported.
 */
#ifndef W4A8_H
#define W4A8_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4A8_OK = 0,
    W4A8_ERR_INVALID_VALUE = 1,   /* a size is out of range (M, N < 1, K < 32, K % 32 != 0, ...) */
    W4A8_ERR_MISALIGNED = 2,      /* a pointer is NULL or not 16-byte aligned */
    W4A8_ERR_CODE_RANGE = 3,      /* w4a8_pack saw a weight code outside [-8, 7] */
    W4A8_ERR_CUDA = 4,            /* a CUDA runtime call or kernel launch failed */
    W4A8_ERR_TIMEOUT = 5,         /* a bounded device-side wait ran out (see w4a8_get_device_status) */
    W4A8_ERR_UNSUPPORTED = 6,     /* the current device is not sm_103, or the shape exceeds a kernel limit */
    W4A8_ERR_WORKSPACE = 7        /* the workspace passed is NULL or smaller than w4a8_workspace_bytes */
} w4a8_status;

/* Kernel choice.  The pages switch kernels with the inference phase; here
 * the phase is read off M (tokens per call). */
typedef enum {
    W4A8_PATH_AUTO = 0,     /* w4a8_select_path decides */
    W4A8_PATH_DECODE = 1,   /* memory-bound GEMV, activations quantised in the kernel; M <= 8 per launch */
    W4A8_PATH_PREFILL = 2,  /* compute-bound tensor-core GEMM (tcgen05) after a quantisation pass */
    W4A8_PATH_MID = 3       /* short sequences, M <= 64, K % 256 == 0: tensor-core kernels with the weights
                               as the 128-row operand (held in tensor memory for up to 32 tokens) and the
                               tokens (padded to 16, 32 or 64) as its N, streaming the weights once, after
                               a quantisation pass */
} w4a8_path;

/* Activation of the gated pair's gate branch (w4a8_linear_gated). */
typedef enum {
    W4A8_ACT_SILU = 1,        /* g / (1 + exp(-g)) */
    W4A8_ACT_GELU_TANH = 2    /* 0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) */
} w4a8_act;

/* Human-readable name of a status code (static storage, never NULL). */
const char *w4a8_status_string(w4a8_status s);

/* Bytes of the packed weight buffer for an N x K layer: N*K/2, or 0 when
 * N < 1, K < 32 or K % 32 != 0.
 *
 * Packed layout (this library's, not the pages'): row-major, row n takes
 * K/2 bytes; byte j of a row holds weight k = 2j in its low nibble and
 * k = 2j+1 in its high nibble, each stored as w + 8 (so 0..15 encodes
 * -8..7).  One 32-weight block is therefore 16 contiguous bytes (one 128-bit
 * load), a row is K/32 such blocks, and an 8-row by 128-column tile is a
 * plain 2-D box for the tensor-memory accelerator. */
size_t w4a8_packed_bytes(int N, int K);

/* Pack int8 weight codes w_codes [N][K] (device, values in [-8, 7]) into
 * packed_w (device, w4a8_packed_bytes(N, K) bytes).
 * Synchronises `stream` so it can report W4A8_ERR_CODE_RANGE when any code is
 * out of range (packed_w then holds those codes' low 4 bits + 8 and must not
 * be used).  Meant for model load, not for the timed path. */
w4a8_status w4a8_pack(const int8_t *w_codes, int N, int K, void *packed_w,
                      cudaStream_t stream);

/* The kernel w4a8_linear would run for this shape: W4A8_PATH_DECODE for one
 * token, for up to 3 tokens when K <= 8192 and for 4 tokens when K <= 2048;
 * W4A8_PATH_MID from there to 64 tokens (when K % 256 == 0; else decode up
 * to 8 tokens); W4A8_PATH_PREFILL above (thresholds measured on GB300).
 * Returns W4A8_PATH_AUTO (0) for an invalid shape. */
int w4a8_select_path(int M, int N, int K);

/* Number of CTAs along K per 128-row tile that W4A8_PATH_MID uses for this
 * shape (1, 2, 4 or 8; a cluster whose fp32 partial tiles are summed in a
 * fixed order through distributed shared memory).  0 when the mid path does
 * not take the shape.  Informational. */
int w4a8_mid_splits(int M, int N, int K);

/* Number of CTAs along K per 128 x 128 output tile that the prefill path
 * uses for this shape: 1, 2, 4 or 8 (a thread-block cluster whose CTAs each
 * take a contiguous range of 32-blocks; their fp32 partial tiles are summed
 * in a fixed order through distributed shared memory, so results are
 * deterministic).  Short sequences leave most SMs idle with one CTA per
 * tile; this spreads K over more of them.  Returns 0 for an invalid shape.
 * Informational: w4a8_linear and w4a8_linear_ex choose it themselves. */
int w4a8_prefill_splits(int M, int N, int K);

/* Debug (host only, no device work): the launch plan of the streaming decode
 * kernel for the first slice of up to 8 tokens of this shape (gated = 1: the
 * gated kernel over 2N stacked rows).  plan, when not NULL, receives 10
 * ints: tokens in the slice, activation-code slices per lane (0: codes in
 * shared memory), K groups (warps sharing a row), weight rows per CTA, rows
 * per ring chunk, ring slots, bytes per slot, dynamic shared memory per CTA,
 * CTAs, rows per warp and pass.  Returns 1 when the kernel takes the shape,
 * 0 otherwise (including an invalid shape). */
int w4a8_debug_decode_plan(int M, int N, int K, int gated, int *plan);

/* Device workspace in bytes that w4a8_linear_ex needs for this shape and
 * path (W4A8_PATH_AUTO resolves as w4a8_select_path); 0 when none.  The
 * prefill and mid paths keep the quantised activations there. */
size_t w4a8_workspace_bytes(int M, int N, int K, int path);

/* y = W4A8 linear of x.
 *   x       [M][K] fp16, device.
 *   packed_w       packed weights from w4a8_pack (w4a8_packed_bytes(N, K) bytes).
 *   scales  [N][K/32] fp16 weight block scales s_w, device, any finite value.
 *   out     [M][N] fp16, device; must not overlap the inputs.
 * Requires M >= 1, N >= 1, K >= 32, K % 32 == 0, and x finite (results are
 * unspecified otherwise).  Asynchronous on `stream`.  When the shape takes
 * the prefill or mid path this call obtains its workspace with
 * cudaMallocAsync on `stream` and releases it with cudaFreeAsync after the
 * kernels, so it is stream-ordered; callers that must not allocate use
 * w4a8_linear_ex.  The tensor-core paths read packed_w and scales before
 * they wait for the previous kernel on the stream (programmatic dependent
 * launch): the weights must not be written by a kernel still running on
 * the stream. */
w4a8_status w4a8_linear(const uint16_t *x, const void *packed_w, const uint16_t *scales,
                        int M, int N, int K, uint16_t *out, cudaStream_t stream);

/* As w4a8_linear, with an explicit path (W4A8_PATH_*) and a caller-owned
 * device workspace of at least w4a8_workspace_bytes(M, N, K, path) bytes
 * (may be NULL when that is 0).  Allocates nothing.  The decode path runs
 * any M by launching once per 8 tokens. */
w4a8_status w4a8_linear_ex(const uint16_t *x, const void *packed_w, const uint16_t *scales,
                           int M, int N, int K, uint16_t *out, int path,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Gated pair of linears: the element-wise operators of two branches fused
 * with the fully connected operator ("Scaling On-Device GPU Inference for
 * Large Generative Models", sciencestack.ai, Figure 4 left), as in a gated
 * feed-forward block:
 *   out[m][n] = act(g) * u,  g = W4A8 linear of x_m with gate row n,
 *                            u = W4A8 linear of x_m with up row n,
 * g and u in fp32 (each exactly the plain linear's sum before its fp16
 * rounding on the fused route), act from w4a8_act, one fp16 rounding.
 *   packed_gu  w4a8_packed_bytes(2N, K) bytes: w4a8_pack of a [2N][K] code
 *              matrix whose rows 0..N-1 are the gate rows and N..2N-1 the up rows.
 *   scales_gu  [2N][K/32] fp16, same row order.
 *   out        [M][N] fp16.
 * Decode shapes (see w4a8_gated_workspace_bytes == 0) run one fused kernel
 * that streams each gate row with its up row and applies act(g)*u before the
 * only store.  Other shapes run the linear over all 2N rows into `workspace`
 * (then g and u are rounded to fp16 before the element-wise step) and an
 * element-wise kernel.  Errors as w4a8_linear_ex; W4A8_ERR_INVALID_VALUE for
 * an unknown act; W4A8_ERR_WORKSPACE when a needed workspace is missing. */
size_t w4a8_gated_workspace_bytes(int M, int N, int K);
w4a8_status w4a8_linear_gated(const uint16_t *x, const void *packed_gu, const uint16_t *scales_gu,
                              int M, int N, int K, uint16_t *out, int act,
                              void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* RMS normalisation with the residual add, quantising its output for the
 * next linear (producer-side quantisation): the residual connection and the
 * element-wise operations merged into the RMS normalisation operator
 * ("Scaling On-Device GPU Inference for Large Generative Models",
 * sciencestack.ai, Figure 4 right).  Per token row m:
 *   r = fp16(x + residual)           (fp32 sum, one rounding; r = x when residual is NULL)
 *   y = fp16(r / sqrt(mean_k(r^2) + eps) * gamma)   (fp32 arithmetic)
 *   codes, sx = the activation quantiser applied to y (as in w4a8_debug_quantize_act)
 *   x, residual      [M][K] fp16, device (residual may be NULL)
 *   gamma            [K] fp16, device
 *   residual_out     [M][K] fp16 or NULL: receives r (may alias neither input)
 *   y_out            [M][K] fp16 or NULL: receives y
 *   codes            [M][K] int8, natural k order; sx [M][K/32] fp32 -- the
 *                    input of w4a8_linear_q8.
 * eps must be finite and >= 0.  Asynchronous on `stream`. */
w4a8_status w4a8_rmsnorm_quant(const uint16_t *x, const uint16_t *residual, const uint16_t *gamma, float eps,
                               int M, int K, uint16_t *residual_out, uint16_t *y_out, int8_t *codes, float *sx,
                               cudaStream_t stream);

/* The linear on activations quantised by their producer: codes int8 [M][K]
 * and sx fp32 [M][K/32] as w4a8_rmsnorm_quant writes them (codes in
 * [-127, 127]; sx the block scales).  Same result as w4a8_linear of the fp16
 * activations these codes came from.  Decode shapes run the streaming GEMV
 * without its quantisation step; others convert the codes into the prefill
 * layout in `workspace` (w4a8_linear_q8_workspace_bytes, 0 when none is
 * needed) and run the tensor-core GEMM. */
size_t w4a8_linear_q8_workspace_bytes(int M, int N, int K);
w4a8_status w4a8_linear_q8(const int8_t *codes, const float *sx, const void *packed_w, const uint16_t *scales,
                           int M, int N, int K, uint16_t *out, void *workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/* Decode attention over an fp16 KV cache, one new token per sequence (the
 * other decode hot spot beside the linears; "Що змінює ML Drift для
 * on-device AI-інференсу на вашому телефоні?", tech.dede.sh, section
 * "Stage-aware оптимізація для великих мовних моделей").
 *   q        [B][Hq][D] fp16, device
 *   k_cache, v_cache  [B][Hkv][Lmax][D] fp16, device (this library's layout);
 *            row t of sequence b is used for t < lens[b]
 *   lens     [B] int32, device; values are clamped to [0, Lmax] (a sequence
 *            of length 0 gets zeros)
 *   out      [B][Hq][D] fp16:  out[b][h] = sum_t softmax_t(q.k_t / sqrt(D)) v_t,
 *            KV head h / (Hq/Hkv) for query head h, fp32 arithmetic.
 * Requires D in {64, 128, 256}, Hq % Hkv == 0, Hq/Hkv <= 16 and
 * Lmax <= 131072, else W4A8_ERR_INVALID_VALUE.  Sequences are split into
 * chunks (64 tokens on the tensor cores for D = 128 and 256, 128 tokens for
 * D = 64) whose partial softmax sums are merged by a second kernel in
 * `workspace` (w4a8_decode_attention_workspace_bytes; 0 when one chunk
 * covers Lmax). */
size_t w4a8_decode_attention_workspace_bytes(int B, int Hq, int Hkv, int D, int Lmax);
w4a8_status w4a8_decode_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                  const int32_t *lens, int B, int Hq, int Hkv, int D, int Lmax, uint16_t *out,
                                  void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Debug: the activation quantiser alone, through the same device routine
 * the linear kernels use.  codes [M][K] int8 and sx [M][K/32] fp32, device. */
w4a8_status w4a8_debug_quantize_act(const uint16_t *x, int M, int K, int8_t *codes,
                                    float *sx, cudaStream_t stream);

/* Debug: the per-block integer dots d[m][n][b] (int32 [M][N][K/32], device)
 * as the chosen path's kernel computes them (its debug instantiation, which
 * also stores every block dot).  `out` receives the ordinary fp16 result.
 * Workspace as for w4a8_linear_ex. */
w4a8_status w4a8_debug_block_dots(const uint16_t *x, const void *packed_w,
                                  const uint16_t *scales, int M, int N, int K,
                                  int32_t *dots, uint16_t *out, int path,
                                  void *workspace, size_t workspace_bytes,
                                  cudaStream_t stream);

/* Measurement aid (not part of the operator).  Decode is bound by reading
 * the weights from memory ("Що змінює ML Drift для on-device
 * AI-інференсу на вашому телефоні?", tech.dede.sh, section "Stage-aware
 * оптимізація для великих мовних моделей"), so the benchmark reports the
 * decode kernel against a read-only ceiling besides the copy peak: this
 * reads `bytes` (a non-zero multiple of 16) at `buf` (device, 16-byte
 * aligned) once, spread over 152 CTAs, and discards it.  mode 0 streams
 * each CTA's slice through shared memory with bulk asynchronous copies (the
 * decode kernel's weight stream); mode 1 uses 128-bit loads from every
 * thread.  sink: int[152], device, zeroed by the caller (receives one word
 * per CTA).  Asynchronous on `stream`. */
w4a8_status w4a8_debug_stream_read(const void *buf, size_t bytes, int mode, int *sink, cudaStream_t stream);

/* Prefill (tensor-core) linear that allocates nothing, for callers that
 * cannot allocate device memory: code running in a CUDA-graph node or host
 * callback, plugins of engines that own every allocation, or real-time loops
 * where an allocator call (which may synchronise, or fail under memory
 * pressure) is not allowed.  The pages have no counterpart to this entry
 * point; it exists for such callers only.
 *   Arguments, layouts and results are those of w4a8_linear_ex with
 *   W4A8_PATH_PREFILL.  The quantised activations go to a fixed 16 MiB
 *   scratch array compiled into the library; every GPU that loads the library
 *   keeps that array until the process exits.  A shape whose scratch need
 *   (w4a8_workspace_bytes(M, N, K, W4A8_PATH_PREFILL)) exceeds 16 MiB is
 *   rejected with W4A8_ERR_WORKSPACE before anything is launched.
 *   The first call on each device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 *   All calls share the one array: calls whose work overlaps on the GPU (on
 *   different streams, or from different host threads) race and must be
 *   ordered by the caller.  Each call overwrites all of the scratch it reads,
 *   so nothing from an earlier call leaks into a later one. */
w4a8_status w4a8_linear_prefill_noalloc(const uint16_t *x, const void *packed_w, const uint16_t *scales,
                                        int M, int N, int K, uint16_t *out, cudaStream_t stream);

/* Synchronises `stream`, then returns and clears the library's sticky device
 * status for the current device: W4A8_OK, or W4A8_ERR_TIMEOUT when a bounded
 * wait inside a kernel ran out since the last call (that kernel's output is
 * then invalid). */
w4a8_status w4a8_get_device_status(cudaStream_t stream);

/* Budget, in SM clock cycles, for each bounded device-side wait (default
 * about two seconds).  For tests of the timeout path; 0 restores the default. */
w4a8_status w4a8_set_wait_budget(long long cycles);

/* Test hook for the timeout path: launches one CTA that waits, within the
 * wait budget, on a shared-memory barrier that nothing completes, records
 * W4A8_ERR_TIMEOUT in the device status and returns. */
w4a8_status w4a8_debug_wait_timeout(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A8_H */
