// kernels.h -- host-side launchers shared between the library's translation units.
#pragma once

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

#include "w4a8.h"

namespace w4a8_host {

// Activation quantiser alone, natural layout (debug entry point).
w4a8_status launch_quant_debug(const uint16_t *x, int M, int K, int8_t *codes, float *sx,
                               cudaStream_t stream);

// Prefill quantisation pass: fp16 codes [Mp][K] (k permuted within groups of
// 8) and scales [K/32][Mp]; rows M..Mp-1 zero.
w4a8_status launch_quant_prefill(const uint16_t *x, int M, int K, int Mp, uint16_t *q16, float *sx,
                                 cudaStream_t stream);

// Decode GEMV for any M (one launch per 8 tokens); `dots` non-NULL selects
// the debug instantiation that also stores every block dot.
w4a8_status launch_gemv(const uint16_t *x, const void *packed_w, const uint16_t *scales,
                        int M, int N, int K, uint16_t *out, int32_t *dots, cudaStream_t stream);

// Whether the decode GEMV can take this shape (its shared-memory plan fits).
bool gemv_supported(int M, int N, int K);

// Decode GEMV that streams weight rows through a shared-memory ring with
// bulk copies (programmatic dependent launch); supported when its
// shared-memory plan (ring + the quantised activations) fits one SM.
bool gemv_stream_supported(int M, int N, int K);
// The streaming kernel is the better decode kernel when each lane can keep
// its activation codes in registers or there are at most two tokens;
// otherwise the cluster split-K kernel (when it supports the shape) is faster.
bool gemv_stream_preferred(int M, int N, int K);
// The streaming decode kernel's launch plan for the first (up to 8-token)
// slice of M (nv = 2 for the gated kernel), as kPlanFields ints: tokens,
// code slices per lane, K groups, rows per CTA, rows per chunk, ring slots,
// bytes per slot, dynamic shared memory, CTAs, rows per warp and pass.
constexpr int kPlanFields = 10;
bool gemv_stream_plan_info(int M, int N, int K, int nv, int *out);
// Gated pair (gate rows 0..N-1 over up rows N..2N-1 of one packed matrix):
// out[m][n] = act(gate_n . x_m) * (up_n . x_m), act 1 = SiLU, 2 = GELU (tanh).
// Decode GEMV on activations quantised by their producer: codes int8 [M][K]
// (natural k order) and s_x fp32 [M][K/32].
w4a8_status launch_gemv_stream_q8(const int8_t *codes, const float *sx, const void *packed_w, const uint16_t *scales,
                                  int M, int N, int K, uint16_t *out, cudaStream_t stream);
bool gemv_stream_gated_supported(int M, int N, int K);
bool gemv_stream_gated_preferred(int M, int N, int K);
w4a8_status launch_gemv_stream_gated(const uint16_t *x, const void *packed_gu, const uint16_t *scales_gu,
                                     int M, int N, int K, uint16_t *out, int act, cudaStream_t stream);
w4a8_status launch_gemv_stream(const uint16_t *x, const void *packed_w, const uint16_t *scales,
                               int M, int N, int K, uint16_t *out, int32_t *dots, cudaStream_t stream);

// Prefill path: quantisation pass into `workspace`, then the tensor-core GEMM.
size_t prefill_workspace_bytes(int M, int N, int K);
// The GEMM alone, on activations already in the prefill layout: q16 fp16
// codes [Mp][K] (k permuted 0,4,1,5,2,6,3,7 in every 8) and sx fp32 [K/32][Mp],
// Mp = prefill_tokens_padded(M, N, K) (rows past M zero).
w4a8_status launch_prefill_gemm(const uint16_t *q16, const float *sx, const void *packed_w, const uint16_t *scales,
                                int M, int N, int K, uint16_t *out, int32_t *dots, cudaStream_t stream);

// CTAs along K per output tile of the prefill GEMM (1, 2, 4 or 8), and the
// token rows its quantised activations are padded to.
int prefill_splits(int M, int N, int K);
int prefill_tokens_padded(int M, int N, int K);

// Tensor-core linear with the weights as the 128-row MMA operand
// (gemm_mid.cu): tokens as the MMA's N, in tiles of 16, 32 or 64 (one tile,
// M <= 64: the short-sequence path) or 128 (longer sequences), after the
// quantisation pass into `workspace` (fp16 codes [Mp][K], scales [K/32][Mp],
// Mp = tc_tokens_padded(M)).  Needs K % 256 == 0.
bool tc_supported(int M, int N, int K);
bool mid_supported(int M, int N, int K);
int tc_tokens_padded(int M);
int tc_splits(int M, int N, int K);
size_t tc_workspace_bytes(int M, int N, int K);
w4a8_status launch_tc_gemm(const uint16_t *q16, const float *sx, const void *packed_w, const uint16_t *scales, int M,
                           int N, int K, uint16_t *out, int32_t *dots, cudaStream_t stream);
w4a8_status launch_tc_linear(const uint16_t *x, const void *packed_w, const uint16_t *scales, int M, int N, int K,
                             uint16_t *out, int32_t *dots, void *workspace, cudaStream_t stream);

// RMS normalisation (+ residual) emitting activation codes (norm.cu), and the
// linear on such codes (decode GEMV when it takes the shape, else conversion
// to the prefill layout + the GEMM, in the workspace).
w4a8_status launch_rmsnorm_quant(const uint16_t *x, const uint16_t *res, const uint16_t *gamma, float eps, int M, int K,
                                 uint16_t *res_out, uint16_t *y_out, int8_t *codes, float *sx, cudaStream_t stream);
size_t q8_workspace_bytes(int M, int N, int K);
w4a8_status launch_linear_q8(const int8_t *codes, const float *sx, const void *packed_w, const uint16_t *scales, int M,
                             int N, int K, uint16_t *out, void *workspace, size_t workspace_bytes, cudaStream_t stream);

// Decode attention over an fp16 KV cache (attention.cu).
bool attention_shape_ok(int B, int Hq, int Hkv, int D, int Lmax);
size_t attention_workspace_bytes(int B, int Hq, int D, int Lmax);
// tensor-core chunk kernel (attention_tc.cu): head dimension 128 or 256, up
// to 16 query heads per KV head, 64-token chunks; same chunk outputs as
// attention.cu's
bool attention_tc_supported(int D, int Hq, int Hkv);
int attention_tc_chunk();     // cached tokens per chunk of the tensor-core kernel
w4a8_status launch_attention_tc(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *lens, int B,
                                int Hq, int Hkv, int D, int Lmax, int nsplit, uint16_t *out, float *ws_o, float *ws_ml,
                                cudaStream_t stream, bool *merged);   // merged: no combine pass needed
w4a8_status launch_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *lens, int B, int Hq,
                             int Hkv, int D, int Lmax, uint16_t *out, void *workspace, size_t workspace_bytes,
                             cudaStream_t stream);

// The plain linear on the automatically chosen path (api.cu), and its
// workspace size; used by the gated pair's unfused route.
size_t linear_workspace_bytes(int M, int N, int K);
w4a8_status run_linear_auto(const uint16_t *x, const void *packed_w, const uint16_t *scales, int M, int N, int K,
                            uint16_t *out, void *workspace, size_t workspace_bytes, cudaStream_t stream);

// Gated pair of linears (gated.cu): fused decode kernel when it takes the
// shape, else the linear over 2N rows into the workspace + an element-wise pass.
bool gated_fused(int M, int N, int K);
size_t gated_workspace_bytes(int M, int N, int K);
w4a8_status launch_gated(const uint16_t *x, const void *packed_gu, const uint16_t *scales_gu, int M, int N, int K,
                         uint16_t *out, int act, void *workspace, size_t workspace_bytes, cudaStream_t stream);
w4a8_status launch_prefill(const uint16_t *x, const void *packed_w, const uint16_t *scales,
                           int M, int N, int K, uint16_t *out, int32_t *dots, void *workspace,
                           cudaStream_t stream);

// Cycle budget of every bounded device wait, and the device status word of
// the current device (nullptr if it cannot be resolved).
long long wait_budget();
int *device_status_ptr();

}  // namespace w4a8_host
