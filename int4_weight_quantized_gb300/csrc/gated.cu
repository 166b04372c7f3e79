// gated.cu -- the gated pair of linears, act(x . gate) * (x . up).
//
// "Scaling On-Device GPU Inference for Large Generative Models"
// (sciencestack.ai), Figure 4 left: element-wise operators of two branches
// are fused with the fully connected operator.  Here the two branches are
// the gate and up projections of a gated feed-forward block; their weights
// are packed as one [2N][K] matrix (gate rows over up rows) and
//   out[m][n] = act(g) * u,  g = x_m . gate_n,  u = x_m . up_n,
// with act SiLU or GELU (tanh form).
//
// Decode shapes run the streaming GEMV's gated instantiation: each CTA
// streams the gate rows of its range and the matching up rows, and the
// epilogue applies act(g)*u before the only store.  Other shapes run the
// linear over all 2N rows into a workspace and this file's element-wise
// kernel.
#include "common.cuh"
#include "kernels.h"

namespace {

__global__ void gated_combine_kernel(const uint16_t *__restrict__ h, int M, int N, int act, uint16_t *__restrict__ out) {
    const size_t total = (size_t)M * N;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const size_t m = i / (size_t)N, n = i - m * (size_t)N;
        const float g = __half2float(__ushort_as_half(h[m * 2 * N + n]));
        const float u = __half2float(__ushort_as_half(h[m * 2 * N + N + n]));
        float a;
        if (act == 1) {
            a = g / (1.0f + expf(-g));
        } else {
            const float c = 0.7978845608028654f;   // sqrt(2/pi)
            a = 0.5f * g * (1.0f + tanhf(c * (g + 0.044715f * g * g * g)));
        }
        out[i] = __half_as_ushort(__float2half_rn(a * u));
    }
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

}  // namespace

namespace w4a8_host {

bool gated_fused(int M, int N, int K) {
    return M <= 8 && gemv_stream_gated_supported(M, N, K) && gemv_stream_gated_preferred(M, N, K);
}

size_t gated_workspace_bytes(int M, int N, int K) {
    if (gated_fused(M, N, K)) return 0;
    const size_t h = align256((size_t)M * 2 * N * 2);
    return h + linear_workspace_bytes(M, 2 * N, K);
}

w4a8_status launch_gated(const uint16_t *x, const void *packed_gu, const uint16_t *scales_gu, int M, int N, int K,
                         uint16_t *out, int act, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (act != 1 && act != 2) return W4A8_ERR_INVALID_VALUE;
    if (gated_fused(M, N, K)) return launch_gemv_stream_gated(x, packed_gu, scales_gu, M, N, K, out, act, stream);
    const size_t need = gated_workspace_bytes(M, N, K);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return W4A8_ERR_WORKSPACE;
    uint16_t *h = static_cast<uint16_t *>(workspace);
    const size_t hb = align256((size_t)M * 2 * N * 2);
    w4a8_status st = run_linear_auto(x, packed_gu, scales_gu, M, 2 * N, K, h, static_cast<uint8_t *>(workspace) + hb,
                                     workspace_bytes - hb, stream);
    if (st != W4A8_OK) return st;
    const size_t total = (size_t)M * N;
    const int threads = 256;
    const int blocks = (int)((total + threads - 1) / threads < 152 * 8 ? (total + threads - 1) / threads : 152 * 8);
    gated_combine_kernel<<<blocks, threads, 0, stream>>>(h, M, N, act, out);
    return launch_status();
}

}  // namespace w4a8_host
