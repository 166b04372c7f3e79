// norm.cu -- RMS normalisation with the residual add, emitting the linear's
// activation codes, and the conversion of such codes to the prefill layout.
//
// "Scaling On-Device GPU Inference for Large Generative Models"
// (sciencestack.ai), Figure 4 right: the residual connection and element-wise
// operations are merged into the RMS normalisation operator.  Here that
// operator also quantises its output for the next linear (producer-side
// quantisation), so the linear reads int8 codes and block scales instead of
// re-reading and re-quantising fp16 activations.  Per token row:
//   r = fp16(x + res)                       (the updated residual stream)
//   y = fp16(r / sqrt(mean(r^2) + eps) * gamma)
//   codes, s_x = the activation quantiser (quant8_group4) applied to y.
#include "common.cuh"
#include "kernels.h"

namespace {

using namespace w4a8;

constexpr int NT = 256;   // threads per row; thread i takes the 8-value groups i, i+256, ...

__device__ __forceinline__ uint4 residual_group(const uint16_t *x, const uint16_t *res, size_t off) {
    uint4 xv = *reinterpret_cast<const uint4 *>(x + off);
    if (!res) return xv;
    const uint4 rv = *reinterpret_cast<const uint4 *>(res + off);
    const __half2 *a = reinterpret_cast<const __half2 *>(&xv);
    const __half2 *b = reinterpret_cast<const __half2 *>(&rv);
    uint4 o;
    __half2 *c = reinterpret_cast<__half2 *>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // fp32 sum of the two fp16 values, one rounding to fp16
        const float2 fa = __half22float2(a[i]), fb = __half22float2(b[i]);
        c[i] = __floats2half2_rn(fa.x + fb.x, fa.y + fb.y);
    }
    return o;
}

__global__ void __launch_bounds__(NT) rmsnorm_quant_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ res,
                                                           const uint16_t *__restrict__ gamma, float eps, int K,
                                                           uint16_t *__restrict__ res_out, uint16_t *__restrict__ y_out,
                                                           int8_t *__restrict__ codes, float *__restrict__ sx) {
    __shared__ float part[NT / 32];
    // Programmatic dependent launch: the next kernel on the stream (the
    // linear on these codes) may start now and issue its weight copies; all
    // this kernel reads may come from the kernel before it, so it waits for
    // that one first.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int m = blockIdx.x;
    const int groups = K / 8;
    const size_t row = (size_t)m * K;
    // pass 1: residual stream and sum of squares (fp32)
    float ss = 0.0f;
    for (int g = threadIdx.x; g < groups; g += NT) {
        const uint4 r = residual_group(x, res, row + (size_t)g * 8);
        if (res_out) *reinterpret_cast<uint4 *>(res_out + row + (size_t)g * 8) = r;
        const __half2 *h = reinterpret_cast<const __half2 *>(&r);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(h[i]);
            ss = fmaf(f.x, f.x, ss);
            ss = fmaf(f.y, f.y, ss);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) tot += part[w];
    const float inv = __fdiv_rn(1.0f, sqrtf(__fdiv_rn(tot, (float)K) + eps));
    // pass 2: normalise, round to fp16, quantise (4 consecutive lanes hold one 32-block)
    for (int g0 = 0; g0 < groups; g0 += NT) {
        const int g = g0 + threadIdx.x;
        const bool act = g < groups;
        uint4 yv = make_uint4(0u, 0u, 0u, 0u);
        if (act) {
            const uint4 r = residual_group(x, res, row + (size_t)g * 8);
            const uint4 gv = *reinterpret_cast<const uint4 *>(gamma + (size_t)g * 8);
            const __half2 *h = reinterpret_cast<const __half2 *>(&r);
            const __half2 *gm = reinterpret_cast<const __half2 *>(&gv);
            __half2 *yo = reinterpret_cast<__half2 *>(&yv);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(h[i]), gg = __half22float2(gm[i]);
                yo[i] = __floats2half2_rn(f.x * inv * gg.x, f.y * inv * gg.y);
            }
            if (y_out) *reinterpret_cast<uint4 *>(y_out + row + (size_t)g * 8) = yv;
        }
        const Quant8 q = quant8_group4(yv);    // whole warp: groups are lane-consecutive, 4 per block
        if (act) {
            const uint32_t lo = pack_bytes4(q.q[0], q.q[1], q.q[2], q.q[3]);
            const uint32_t hi = pack_bytes4(q.q[4], q.q[5], q.q[6], q.q[7]);
            *reinterpret_cast<uint2 *>(codes + row + (size_t)g * 8) = make_uint2(lo, hi);
            if ((g & 3) == 0) sx[(size_t)m * (K / 32) + g / 4] = q.s;
        }
    }
}

// int8 codes [M][K] (natural k order) + s_x [M][K/32] -> the prefill GEMM's
// layout: fp16 codes [Mp][K] with k permuted 0,4,1,5,2,6,3,7 in every 8, and
// s_x transposed to [K/32][Mp]; rows M..Mp-1 zero.
__global__ void codes_to_prefill_kernel(const int8_t *__restrict__ codes, const float *__restrict__ sxin, int M, int K,
                                        int Mp, uint16_t *__restrict__ q16, float *__restrict__ sx) {
    const int nb = K / 32;
    const long long items = (long long)Mp * nb * 4;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= items) return;
    const int m = (int)(i / (nb * 4));
    const int rem = (int)(i - (long long)m * nb * 4);
    const int b = rem >> 2, t = rem & 3;
    int8_t c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (m < M) {
        const uint2 v = *reinterpret_cast<const uint2 *>(codes + (size_t)m * K + (size_t)b * 32 + t * 8);
        const uint32_t w[2] = {v.x, v.y};
#pragma unroll
        for (int j = 0; j < 8; ++j) c[j] = (int8_t)((w[j >> 2] >> (8 * (j & 3))) & 0xffu);
    }
    static constexpr int perm[8] = {0, 4, 1, 5, 2, 6, 3, 7};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t lo = __half_as_ushort(__int2half_rn(c[perm[2 * j]]));
        const uint32_t hi = __half_as_ushort(__int2half_rn(c[perm[2 * j + 1]]));
        o[j] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4 *>(q16 + (size_t)m * K + (size_t)b * 32 + t * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    if (t == 0) sx[(size_t)b * Mp + m] = (m < M) ? sxin[(size_t)m * nb + b] : 0.0f;
}

}  // namespace

namespace w4a8_host {

w4a8_status launch_rmsnorm_quant(const uint16_t *x, const uint16_t *res, const uint16_t *gamma, float eps, int M, int K,
                                 uint16_t *res_out, uint16_t *y_out, int8_t *codes, float *sx, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)M, 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, rmsnorm_quant_kernel, x, res, gamma, eps, K, res_out, y_out, codes, sx) != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    return launch_status();
}

size_t q8_workspace_bytes(int M, int N, int K) {
    if (M <= 8 && gemv_stream_supported(M, N, K)) return 0;
    return prefill_workspace_bytes(M, N, K);
}

w4a8_status launch_linear_q8(const int8_t *codes, const float *sx, const void *packed_w, const uint16_t *scales, int M,
                             int N, int K, uint16_t *out, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (M <= 8 && gemv_stream_supported(M, N, K))
        return launch_gemv_stream_q8(codes, sx, packed_w, scales, M, N, K, out, stream);
    const size_t need = prefill_workspace_bytes(M, N, K);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return W4A8_ERR_WORKSPACE;
    const int mp = prefill_tokens_padded(M, N, K);
    uint16_t *q16 = static_cast<uint16_t *>(workspace);
    float *sxt = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + (size_t)mp * K * 2);
    const long long items = (long long)mp * (K / 32) * 4;
    codes_to_prefill_kernel<<<(unsigned)((items + 255) / 256), 256, 0, stream>>>(codes, sx, M, K, mp, q16, sxt);
    w4a8_status st = launch_status();
    if (st != W4A8_OK) return st;
    return launch_prefill_gemm(q16, sxt, packed_w, scales, M, N, K, out, nullptr, stream);
}

}  // namespace w4a8_host
