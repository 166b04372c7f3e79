// quant.cu -- stand-alone activation quantisation passes.
//
// The decode GEMV quantises its activations in the kernel; the prefill GEMM
// takes them from this pass (the pages: decode quantises activations inside
// the kernel to save memory traffic, "Що змінює ML Drift для on-device
// AI-інференсу на вашому телефоні?", tech.dede.sh, section "Stage-aware
// оптимізація для великих мовних моделей").  Both use the same device
// routine, w4a8::quant8_group4.
#include "common.cuh"
#include "kernels.h"

namespace {

using namespace w4a8;

// Natural-layout codes [M][K] int8 and scales [M][K/32] fp32; 4 threads per
// 32-wide block, 8 activations each.
__global__ void __launch_bounds__(256) quant_debug_kernel(const uint16_t *__restrict__ x, int M, int K,
                                                          int8_t *__restrict__ codes, float *__restrict__ sx) {
    const int nb = K / kBlock;
    const long long items = (long long)M * nb * 4;
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    bool act = i < items;   // the grid covers whole warps; idle lanes still join the shuffles
    uint4 xv = make_uint4(0u, 0u, 0u, 0u);
    if (act) xv = *reinterpret_cast<const uint4 *>(x + 8 * i);
    Quant8 r = quant8_group4(xv);
    if (act) {
        uint2 out;
        out.x = pack_bytes4(r.q[0], r.q[1], r.q[2], r.q[3]);
        out.y = pack_bytes4(r.q[4], r.q[5], r.q[6], r.q[7]);
        *reinterpret_cast<uint2 *>(codes + 8 * i) = out;
        if ((i & 3) == 0) sx[i >> 2] = r.s;
    }
}

// Prefill pass: codes as fp16 [Mp][K] for the tensor-core GEMM, with each
// group of 8 consecutive k stored in the order [0,4,1,5,2,6,3,7] (the order
// in which the GEMM unpacks nibbles), and scales s_x transposed to
// [K/32][Mp].  Token rows M..Mp-1 are written as zeros (codes and scales).
__global__ void __launch_bounds__(256) quant_prefill_kernel(const uint16_t *__restrict__ x, int M, int K, int Mp,
                                                            uint16_t *__restrict__ q16, float *__restrict__ sx) {
    // The GEMM that reads this pass's output may start now and prefetch its
    // weights; it waits for this grid to finish before reading the codes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int nb = K / kBlock;
    const long long items = (long long)Mp * nb * 4;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const bool act = i < items;
    int m = 0, b = 0, t = 0;
    uint4 xv = make_uint4(0u, 0u, 0u, 0u);
    if (act) {
        m = (int)(i / (nb * 4));
        const int rem = (int)(i - (long long)m * nb * 4);
        b = rem >> 2;
        t = rem & 3;
        if (m < M) xv = *reinterpret_cast<const uint4 *>(x + (size_t)m * K + (size_t)b * kBlock + t * 8);
    }
    Quant8 r = quant8_group4(xv);
    if (act) {
        static constexpr int perm[8] = {0, 4, 1, 5, 2, 6, 3, 7};
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t lo = __half_as_ushort(__int2half_rn(r.q[perm[2 * j]]));
            const uint32_t hi = __half_as_ushort(__int2half_rn(r.q[perm[2 * j + 1]]));
            w[j] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4 *>(q16 + (size_t)m * K + (size_t)b * kBlock + t * 8) = make_uint4(w[0], w[1], w[2], w[3]);
        if (t == 0) sx[(size_t)b * Mp + m] = (m < M) ? r.s : 0.0f;
    }
}

}  // namespace

namespace w4a8_host {

w4a8_status launch_quant_prefill(const uint16_t *x, int M, int K, int Mp, uint16_t *q16, float *sx,
                                 cudaStream_t stream) {
    long long items = (long long)Mp * (K / 32) * 4;
    unsigned grid = (unsigned)((items + 255) / 256);
    quant_prefill_kernel<<<grid, 256, 0, stream>>>(x, M, K, Mp, q16, sx);
    return launch_status();
}


w4a8_status launch_quant_debug(const uint16_t *x, int M, int K, int8_t *codes, float *sx, cudaStream_t stream) {
    long long items = (long long)M * (K / 32) * 4;
    unsigned grid = (unsigned)((items + 255) / 256);
    quant_debug_kernel<<<grid, 256, 0, stream>>>(x, M, K, codes, sx);
    return launch_status();
}

}  // namespace w4a8_host
