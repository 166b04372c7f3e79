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

}  // namespace

namespace w4a8_host {

w4a8_status launch_quant_debug(const uint16_t *x, int M, int K, int8_t *codes, float *sx, cudaStream_t stream) {
    long long items = (long long)M * (K / 32) * 4;
    unsigned grid = (unsigned)((items + 255) / 256);
    quant_debug_kernel<<<grid, 256, 0, stream>>>(x, M, K, codes, sx);
    return launch_status();
}

}  // namespace w4a8_host
