// pack.cu -- int8 weight codes [N][K] -> the packed int4 layout of w4a8.h.
//
// Offline step (model load): the pages store LLM weights as 4-bit integers
// in blocks of 32 ("Що змінює ML Drift для on-device AI-інференсу на вашому
// телефоні?", tech.dede.sh, section "Stage-aware оптимізація для великих
// мовних моделей"); the byte layout is this library's.
#include <mutex>

#include "common.cuh"

namespace {

__device__ int g_pack_range_flag;

// One thread packs 16 consecutive codes (one 128-bit load) into 8 bytes.
__global__ void __launch_bounds__(256) pack_kernel(const int8_t *__restrict__ codes,
                                                   uint8_t *__restrict__ packed, size_t n16) {
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n16) return;
    uint4 v = *reinterpret_cast<const uint4 *>(codes + 16 * i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[2] = {0u, 0u};
    bool bad = false;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        int c = (int)(int8_t)((w[j >> 2] >> (8 * (j & 3))) & 0xffu);
        bad |= (c < -8) | (c > 7);
        uint32_t u = (uint32_t)(c + 8) & 0xfu;
        out[j >> 3] |= u << (4 * (j & 7));
    }
    if (bad) atomicOr(&g_pack_range_flag, 1);
    *reinterpret_cast<uint2 *>(packed + 8 * i) = make_uint2(out[0], out[1]);
}

std::mutex g_pack_mutex;   // the range flag is one per device; packs are serialised

}  // namespace

extern "C" w4a8_status w4a8_pack(const int8_t *w_codes, int N, int K, void *packed_w,
                                 cudaStream_t stream) {
    if (N < 1 || K < 32 || K % 32 != 0) return W4A8_ERR_INVALID_VALUE;
    if (!w4a8_host::aligned16(w_codes) || !w4a8_host::aligned16(packed_w)) return W4A8_ERR_MISALIGNED;
    std::lock_guard<std::mutex> lock(g_pack_mutex);
    cudaGetLastError();
    const int zero = 0;
    int flag = 0;
    if (cudaMemcpyToSymbolAsync(g_pack_range_flag, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return W4A8_ERR_CUDA;
    size_t n16 = (size_t)N * (size_t)K / 16;
    unsigned grid = (unsigned)((n16 + 255) / 256);
    pack_kernel<<<grid, 256, 0, stream>>>(w_codes, static_cast<uint8_t *>(packed_w), n16);
    if (w4a8_host::launch_status() != W4A8_OK) return W4A8_ERR_CUDA;
    if (cudaMemcpyFromSymbolAsync(&flag, g_pack_range_flag, sizeof(int), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return W4A8_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return W4A8_ERR_CUDA;
    return flag ? W4A8_ERR_CODE_RANGE : W4A8_OK;
}
