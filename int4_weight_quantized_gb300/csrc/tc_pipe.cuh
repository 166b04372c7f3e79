// tc_pipe.cuh -- pieces shared by the tensor-core linear kernels (gemm_mid.cu,
// gemm_small.cu): kernel arguments, programmatic-dependent-launch hooks,
// bounded waits with a CTA-wide abort flag, and the per-block fp32 scaling
// of exact integer dots read from tensor memory.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "sync.cuh"

namespace w4a8 {

struct MidArgs {
    uint16_t *out;           // [M][N] fp16
    int32_t *dots;           // debug: [M][N][nb]
    int *status;
    long long budget;
    int M, N, nb;            // blockIdx.y is the tile of NT tokens
    int splits;              // CTAs of a cluster along K; blockIdx.z is the split
    int bps;                 // 32-blocks per split (multiple of 16)
};

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Bounded wait by every lane of a warp, with one warp-wide outcome.  A failed
// wait raises the CTA's abort flag; once it is up, waits fail at once.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const MidArgs &a,
                                          volatile uint32_t *abort_flag) {
    bool ok = mbar_test_wait(bar, parity) || ((*abort_flag == 0u) && mbar_wait_bounded(bar, parity, a.budget, a.status));
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && (threadIdx.x & 31) == 0) *abort_flag = 1u;
    return ok;
}

// Single-thread bounded wait; raises the abort flag on failure.
__device__ __forceinline__ bool one_wait(uint64_t *bar, uint32_t parity, const MidArgs &a, volatile uint32_t *abort_flag) {
    if (mbar_test_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (mbar_wait_bounded(bar, parity, a.budget, a.status)) return true;
    *abort_flag = 1u;
    return false;
}

// fp32 pair ops (two lanes of work per instruction; each result is the
// correctly rounded fp32 operation, as with the scalar forms).  The compiler
// builtins let register allocation keep the pairs adjacent, so no moves are
// spent packing operands.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// acc[token pairs] += d * (s_w * s_x) for CNT consecutive tokens of one
// block (d: exact integer dots from TMEM as fp32 bit patterns; sxp: the
// block's s_x of those tokens); the debug instantiation also stores each dot.
template <int CNT, bool DEBUG>
__device__ __forceinline__ void scale_acc(float2 *acc, const uint32_t *d, float sw, const float *sxp, int n, int mbase,
                                          int b, const MidArgs &a) {
    const float2 sw2 = make_float2(sw, sw);
#pragma unroll
    for (int i = 0; i < CNT; i += 4) {
        const float4 s4 = *reinterpret_cast<const float4 *>(sxp + i);
        const float2 p01 = mul2(sw2, make_float2(s4.x, s4.y));
        const float2 p23 = mul2(sw2, make_float2(s4.z, s4.w));
        const float2 d01 = make_float2(__uint_as_float(d[i]), __uint_as_float(d[i + 1]));
        const float2 d23 = make_float2(__uint_as_float(d[i + 2]), __uint_as_float(d[i + 3]));
        acc[i / 2] = fma2(d01, p01, acc[i / 2]);
        acc[i / 2 + 1] = fma2(d23, p23, acc[i / 2 + 1]);
        if (DEBUG && n < a.N) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int m = mbase + i + v;
                if (m < a.M) a.dots[((size_t)m * a.N + n) * a.nb + b] = (int32_t)__uint_as_float(d[i + v]);
            }
        }
    }
}

}  // namespace w4a8

namespace w4a8_host {

// The 16/32-token kernel (gemm_small.cu) on tensor maps built by
// launch_tc_gemm: nt is 16 or 32, grid (N tiles, token tiles, splits).
w4a8_status launch_small_gemm(int nt, const CUtensorMap &tw, const CUtensorMap &tx, const CUtensorMap &tsw,
                              const CUtensorMap &tsx, const w4a8::MidArgs &a, dim3 grid, cudaStream_t stream);

}  // namespace w4a8_host
