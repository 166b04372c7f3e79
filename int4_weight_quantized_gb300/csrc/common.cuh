// common.cuh -- device helpers shared by the W4A8 kernels (sm_103a).
//
// Holds the one activation quantiser every kernel uses (in-kernel in the
// decode GEMV, as a pass before the prefill GEMM, and in the debug entry
// point), the int4 unpacking, and the launch-side status plumbing.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "w4a8.h"

namespace w4a8 {

constexpr int kBlock = 32;                 // weights and activations share 32-wide K blocks
constexpr float kMagic = 12582912.0f;      // 1.5 * 2^23: float whose ulp is 1
constexpr int kMagicBits = 0x4B400000;     // its bit pattern

// ---------------------------------------------------------------- int math

// Four unsigned bytes of a times four signed bytes of b, plus c.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// 128-bit streaming load of read-only data that is used once (weights).
__device__ __forceinline__ uint4 ld_stream_u4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t ld_stream_u16(const void *p) {
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// -------------------------------------------------- activation quantiser

// Block scale from the block's largest magnitude: amax/127 as one IEEE fp32
// division; an all-zero block gets scale 1.
__device__ __forceinline__ float act_scale(float amax) {
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 127.0f);
}

// One code: the fp32 quotient x/s (IEEE division), rounded half to even,
// clamped to [-127, 127].
__device__ __forceinline__ int act_code(float x, float s) {
    float r = rintf(__fdiv_rn(x, s));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return (int)r;
}

// Result of quantising the 8 consecutive activations k = 8t .. 8t+7 of one
// 32-wide block (t = 0..3 is the thread's slot in its group of 4 lanes).
struct Quant8 {
    int q[8];      // codes
    float s;       // the block's scale (same in all 4 lanes)
    int sum;       // sum of the block's 32 codes (same in all 4 lanes)
};

// Reciprocal of the block scale used by the quantiser's fast path:
// fl(127 / amax), with amax 0 mapped to 0 (every x of such a block is 0).
__device__ __forceinline__ float act_recip(float amax) { return amax == 0.0f ? 0.0f : __fdiv_rn(127.0f, amax); }

// Quantise one block held by 4 consecutive lanes (lane % 4 == t), 8 fp16
// values each.  Every lane of the warp must call this together (full-mask
// shuffles of width 4); lanes with no data pass zeros.
//
// The codes equal rint(fl(x / s)) clamped to [-127, 127], s = fl(amax / 127),
// but only the block's two scale divisions are IEEE divisions.  With
// r = fl(127 / amax) and t = fl(x * r), the three roundings (of s, r and t)
// each add a relative error of at most 2^-24, so for |x| <= amax
//   |t - x/s| <= 127 * 3.0001 * 2^-24 < 2.28e-5,
// and |fl(x/s) - x/s| <= 127 * 2^-24 < 7.6e-6, hence |t - fl(x/s)| < 2^-15.
// When t is at least 2^-14 away from every half-integer, no rounding
// boundary lies between t and fl(x/s), so rint(t) = rint(fl(x/s)); the
// elements closer than that to a boundary (one in several thousand for
// random data, and every exact tie) are divided exactly instead, each on
// its own and inline (a called routine with a stack frame cost ~0.6 us per
// launch whenever one element of the activations needed it).  In both
// cases |code| <= 127, so the clamp never changes a value.
__device__ __forceinline__ Quant8 quant8_group4(uint4 xv) {
    const __half2 *h = reinterpret_cast<const __half2 *>(&xv);
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __half22float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(f[i]));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1, 4));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2, 4));
    Quant8 r;
    r.s = act_scale(a);
    const float rc = act_recip(a);
    unsigned near = 0u;
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float t = f[i] * rc;
        const float c = rintf(t);
        if (fabsf(t - c) > 0.5f - 0x1p-14f) near |= 1u << i;
        r.q[i] = (int)c;
    }
    if (near) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (near & (1u << i)) r.q[i] = act_code(f[i], r.s);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) sum += r.q[i];
    sum += __shfl_xor_sync(0xffffffffu, sum, 1, 4);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2, 4);
    r.sum = sum;
    return r;
}

__device__ __forceinline__ uint32_t pack_bytes4(int a, int b, int c, int d) {
    return (uint32_t)(a & 0xff) | ((uint32_t)(b & 0xff) << 8) |
           ((uint32_t)(c & 0xff) << 16) | ((uint32_t)(d & 0xff) << 24);
}

// ------------------------------------------------------------ int4 unpack
//
// A packed 32-bit word holds 8 weights k = 8j .. 8j+7: byte t has k = 8j+2t
// in its low nibble and k = 8j+2t+1 in its high nibble, each as w + 8.
// Masking the low nibbles yields the unsigned bytes of the even k, shifting
// by 4 first yields the odd k.  The matching activation words therefore
// hold codes (q0, q2, q4, q6) and (q1, q3, q5, q7).
__device__ __forceinline__ uint32_t nib_even(uint32_t w) { return w & 0x0F0F0F0Fu; }
__device__ __forceinline__ uint32_t nib_odd(uint32_t w) { return (w >> 4) & 0x0F0F0F0Fu; }

}  // namespace w4a8

// ------------------------------------------------------ host-side helpers

namespace w4a8_host {

inline bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Maps the pending CUDA error, if any, to a status and clears it.
inline w4a8_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? W4A8_OK : W4A8_ERR_CUDA;
}

constexpr int kDeviceSlots = 64;   // devices a per-device table can hold

// Raises a kernel's opt-in dynamic shared-memory limit on the current device
// the first time it is launched there.  `done` is the kernel's own table of
// per-device flags; it is atomic, so first calls from several host threads
// at once are safe (each may set the attribute, which is idempotent).
template <class Kernel>
inline w4a8_status ensure_smem_limit(Kernel kern, int bytes, std::atomic<int> (&done)[kDeviceSlots]) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDeviceSlots) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    if (done[dev].load(std::memory_order_acquire)) return W4A8_OK;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    done[dev].store(1, std::memory_order_release);
    return W4A8_OK;
}

}  // namespace w4a8_host
