// no_alloc.cu -- prefill linear for callers that cannot allocate device memory.
//
// The tensor-core prefill path needs a scratch buffer for the quantised
// activations (fp16 codes and per-block scales).  w4a8_linear allocates it
// with cudaMallocAsync and w4a8_linear_ex takes it from the caller.  Some
// callers can do neither: code running inside a CUDA-graph node callback or a
// host function on the stream, plugins of engines that own every allocation
// and forbid others, or real-time loops where any allocator call (which may
// synchronise or fail under memory pressure) is not allowed.  For them the
// entry point below runs the same quantisation pass and GEMM on a fixed
// scratch array that lives in the library's device memory for as long as the
// library is loaded.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

// 16 MiB: enough for M = 512 tokens at K = 14336 (codes 14.7 MB + scales
// 0.9 MB).  Every GPU that loads the library holds this array until the
// process exits.
constexpr size_t kScratchBytes = 16u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.  Host code must not pass
// the array's name itself to a kernel: in host code that name is only a
// host-side stand-in, not a device address.
void *scratch_on_current_device(w4a8_status *st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        *st = W4A8_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            *st = W4A8_ERR_CUDA;
            return nullptr;
        }
        g_scratch_ptr[dev] = p;
    }
    *st = W4A8_OK;
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" w4a8_status w4a8_linear_prefill_noalloc(const uint16_t *x, const void *packed_w,
                                                   const uint16_t *scales, int M, int N, int K,
                                                   uint16_t *out, cudaStream_t stream) {
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0) return W4A8_ERR_INVALID_VALUE;
    if (!w4a8_host::aligned16(x) || !w4a8_host::aligned16(packed_w) || !w4a8_host::aligned16(scales) ||
        !w4a8_host::aligned16(out))
        return W4A8_ERR_MISALIGNED;
    if (w4a8_host::prefill_workspace_bytes(M, N, K) > kScratchBytes) return W4A8_ERR_WORKSPACE;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    if (major * 10 + minor != 103) return W4A8_ERR_UNSUPPORTED;
    w4a8_status st;
    void *scratch = scratch_on_current_device(&st);
    if (!scratch) return st;
    cudaGetLastError();
    // The quantisation pass rewrites every byte of the scratch that the GEMM
    // reads (padding rows included), so nothing left by an earlier call leaks
    // into this one and no clearing is needed.
    return w4a8_host::launch_prefill(x, packed_w, scales, M, N, K, out, nullptr, scratch, stream);
}
