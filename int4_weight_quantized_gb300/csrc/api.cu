// api.cu -- the C ABI of include/w4a8.h: argument checks, the stage-aware
// dispatcher, and the library's device status word.
//
// Stage awareness: the pages have the engine switch kernels and layouts with
// the inference phase, prefill being compute-bound and decode memory-bound
// ("Що змінює ML Drift для on-device AI-інференсу на вашому телефоні?",
// tech.dede.sh, section "Stage-aware оптимізація для великих мовних
// моделей"; "谷歌突然开源！端侧 AI 的 GPU 底座，要变了", m.x-techcon.com,
// section "对大模型，重点已经从“算得快”变成“数据少搬”").  Here the phase is
// read off M: a few tokens per call is decode, a long sequence is prefill.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"

namespace {

// Sticky device status: W4A8_OK or the first error a kernel recorded.
__device__ int g_device_status;

constexpr int kMaxDevices = 64;
std::atomic<int> g_cc[kMaxDevices];          // 0 = unknown, else major*10 + minor
std::atomic<long long> g_wait_budget{0};     // 0 = default
constexpr long long kDefaultWaitBudget = 4000000000LL;   // ~2 s at 2 GHz

int device_cc(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return -1;
    int cc = g_cc[dev].load(std::memory_order_relaxed);
    if (cc == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return -1;
        }
        cc = major * 10 + minor;
        g_cc[dev].store(cc, std::memory_order_relaxed);
    }
    return cc;
}

// The library's kernels are built for sm_103a only.
w4a8_status check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    return device_cc(dev) == 103 ? W4A8_OK : W4A8_ERR_UNSUPPORTED;
}

bool shape_ok(int M, int N, int K) { return M >= 1 && N >= 1 && K >= 32 && K % 32 == 0; }

__global__ void wait_timeout_kernel(int *status, long long budget) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        w4a8::mbar_init(&bar, 1);
        w4a8::fence_barrier_init();
    }
    __syncthreads();
    // Nothing arrives on this barrier: phase 0 never completes.
    if (threadIdx.x == 0) w4a8::mbar_wait_bounded(&bar, 0, budget, status);
    __syncthreads();
    if (threadIdx.x == 0) w4a8::mbar_inval(&bar);
}

}  // namespace

namespace w4a8_host {

long long wait_budget() {
    long long b = g_wait_budget.load(std::memory_order_relaxed);
    return b > 0 ? b : kDefaultWaitBudget;
}

int *device_status_ptr() {
    static std::mutex mu;
    static int *ptrs[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        ptrs[dev] = static_cast<int *>(p);
    }
    return ptrs[dev];
}

}  // namespace w4a8_host

using namespace w4a8_host;

extern "C" {

const char *w4a8_status_string(w4a8_status s) {
    switch (s) {
        case W4A8_OK: return "ok";
        case W4A8_ERR_INVALID_VALUE: return "invalid value (shape out of range)";
        case W4A8_ERR_MISALIGNED: return "pointer is NULL or not 16-byte aligned";
        case W4A8_ERR_CODE_RANGE: return "weight code outside [-8, 7]";
        case W4A8_ERR_CUDA: return "CUDA call or kernel launch failed";
        case W4A8_ERR_TIMEOUT: return "bounded device wait timed out";
        case W4A8_ERR_UNSUPPORTED: return "unsupported device or shape";
        case W4A8_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

size_t w4a8_packed_bytes(int N, int K) {
    if (N < 1 || K < 32 || K % 32 != 0) return 0;
    return (size_t)N * (size_t)K / 2;
}

int w4a8_select_path(int M, int N, int K) {
    if (!shape_ok(M, N, K)) return W4A8_PATH_AUTO;
    // Thresholds measured on GB300 (decode GEMV against the tensor-core
    // kernels over M = 1..64 at N x K = 8192x2048, 2048x2048, 14336x4096,
    // 4096x14336, 2048x8192): the GEMV wins at one token, and while its
    // codes stay in registers or nearly so (up to 3 tokens with K <= 8192, 4
    // tokens with K <= 2048); the tensor-core kernels from there to 64 tokens.
    const bool decode_ok = M <= 8 && (gemv_stream_supported(M, N, K) || gemv_supported(M, N, K));
    if (decode_ok && (M == 1 || (M <= 3 && K <= 8192) || (M == 4 && K <= 2048))) return W4A8_PATH_DECODE;
    if (M <= 64 && mid_supported(M, N, K)) return W4A8_PATH_MID;
    if (decode_ok) return W4A8_PATH_DECODE;
    return W4A8_PATH_PREFILL;
}

int w4a8_debug_decode_plan(int M, int N, int K, int gated, int *plan) {
    if (!shape_ok(M, N, K) || (gated != 0 && gated != 1)) return 0;
    return gemv_stream_plan_info(M, N, K, gated ? 2 : 1, plan) ? 1 : 0;
}

int w4a8_mid_splits(int M, int N, int K) {
    if (!shape_ok(M, N, K) || !mid_supported(M, N, K)) return 0;
    return tc_splits(M, N, K);
}

int w4a8_prefill_splits(int M, int N, int K) {
    if (!shape_ok(M, N, K)) return 0;
    return prefill_splits(M, N, K);
}

size_t w4a8_workspace_bytes(int M, int N, int K, int path) {
    if (!shape_ok(M, N, K)) return 0;
    if (path == W4A8_PATH_AUTO) path = w4a8_select_path(M, N, K);
    if (path == W4A8_PATH_PREFILL) return prefill_workspace_bytes(M, N, K);
    if (path == W4A8_PATH_MID) return mid_supported(M, N, K) ? tc_workspace_bytes(M, N, K) : 0;
    return 0;
}

static w4a8_status check_linear_args(const uint16_t *x, const void *packed_w, const uint16_t *scales,
                                     int M, int N, int K, const void *out) {
    if (!shape_ok(M, N, K)) return W4A8_ERR_INVALID_VALUE;
    if (!aligned16(x) || !aligned16(packed_w) || !aligned16(scales) || !aligned16(out))
        return W4A8_ERR_MISALIGNED;
    return check_device();
}

static w4a8_status run_linear(const uint16_t *x, const void *packed_w, const uint16_t *scales,
                              int M, int N, int K, uint16_t *out, int32_t *dots, int path,
                              void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (path == W4A8_PATH_AUTO) path = w4a8_select_path(M, N, K);
    cudaGetLastError();
    if (path == W4A8_PATH_DECODE) {
        const bool v1 = gemv_supported(M < 8 ? M : 8, N, K);
        if (gemv_stream_supported(M, N, K) && (!v1 || gemv_stream_preferred(M, N, K)))
            return launch_gemv_stream(x, packed_w, scales, M, N, K, out, dots, stream);
        if (!v1) return W4A8_ERR_UNSUPPORTED;
        return launch_gemv(x, packed_w, scales, M, N, K, out, dots, stream);
    }
    if (path == W4A8_PATH_PREFILL) {
        size_t need = prefill_workspace_bytes(M, N, K);
        if (need && (workspace_bytes < need || !aligned16(workspace))) return W4A8_ERR_WORKSPACE;
        return launch_prefill(x, packed_w, scales, M, N, K, out, dots, workspace, stream);
    }
    if (path == W4A8_PATH_MID) {
        if (!mid_supported(M, N, K)) return W4A8_ERR_UNSUPPORTED;
        size_t need = tc_workspace_bytes(M, N, K);
        if (workspace_bytes < need || !aligned16(workspace)) return W4A8_ERR_WORKSPACE;
        return launch_tc_linear(x, packed_w, scales, M, N, K, out, dots, workspace, stream);
    }
    return W4A8_ERR_INVALID_VALUE;
}

w4a8_status w4a8_linear(const uint16_t *x, const void *packed_w, const uint16_t *scales,
                        int M, int N, int K, uint16_t *out, cudaStream_t stream) {
    w4a8_status st = check_linear_args(x, packed_w, scales, M, N, K, out);
    if (st != W4A8_OK) return st;
    int path = w4a8_select_path(M, N, K);
    size_t need = w4a8_workspace_bytes(M, N, K, path);
    void *ws = nullptr;
    if (need) {
        if (cudaMallocAsync(&ws, need, stream) != cudaSuccess) {
            cudaGetLastError();
            return W4A8_ERR_CUDA;
        }
    }
    st = run_linear(x, packed_w, scales, M, N, K, out, nullptr, path, ws, need, stream);
    if (ws && cudaFreeAsync(ws, stream) != cudaSuccess) {
        cudaGetLastError();
        if (st == W4A8_OK) st = W4A8_ERR_CUDA;
    }
    return st;
}

w4a8_status w4a8_linear_ex(const uint16_t *x, const void *packed_w, const uint16_t *scales,
                           int M, int N, int K, uint16_t *out, int path,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    w4a8_status st = check_linear_args(x, packed_w, scales, M, N, K, out);
    if (st != W4A8_OK) return st;
    if (path < W4A8_PATH_AUTO || path > W4A8_PATH_MID) return W4A8_ERR_INVALID_VALUE;
    return run_linear(x, packed_w, scales, M, N, K, out, nullptr, path, workspace, workspace_bytes, stream);
}

size_t w4a8_gated_workspace_bytes(int M, int N, int K) {
    if (!shape_ok(M, N, K)) return 0;
    return gated_workspace_bytes(M, N, K);
}

w4a8_status w4a8_linear_gated(const uint16_t *x, const void *packed_gu, const uint16_t *scales_gu,
                              int M, int N, int K, uint16_t *out, int act,
                              void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    w4a8_status st = check_linear_args(x, packed_gu, scales_gu, M, N, K, out);
    if (st != W4A8_OK) return st;
    if (act != W4A8_ACT_SILU && act != W4A8_ACT_GELU_TANH) return W4A8_ERR_INVALID_VALUE;
    cudaGetLastError();
    return launch_gated(x, packed_gu, scales_gu, M, N, K, out, act, workspace, workspace_bytes, stream);
}

w4a8_status w4a8_rmsnorm_quant(const uint16_t *x, const uint16_t *residual, const uint16_t *gamma, float eps,
                               int M, int K, uint16_t *residual_out, uint16_t *y_out, int8_t *codes, float *sx,
                               cudaStream_t stream) {
    if (!shape_ok(M, 1, K) || !(eps >= 0.0f) || eps > 3.0e38f) return W4A8_ERR_INVALID_VALUE;
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(codes) || !aligned16(sx)) return W4A8_ERR_MISALIGNED;
    if ((residual && !aligned16(residual)) || (residual_out && !aligned16(residual_out)) || (y_out && !aligned16(y_out)))
        return W4A8_ERR_MISALIGNED;
    w4a8_status st = check_device();
    if (st != W4A8_OK) return st;
    cudaGetLastError();
    return launch_rmsnorm_quant(x, residual, gamma, eps, M, K, residual_out, y_out, codes, sx, stream);
}

size_t w4a8_linear_q8_workspace_bytes(int M, int N, int K) {
    if (!shape_ok(M, N, K)) return 0;
    return q8_workspace_bytes(M, N, K);
}

w4a8_status w4a8_linear_q8(const int8_t *codes, const float *sx, const void *packed_w, const uint16_t *scales,
                           int M, int N, int K, uint16_t *out, void *workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
    if (!shape_ok(M, N, K)) return W4A8_ERR_INVALID_VALUE;
    if (!aligned16(codes) || !aligned16(sx) || !aligned16(packed_w) || !aligned16(scales) || !aligned16(out))
        return W4A8_ERR_MISALIGNED;
    w4a8_status st = check_device();
    if (st != W4A8_OK) return st;
    cudaGetLastError();
    return launch_linear_q8(codes, sx, packed_w, scales, M, N, K, out, workspace, workspace_bytes, stream);
}

size_t w4a8_decode_attention_workspace_bytes(int B, int Hq, int Hkv, int D, int Lmax) {
    if (!attention_shape_ok(B, Hq, Hkv, D, Lmax)) return 0;
    return attention_workspace_bytes(B, Hq, D, Lmax);
}

w4a8_status w4a8_decode_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                  const int32_t *lens, int B, int Hq, int Hkv, int D, int Lmax, uint16_t *out,
                                  void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!attention_shape_ok(B, Hq, Hkv, D, Lmax)) return W4A8_ERR_INVALID_VALUE;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(lens) || !aligned16(out))
        return W4A8_ERR_MISALIGNED;
    w4a8_status st = check_device();
    if (st != W4A8_OK) return st;
    cudaGetLastError();
    return launch_attention(q, k_cache, v_cache, lens, B, Hq, Hkv, D, Lmax, out, workspace, workspace_bytes, stream);
}

w4a8_status w4a8_debug_quantize_act(const uint16_t *x, int M, int K, int8_t *codes, float *sx,
                                    cudaStream_t stream) {
    if (!shape_ok(M, 1, K)) return W4A8_ERR_INVALID_VALUE;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(sx)) return W4A8_ERR_MISALIGNED;
    w4a8_status st = check_device();
    if (st != W4A8_OK) return st;
    cudaGetLastError();
    return launch_quant_debug(x, M, K, codes, sx, stream);
}

w4a8_status w4a8_debug_block_dots(const uint16_t *x, const void *packed_w, const uint16_t *scales,
                                  int M, int N, int K, int32_t *dots, uint16_t *out, int path,
                                  void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    w4a8_status st = check_linear_args(x, packed_w, scales, M, N, K, out);
    if (st != W4A8_OK) return st;
    if (!aligned16(dots)) return W4A8_ERR_MISALIGNED;
    if (path < W4A8_PATH_AUTO || path > W4A8_PATH_MID) return W4A8_ERR_INVALID_VALUE;
    return run_linear(x, packed_w, scales, M, N, K, out, dots, path, workspace, workspace_bytes, stream);
}

w4a8_status w4a8_get_device_status(cudaStream_t stream) {
    int *p = device_status_ptr();
    if (!p) return W4A8_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    int v = 0;
    const int zero = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    return (w4a8_status)v;
}

w4a8_status w4a8_set_wait_budget(long long cycles) {
    if (cycles < 0) return W4A8_ERR_INVALID_VALUE;
    g_wait_budget.store(cycles, std::memory_order_relaxed);
    return W4A8_OK;
}

w4a8_status w4a8_debug_wait_timeout(cudaStream_t stream) {
    w4a8_status st = check_device();
    if (st != W4A8_OK) return st;
    int *p = device_status_ptr();
    if (!p) return W4A8_ERR_CUDA;
    cudaGetLastError();
    wait_timeout_kernel<<<1, 32, 0, stream>>>(p, wait_budget());
    return launch_status();
}

}  // extern "C"

namespace w4a8_host {

size_t linear_workspace_bytes(int M, int N, int K) { return w4a8_workspace_bytes(M, N, K, W4A8_PATH_AUTO); }

w4a8_status run_linear_auto(const uint16_t *x, const void *packed_w, const uint16_t *scales, int M, int N, int K,
                            uint16_t *out, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return run_linear(x, packed_w, scales, M, N, K, out, nullptr, W4A8_PATH_AUTO, workspace, workspace_bytes, stream);
}

}  // namespace w4a8_host
