// probe.cu -- read-only HBM ceilings, measured with the two load mechanisms
// the library's kernels use, as denominators beside the copy-based peak.
//
// Mode 0 streams each CTA's contiguous slice of the buffer through a
// shared-memory ring with bulk asynchronous copies (the decode kernel's
// weight stream, L2 evict-first); mode 1 reads it with 128-bit loads from
// every thread (L1 bypass) and folds the words into a checksum.  Nothing is
// written except one word per CTA, so the bytes moved are the buffer's.
#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"

namespace {

using namespace w4a8;

constexpr int kSlot = 32768;       // bytes per bulk copy
constexpr int kSlots = 4;          // ring depth (128 KB in flight per CTA)

__global__ void __launch_bounds__(256, 1) stream_read_kernel(const uint8_t *buf, size_t bytes, int mode, int *sink,
                                                            int *status, long long budget) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full[kSlots];
    const size_t per = ((bytes / gridDim.x) + 15) & ~(size_t)15;          // this CTA's slice, 16-byte multiple
    const size_t lo = (size_t)blockIdx.x * per;
    const size_t hi = lo + per < bytes ? lo + per : bytes;
    if (mode == 0) {
        if (threadIdx.x == 0) {
            for (int s = 0; s < kSlots; ++s) mbar_init(&full[s], 1);
            fence_barrier_init();
        }
        __syncthreads();
        if (threadIdx.x != 0) return;
        uint64_t pol;
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
        int issued = 0;
        for (size_t off = lo; off < hi; off += kSlot, ++issued) {
            const int s = issued % kSlots;
            if (issued >= kSlots && !mbar_wait_bounded(&full[s], (uint32_t)((issued / kSlots - 1) & 1), budget, status))
                return;
            const uint32_t n = (uint32_t)(hi - off < (size_t)kSlot ? hi - off : (size_t)kSlot);
            mbar_arrive_expect_tx(&full[s], n);
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                ::"r"(smem_u32(smem + s * kSlot)), "l"(buf + off), "r"(n), "r"(smem_u32(&full[s])), "l"(pol) : "memory");
        }
        for (int c = (issued > kSlots ? issued - kSlots : 0); c < issued; ++c)
            mbar_wait_bounded(&full[c % kSlots], (uint32_t)((c / kSlots) & 1), budget, status);
        sink[blockIdx.x] = issued;
    } else {
        uint32_t acc = 0;
        for (size_t off = lo + (size_t)threadIdx.x * 16; off < hi; off += (size_t)blockDim.x * 16) {
            const uint4 v = ld_stream_u4(buf + off);
            acc ^= v.x ^ v.y ^ v.z ^ v.w;
        }
        acc = __reduce_xor_sync(0xffffffffu, acc);
        if ((threadIdx.x & 31) == 0) atomicXor(sink + blockIdx.x, (int)acc);
    }
}

}  // namespace

extern "C" w4a8_status w4a8_debug_stream_read(const void *buf, size_t bytes, int mode, int *sink, cudaStream_t stream) {
    if (bytes == 0 || bytes % 16 != 0 || (mode != 0 && mode != 1)) return W4A8_ERR_INVALID_VALUE;
    if (!w4a8_host::aligned16(buf) || !w4a8_host::aligned16(sink)) return W4A8_ERR_MISALIGNED;
    int *status = w4a8_host::device_status_ptr();
    if (!status) return W4A8_ERR_CUDA;
    static std::atomic<int> attr_done[w4a8_host::kDeviceSlots];
    const w4a8_status ast = w4a8_host::ensure_smem_limit(stream_read_kernel, kSlot * kSlots, attr_done);
    if (ast != W4A8_OK) return ast;
    cudaGetLastError();
    // one CTA per SM (the ring holds 128 KB)
    stream_read_kernel<<<152, 256, mode == 0 ? kSlot * kSlots : 0, stream>>>(
        static_cast<const uint8_t *>(buf), bytes, mode, sink, status, w4a8_host::wait_budget());
    return w4a8_host::launch_status();
}
