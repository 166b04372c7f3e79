// gemv.cu -- decode-phase W4A8 linear (M <= 8 tokens per launch).
//
// Decode is memory-bound: each weight byte is read once and the time is the
// weight stream ("Що змінює ML Drift для on-device AI-інференсу на вашому
// телефоні?", tech.dede.sh, section "Stage-aware оптимізація для великих
// мовних моделей"; "谷歌突然开源！端侧 AI 的 GPU 底座，要变了",
// m.x-techcon.com, the decode paragraph of the section on prefill and
// decode).  The same pages have decode quantise activations inside the
// kernel so they never travel through memory as a separate tensor; this
// kernel does that in shared memory.
//
// Work split:
//   - grid.x tiles the N rows (R rows per CTA); grid.y splits K into ksplit
//     ranges, and the ksplit CTAs of one row tile form a thread-block
//     cluster that sums its partial results through distributed shared memory
//     (deterministic order, no atomics, no global scratch).
//   - Each CTA quantises only its own K range (x rows are at most 8 tokens).
//   - A warp owns one "slice" of 32 consecutive K blocks; lane l owns block
//     l of the slice and keeps that block's codes for all tokens in
//     registers, then walks rows G at a time: one 128-bit load per row
//     (a whole block of 32 int4 weights), 8 dp4a per token, and one fp32
//     FMA with s_w * s_x per token.  The warp's 32 lanes read 512
//     contiguous bytes of a row per load.
//   - Packed weights are stored as w + 8, so dp4a of the unsigned nibbles
//     gives d + 8 * sum(q); the accumulator starts at 0x4B400000 - 8*sum(q),
//     which leaves the float 1.5*2^23 + d in the register: subtracting
//     1.5*2^23 yields d exactly as an fp32 value with no int-to-float
//     conversion.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace {

using namespace w4a8;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxSmem = 200 * 1024;
constexpr int kMaxKsplit = 8;

struct GemvArgs {
    const uint16_t *x;
    const uint8_t *pw;
    const uint16_t *sw;
    uint16_t *out;
    int32_t *dots;     // debug instantiation only
    int M;             // tokens in this launch (<= MT)
    int N, K, nb;
    int R;             // rows per CTA (multiple of G)
    int kbpc;          // K blocks per CTA
    int ksplit;        // CTAs per cluster along K (= gridDim.y)
};

template <int MT, int G>
struct GemvSmem {
    // Byte offsets of the shared-memory regions for kbpc blocks and R rows.
    static __host__ __device__ size_t codes_off() { return 0; }
    static __host__ __device__ size_t sx_off(int kbpc) { return (size_t)MT * kbpc * 32; }
    static __host__ __device__ size_t cb_off(int kbpc) { return sx_off(kbpc) + (size_t)MT * kbpc * 4; }
    static __host__ __device__ size_t part_off(int kbpc) { return cb_off(kbpc) + (size_t)MT * kbpc * 4; }
    static __host__ __device__ size_t sum_off(int kbpc, int R) {
        return part_off(kbpc) + (size_t)((kbpc + 31) / 32) * R * MT * 4;
    }
    static __host__ __device__ size_t bytes(int kbpc, int R) { return sum_off(kbpc, R) + (size_t)R * MT * 4; }
};

template <int MT, int G, bool DEBUG>
__global__ void __launch_bounds__(kThreads) gemv_kernel(GemvArgs a) {
    using S = GemvSmem<MT, G>;
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t *codes = reinterpret_cast<uint32_t *>(smem + S::codes_off());
    float *sxs = reinterpret_cast<float *>(smem + S::sx_off(a.kbpc));
    int *cbs = reinterpret_cast<int *>(smem + S::cb_off(a.kbpc));
    float *part = reinterpret_cast<float *>(smem + S::part_off(a.kbpc));
    float *ctasum = reinterpret_cast<float *>(smem + S::sum_off(a.kbpc, a.R));

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kb0 = blockIdx.y * a.kbpc;
    const int kbr = max(0, min(a.nb, kb0 + a.kbpc) - kb0);
    const int ksc = (kbr + 31) / 32;
    const int R = a.R;
    const int n0 = blockIdx.x * R;
    const size_t row_bytes = (size_t)a.K / 2;

    // ---- quantise x[0:M, this CTA's K range] into shared memory
    {
        const int items = MT * kbr * 4;
        for (int base = 0; base < items; base += kThreads) {
            const int i = base + tid;
            const bool act = i < items;
            int m = 0, b = 0, t = 0;
            uint4 xv = make_uint4(0u, 0u, 0u, 0u);
            if (act) {
                m = i / (kbr * 4);
                const int rem = i - m * kbr * 4;
                b = rem >> 2;
                t = rem & 3;
                if (m < a.M)
                    xv = *reinterpret_cast<const uint4 *>(a.x + (size_t)m * a.K + (size_t)(kb0 + b) * kBlock + t * 8);
            }
            Quant8 r = quant8_group4(xv);
            if (act) {
                uint32_t *cw = codes + ((size_t)m * a.kbpc + b) * 8;
                cw[2 * t] = pack_bytes4(r.q[0], r.q[2], r.q[4], r.q[6]);
                cw[2 * t + 1] = pack_bytes4(r.q[1], r.q[3], r.q[5], r.q[7]);
                if (t == 0) {
                    sxs[m * a.kbpc + b] = r.s;
                    cbs[m * a.kbpc + b] = kMagicBits - 8 * r.sum;
                }
            }
        }
    }
    __syncthreads();

    // ---- stream the weights
    const int RG = R / G;
    const int units = ksc * RG;
    uint32_t qa[MT][8];
    float sxr[MT];
    int cbr[MT];
    int cur_slice = -1;
    for (int u = warp; u < units; u += kWarps) {
        const int slice = u / RG;
        const int rg = u - slice * RG;
        const int b = slice * 32 + lane;          // block within this CTA's range
        const bool bact = b < kbr;
        if (slice != cur_slice) {
            cur_slice = slice;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (bact) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(codes + ((size_t)m * a.kbpc + b) * 8);
                    uint4 c0 = src[0], c1 = src[1];
                    qa[m][0] = c0.x; qa[m][1] = c0.y; qa[m][2] = c0.z; qa[m][3] = c0.w;
                    qa[m][4] = c1.x; qa[m][5] = c1.y; qa[m][6] = c1.z; qa[m][7] = c1.w;
                    sxr[m] = sxs[m * a.kbpc + b];
                    cbr[m] = cbs[m * a.kbpc + b];
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) qa[m][j] = 0u;
                    sxr[m] = 0.0f;
                    cbr[m] = kMagicBits;
                }
            }
        }
        uint4 wv[G];
        float swv[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int n = n0 + rg * G + g;
            if (bact && n < a.N) {
                wv[g] = ld_stream_u4(a.pw + (size_t)n * row_bytes + (size_t)(kb0 + b) * 16);
                swv[g] = __half2float(__ushort_as_half(ld_stream_u16(a.sw + (size_t)n * a.nb + kb0 + b)));
            } else {
                wv[g] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);   // weights 0
                swv[g] = 0.0f;
            }
        }
        float acc[G][MT];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const uint32_t w4[4] = {wv[g].x, wv[g].y, wv[g].z, wv[g].w};
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                lo[j] = nib_even(w4[j]);
                hi[j] = nib_odd(w4[j]);
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                int d = cbr[m];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    d = dp4a_us(lo[j], qa[m][2 * j], d);
                    d = dp4a_us(hi[j], qa[m][2 * j + 1], d);
                }
                if (DEBUG) {
                    const int n = n0 + rg * G + g;
                    if (bact && n < a.N && m < a.M)
                        a.dots[((size_t)m * a.N + n) * a.nb + kb0 + b] = d - kMagicBits;
                }
                const float fd = __int_as_float(d) - kMagic;   // exact block dot
                acc[g][m] = fd * (swv[g] * sxr[m]);
            }
        }
        // sum over the 32 lanes (blocks) of the slice
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float v = acc[g][m];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == ((g * MT + m) & 31)) part[((size_t)slice * R + rg * G + g) * MT + m] = v;
            }
    }
    __syncthreads();

    // ---- sum the slices, then the cluster's K ranges, and store fp16
    for (int i = tid; i < R * MT; i += kThreads) {
        float s = 0.0f;
        for (int sl = 0; sl < ksc; ++sl) s += part[(size_t)sl * R * MT + i];
        ctasum[i] = s;
    }
    if (a.ksplit == 1) {
        // each thread stores the sums it computed
        for (int i = tid; i < R * MT; i += kThreads) {
            const int r = i / MT, m = i - r * MT;
            const int n = n0 + r;
            if (n < a.N && m < a.M) a.out[(size_t)m * a.N + n] = __half_as_ushort(__float2half_rn(ctasum[i]));
        }
    } else {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int rank = (int)cluster.block_rank();
        for (int i = tid; i < R * MT; i += kThreads) {
            const int r = i / MT, m = i - r * MT;
            if (r % a.ksplit != rank) continue;
            float s = 0.0f;
            for (int rk = 0; rk < a.ksplit; ++rk) s += cluster.map_shared_rank(ctasum, rk)[i];
            const int n = n0 + r;
            if (n < a.N && m < a.M) a.out[(size_t)m * a.N + n] = __half_as_ushort(__float2half_rn(s));
        }
        cluster.sync();   // keep every CTA's shared memory alive until all reads are done
    }
}

struct Plan {
    int MT, G, R, ksplit, kbpc;
    size_t smem;
    dim3 grid;
};

constexpr int kSMs = 152;

// GemvSmem<MT, G>::bytes for a runtime MT (the layout does not depend on G).
size_t smem_for(int MT, int kbpc, int R) {
    return (size_t)MT * kbpc * 40 + (size_t)((kbpc + 31) / 32) * R * MT * 4 + (size_t)R * MT * 4;
}

Plan make_plan(int M, int N, int K) {
    Plan p;
    const int nb = K / 32;
    p.MT = M < 8 ? M : 8;
    p.G = p.MT <= 2 ? 4 : 2;
    // split K so each CTA quantises at most ~8K activations
    long long elems = (long long)p.MT * K;
    int ks = (int)((elems + 8191) / 8192);
    ks = ks < 1 ? 1 : (ks > kMaxKsplit ? kMaxKsplit : ks);
    p.kbpc = (nb + ks - 1) / ks;
    p.ksplit = (nb + p.kbpc - 1) / p.kbpc;
    // rows per CTA: aim at ~3 CTAs per SM
    long long target = 3LL * kSMs;
    long long rows = ((long long)N * p.ksplit + target - 1) / target;
    int R = (int)((rows + p.G - 1) / p.G) * p.G;
    if (R < p.G) R = p.G;
    if (R > 64) R = 64;
    // small N: split K further to occupy the SMs
    while ((long long)((N + R - 1) / R) * p.ksplit < 2LL * kSMs && p.ksplit < kMaxKsplit && p.kbpc > 32) {
        int ks2 = p.ksplit * 2;
        p.kbpc = (nb + ks2 - 1) / ks2;
        p.ksplit = (nb + p.kbpc - 1) / p.kbpc;
    }
    p.R = R;
    p.smem = smem_for(p.MT, p.kbpc, p.R);
    p.grid = dim3((unsigned)((N + R - 1) / R), (unsigned)p.ksplit, 1);
    return p;
}

template <int MT, int G, bool DEBUG>
w4a8_status launch_t(const Plan &p, const GemvArgs &a, cudaStream_t stream) {
    auto kern = gemv_kernel<MT, G, DEBUG>;
    // the opt-in limit is raised once per device to the most any plan asks
    // for, so concurrent calls with different plans never lower it
    static std::atomic<int> attr_done[w4a8_host::kDeviceSlots];
    const w4a8_status ast = w4a8_host::ensure_smem_limit(kern, 227 * 1024, attr_done);
    if (ast != W4A8_OK) return ast;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = p.grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)p.ksplit;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.ksplit > 1 ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    return w4a8_host::launch_status();
}

template <bool DEBUG>
w4a8_status dispatch(const Plan &p, const GemvArgs &a, cudaStream_t stream) {
    switch (p.MT) {
        case 1: return launch_t<1, 4, DEBUG>(p, a, stream);
        case 2: return launch_t<2, 4, DEBUG>(p, a, stream);
        case 3: return launch_t<3, 2, DEBUG>(p, a, stream);
        case 4: return launch_t<4, 2, DEBUG>(p, a, stream);
        case 5: return launch_t<5, 2, DEBUG>(p, a, stream);
        case 6: return launch_t<6, 2, DEBUG>(p, a, stream);
        case 7: return launch_t<7, 2, DEBUG>(p, a, stream);
        default: return launch_t<8, 2, DEBUG>(p, a, stream);
    }
}

}  // namespace

namespace w4a8_host {

bool gemv_supported(int M, int N, int K) {
    Plan p = make_plan(M < 8 ? M : 8, N, K);
    return p.smem <= (size_t)kMaxSmem;
}

w4a8_status launch_gemv(const uint16_t *x, const void *packed_w, const uint16_t *scales,
                        int M, int N, int K, uint16_t *out, int32_t *dots, cudaStream_t stream) {
    for (int m0 = 0; m0 < M; m0 += 8) {
        const int mc = (M - m0) < 8 ? (M - m0) : 8;
        Plan p = make_plan(mc, N, K);
        if (p.smem > (size_t)kMaxSmem) return W4A8_ERR_UNSUPPORTED;
        GemvArgs a;
        a.x = x + (size_t)m0 * K;
        a.pw = static_cast<const uint8_t *>(packed_w);
        a.sw = scales;
        a.out = out + (size_t)m0 * N;
        a.dots = dots ? dots + (size_t)m0 * N * (K / 32) : nullptr;
        a.M = mc;
        a.N = N;
        a.K = K;
        a.nb = K / 32;
        a.R = p.R;
        a.kbpc = p.kbpc;
        a.ksplit = p.ksplit;
        w4a8_status st = dots ? dispatch<true>(p, a, stream) : dispatch<false>(p, a, stream);
        if (st != W4A8_OK) return st;
    }
    return W4A8_OK;
}

}  // namespace w4a8_host
