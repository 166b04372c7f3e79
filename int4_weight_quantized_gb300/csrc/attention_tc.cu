// attention_tc.cu -- decode attention over an fp16 KV cache on the
// 5th-generation tensor cores (head dimension 128 or 256).
//
// Decode reads, besides the weights, the KV cache of every sequence once per
// new token ("Що змінює ML Drift для on-device AI-інференсу на вашому
// телефоні?", tech.dede.sh, section "Stage-aware оптимізація для великих
// мовних моделей": fp16 KV cache, 640 tokens of context).  Same operation,
// layout and chunking as attention.cu: k and v [B][Hkv][Lmax][D] fp16, q and
// out [B][Hq][D], query head h reads KV head h / (Hq / Hkv); one CTA per
// (sequence, KV head, chunk of 64 cached tokens: small enough that three
// CTAs fit an SM at D = 256, so a decode batch's chunks are all resident at
// once); a chunk leaves (max m, sum l, unnormalised o) and attention.cu's
// combine kernel merges the chunks.
//
// The two per-chunk contractions run as tcgen05.mma (fp16 in, fp32 out):
//   scores   S[t][h] = K[t] . q[h]      M = 128 rows (the chunk's 64 tokens;
//            rows 64-127 read the bytes that follow in shared memory and are
//            discarded, each score row depending on its own K row only),
//            N = 16 (the group's heads, padded), K = D; K rows and q K-major;
//   output   O^T[d][h] = sum_t V[t][d] p[h][t]   M = 128 dims per MMA, N = 16,
//            K = 64 tokens; the V tile is an MN-major operand, read exactly
//            as TMA lands it (rows = tokens, 64 dims per 128-byte row), p is
//            written K-major.
// Between them four warps (one per TMEM lane quarter, one token per thread)
// take each head's max over the chunk, p = exp(s - m) in fp32 rounded to
// fp16 for the second MMA, and l = sum of the rounded p.  Rows past the
// sequence length are masked out of the softmax and their V rows zeroed, so
// whatever the cache holds there never reaches the output.  Every mbarrier
// wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"
#include "tc.cuh"

namespace {

using namespace w4a8;

constexpr int C = 64;           // cached tokens per CTA
constexpr int NH = 16;          // heads of a group, padded (both MMAs' N)
constexpr int THREADS = 128;    // 4 warps, one per TMEM lane quarter
constexpr int TCOLS = 64;       // tensor memory: scores 16 columns, output 16 per 128 dims

// Rows of q and p stored per 64-column atom: 8 for groups of up to 8 heads
// (the N = 16 MMAs then read 8 more rows from the next 1024 bytes, which
// only feed the padding heads' columns), else 16.
template <int D, int GP>
struct ALayout {
    static constexpr int KT = D / 64;                  // 64-dim column tiles (128-byte rows)
    static constexpr int TILE = C * 128;               // 8 KB: 64 tokens x 64 dims, 128-byte swizzle
    static constexpr int QR = GP <= 8 ? 8 : 16;
    static constexpr int QATOM = QR * 128;             // QR heads x 64 elements
    static constexpr int OFF_K = 0;                    // K tiles; the scores MMA reads 8 KB past each
    static constexpr int OFF_V = OFF_K + KT * TILE;    //   (the next tile, the last one into V)
    static constexpr int OFF_Q = OFF_V + KT * TILE;    // q: KT atoms (K-major over D)
    static constexpr int OFF_P = OFF_Q + KT * QATOM;   // p: one atom (K-major over the 64 tokens)
    static constexpr int OFF_RED = OFF_P + QATOM;      // [2][NH] fp32 max, sum per head (also
    static constexpr int OFF_BAR = OFF_RED + 2 * NH * 4;       //   the 1 KB the p MMA may read past p)
    static constexpr int SMEM = OFF_RED + 1024 + 1024; // + slack to align the base to 1024
    static_assert(D == 128 || D == 256, "head dimension");
    static_assert(2 * NH * 4 + 64 <= 1024, "reduction buffer and barriers");
    static_assert(GP * C * 4 <= KT * TILE, "scores in the K tiles' space");
};

// byte offset of element (row r, column c) of a K-major operand with the
// 128-byte swizzle, stored as atoms of `atom_bytes` (all rows x 64 columns),
// atom c / 64 holding columns 64 (c / 64) ..: 8-row groups 1024 bytes apart,
// 16-byte chunk j of row r at j ^ (r % 8)
__device__ __forceinline__ uint32_t sw128_off(int r, int c, int atom_bytes) {
    return (uint32_t)((c >> 6) * atom_bytes + (r >> 3) * 1024 + (r & 7) * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) +
                      (c & 7) * 2);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// GP: the group size rounded up to a power of two (heads >= G are padding);
// the softmax loops run over GP heads only.  CL: the sequence's chunks are
// one thread-block cluster (grid x = cluster x = nsplit <= 16) and merge
// their partial results through distributed shared memory at the end, with
// no workspace and no second kernel; otherwise each chunk writes (m, l, o)
// to the workspace for the combine kernel.
template <int D, int GP, bool CL>
__global__ void __launch_bounds__(THREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const uint16_t *__restrict__ q, const int32_t *__restrict__ lens, int Hq, int Hkv, int Lmax, float scale,
               int nsplit, uint16_t *__restrict__ out, float *__restrict__ ws_o, float *__restrict__ ws_ml, int *status,
               long long budget) {
    using LY = ALayout<D, GP>;
    constexpr int KT = LY::KT;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + LY::OFF_BAR);
    uint64_t *kbar = bars, *vbar = bars + 1, *sbar = bars + 2, *obar = bars + 3;
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(bars + 4);
    float *red = reinterpret_cast<float *>(smem + LY::OFF_RED);

    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int G = Hq / Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = s * C;
    const size_t hq0 = (size_t)b * Hq + (size_t)g * G;
    // the chunk's K and V rows: KT boxes of 64 rows x 64 dims each; row
    // (b Hkv + g) Lmax + t0 of the [B Hkv Lmax][D] view (rows past the end of
    // the cache read as zero, rows past this sequence's length are masked)
    const int row0 = (b * Hkv + g) * Lmax + t0;
    auto issue_kv = [&]() {
        mbar_arrive_expect_tx(kbar, KT * LY::TILE);
        for (int c = 0; c < KT; ++c) tma_load_2d(sbase + LY::OFF_K + c * LY::TILE, &tm_k, c * 64, row0, smem_u32(kbar));
        mbar_arrive_expect_tx(vbar, KT * LY::TILE);
        for (int c = 0; c < KT; ++c) tma_load_2d(sbase + LY::OFF_V + c * LY::TILE, &tm_v, c * 64, row0, smem_u32(vbar));
    };
    // Ahead of the dependency wait only L2 is touched: the chunk's K and V
    // boxes are prefetched there (L2 is the point of coherence, so rows the
    // previous kernel writes later are updated there).  The length read here
    // is a hint: it decides whether to prefetch, and whether thread 0 starts
    // the copies into shared memory right after the wait, before the length
    // the kernel uses (read after the wait) has arrived.
    bool early = false;
    if (threadIdx.x == 0) {
        const int Lh = lens[b];
        early = Lh > t0 && t0 < Lmax;
        if (early) {
            for (int c = 0; c < KT; ++c) {
                tma_prefetch_2d(&tm_k, c * 64, row0);
                tma_prefetch_2d(&tm_v, c * 64, row0);
            }
        }
        for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
    }
    // q, the lengths and the output buffers may come from the previous kernel
    // on the stream
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        if (early) issue_kv();
    }
    int L = lens[b];
    L = L < 0 ? 0 : (L > Lmax ? Lmax : L);
    const int n = max(0, min(C, L - t0));
    if (n == 0 && early) {
        // the hint was stale: the copies must land before their space is reused
        // or the CTA leaves
        mbar_wait_bounded(kbar, 0, budget, status);
        mbar_wait_bounded(vbar, 0, budget, status);
    }
    if (n == 0) __syncthreads();

    // cluster mode: this chunk's o [G][D] fp32, in the K tiles' space once the
    // MMAs have completed; (m, l) per head are red[h], red[NH + h]
    float *opart = reinterpret_cast<float *>(smem + LY::OFF_K);
    if (n == 0 && CL) {
        // an empty chunk weighs nothing in the merge, but takes part in it
        for (int i = threadIdx.x; i < G * D; i += THREADS) opart[i] = 0.0f;
        if (threadIdx.x < NH) {
            red[threadIdx.x] = -INFINITY;
            red[NH + threadIdx.x] = 0.0f;
        }
    } else if (n == 0) {
        // an empty chunk reads nothing and weighs nothing in the combine
        if (nsplit > 1) {
            for (int i = threadIdx.x; i < G * D; i += THREADS) ws_o[((hq0 + i / D) * nsplit + s) * D + i % D] = 0.0f;
            if (threadIdx.x < G) {
                ws_ml[((hq0 + threadIdx.x) * nsplit + s) * 2] = -INFINITY;
                ws_ml[((hq0 + threadIdx.x) * nsplit + s) * 2 + 1] = 0.0f;
            }
        } else {
            for (int i = threadIdx.x; i < G * D; i += THREADS) out[hq0 * D + i] = 0;
        }
        return;
    } else {

        // q of the group's heads (the scores' B operand; heads >= G zero), in
        // 16-byte pieces of 8 dims.  Its loads go first: behind the chunk's K and
        // V copies (all CTAs' together) they would wait microseconds.
        constexpr int QN = LY::QR * (D / 8);                 // pieces
        constexpr int QPT = (QN + THREADS - 1) / THREADS;    // pieces per thread
        uint4 qv[QPT];
    #pragma unroll
        for (int j = 0; j < QPT; ++j) {
            const int i = threadIdx.x + j * THREADS, h = i / (D / 8), d0 = (i % (D / 8)) * 8;
            qv[j] = make_uint4(0u, 0u, 0u, 0u);
            if (i < QN && h < G) qv[j] = *reinterpret_cast<const uint4 *>(q + (hq0 + h) * D + d0);
        }

        if (threadIdx.x == 0 && !early) issue_kv();      // the hint said empty
        if (warp == 0) tmem_alloc_cols(smem_u32((const void *)tslot), TCOLS);
    #pragma unroll
        for (int j = 0; j < QPT; ++j) {
            const int i = threadIdx.x + j * THREADS, h = i / (D / 8), d0 = (i % (D / 8)) * 8;
            if (i < QN) *reinterpret_cast<uint4 *>(smem + LY::OFF_Q + sw128_off(h, d0, LY::QATOM)) = qv[j];
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const uint32_t tmem = *tslot;

        bool ok = true;
        if (threadIdx.x == 0) {
            // S[t][h] (tensor memory columns 0..15): D / 16 MMAs of K = 16, M = 128
            constexpr uint32_t idesc_s = (1u << 4) | ((uint32_t)(NH >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
            ok = mbar_wait_bounded(kbar, 0, budget, status);
            if (ok) {
                tc_fence_after();
    #pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int c = kk >> 2, sub = kk & 3;
                    const uint64_t ad = smem_desc_sw128(sbase + LY::OFF_K + c * LY::TILE) + (uint64_t)(sub * 2);
                    const uint64_t bd = smem_desc_sw128(sbase + LY::OFF_Q + c * LY::QATOM) + (uint64_t)(sub * 2);
                    tc_mma_f16(tmem, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc_commit(smem_u32(sbar));
            }
        }

        // softmax over the chunk.  The chunk's 64 token threads (warps 0 and 1:
        // TMEM lanes 0-63) put their scaled scores into shared memory (-inf past
        // the length and for padding heads), in the K tiles' space: the scores'
        // MMAs have completed; then warp w takes heads w, w + 4, .., each lane
        // the tokens lane and lane + 32
        ok = mbar_wait_bounded(sbar, 0, budget, status) && ok;
        tc_fence_after();
        float *sc = reinterpret_cast<float *>(smem + LY::OFF_K);     // [GP][C]
        if (warp < C / 32) {
            uint32_t r[NH];
            tmem_ld_cols<16>(tmem + ((uint32_t)(warp * 32) << 16), r);
            tmem_ld_wait();
            const int t = warp * 32 + lane;
    #pragma unroll
            for (int h = 0; h < GP; ++h) sc[h * C + t] = (t < n && h < G) ? __uint_as_float(r[h]) * scale : -INFINITY;
        }
        __syncthreads();
        for (int h = warp; h < GP; h += 4) {
            const float x0 = sc[h * C + lane], x1 = sc[h * C + lane + 32];
            const float m = warp_max(fmaxf(x0, x1));
            // p rounded to fp16 for the MMA; l sums the rounded values
            const __half p0 = __float2half_rn(x0 == -INFINITY ? 0.0f : expf(x0 - m));
            const __half p1 = __float2half_rn(x1 == -INFINITY ? 0.0f : expf(x1 - m));
            *reinterpret_cast<__half *>(smem + LY::OFF_P + sw128_off(h, lane, LY::QATOM)) = p0;
            *reinterpret_cast<__half *>(smem + LY::OFF_P + sw128_off(h, lane + 32, LY::QATOM)) = p1;
            const float l = warp_sum(__half2float(p0) + __half2float(p1));
            if (lane == 0) {
                red[h] = m;
                red[NH + h] = l;
            }
        }
        // V rows past the sequence's length become zero (the cache may hold
        // anything there, and 0 * inf or 0 * nan would reach the sums)
        ok = mbar_wait_bounded(vbar, 0, budget, status) && ok;
        if (n < C) {
            for (int i = threadIdx.x; i < (C - n) * KT * 8; i += THREADS) {
                const int row = n + i / (KT * 8), c = (i / 8) % KT, chunk = i % 8;
                *reinterpret_cast<uint4 *>(smem + LY::OFF_V + c * LY::TILE + row * 128 + chunk * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        if (threadIdx.x == 0 && ok) {
            // O^T[d][h] (columns 16 + 16 mh for dims 128 mh ..): 4 MMAs of K = 16 tokens per 128 dims,
            // A = V tile MN-major (two 64-dim tiles along M), B = p K-major
            constexpr uint32_t idesc_o =
                (1u << 4) | (1u << 15) | ((uint32_t)(NH >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
            tc_fence_after();
    #pragma unroll
            for (int half = 0; half < D / 128; ++half) {
    #pragma unroll
                for (int kk = 0; kk < C / 16; ++kk) {
                    const uint64_t ad =
                        smem_desc_sw128_mn(sbase + LY::OFF_V + 2 * half * LY::TILE + kk * 16 * 128, (uint32_t)LY::TILE);
                    const uint64_t bd = smem_desc_sw128(sbase + LY::OFF_P) + (uint64_t)((kk & 3) * 2);
                    tc_mma_f16(tmem + 16u + (uint32_t)(16 * half), ad, bd, idesc_o, kk > 0 ? 1u : 0u);
                }
            }
            tc_commit(smem_u32(obar));
        }

        // output: thread = dim d (lane quarter of its warp) of each 128-dim half
        ok = mbar_wait_bounded(obar, 0, budget, status) && ok;
        tc_fence_after();
    #pragma unroll
        for (int half = 0; half < D / 128; ++half) {
            uint32_t r[NH];
            tmem_ld_cols<16>(tmem + ((uint32_t)(warp * 32) << 16) + 16u + (uint32_t)(16 * half), r);
            tmem_ld_wait();
            const int d = half * 128 + warp * 32 + lane;
            if (CL) {
    #pragma unroll
                for (int h = 0; h < GP; ++h)
                    if (h < G) opart[h * D + d] = __uint_as_float(r[h]);
            } else if (ok) {
    #pragma unroll
                for (int h = 0; h < GP; ++h) {
                    if (h >= G) break;
                    const size_t hq = hq0 + h;
                    const float o = __uint_as_float(r[h]);
                    if (nsplit == 1) {
                        const float lsum = red[NH + h];
                        const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
                        out[hq * D + d] = __half_as_ushort(__float2half_rn(o * inv));
                    } else {
                        ws_o[(hq * nsplit + s) * D + d] = o;
                    }
                }
            }
        }
        if (!CL && nsplit > 1 && ok && threadIdx.x < G) {
            // the chunk's (m, l) of head h
            const int h = threadIdx.x;
            ws_ml[((hq0 + h) * nsplit + s) * 2] = red[h];
            ws_ml[((hq0 + h) * nsplit + s) * 2 + 1] = red[NH + h];
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            tc_fence_after();
            tmem_dealloc_cols(tmem, TCOLS);
        }
    }

    if constexpr (CL) {
        // merge the cluster's chunks (split order; deterministic):
        //   M = max m_s,  out = sum_s o_s e^(m_s - M) / sum_s l_s e^(m_s - M)
        // first the weights of each head (q's space is free), then this CTA's
        // share of the outputs
        cluster_sync_all();
        const int S = nsplit;
        float *wts = reinterpret_cast<float *>(smem + LY::OFF_Q);       // [G][S], then 1 / L per head
        const uint32_t red_a = smem_u32(red), op_a = smem_u32(opart);
        if (threadIdx.x < G) {
            const int h = threadIdx.x;
            float mz[16], lz[16];
            float M = -INFINITY;
#pragma unroll
            for (int z = 0; z < 16; ++z) {
                mz[z] = z < S ? ld_dsmem_f32(dsmem_addr(red_a + (uint32_t)(h * 4), (uint32_t)z)) : -INFINITY;
                lz[z] = z < S ? ld_dsmem_f32(dsmem_addr(red_a + (uint32_t)((NH + h) * 4), (uint32_t)z)) : 0.0f;
            }
#pragma unroll
            for (int z = 0; z < 16; ++z) M = fmaxf(M, mz[z]);
            float Lsum = 0.0f;
#pragma unroll
            for (int z = 0; z < 16; ++z) {
                const float w = mz[z] == -INFINITY ? 0.0f : expf(mz[z] - M);    // empty chunks weigh nothing
                wts[h * 16 + z] = w;
                Lsum = fmaf(lz[z], w, Lsum);
            }
            wts[16 * 16 + h] = Lsum > 0.0f ? 1.0f / Lsum : 0.0f;
        }
        __syncthreads();
        // four consecutive elements per thread: one 16-byte remote load per
        // CTA of the cluster, all in flight together, summed in split order
        for (int i4 = s * THREADS + threadIdx.x; i4 < G * D / 4; i4 += S * THREADS) {
            const int idx = 4 * i4, h = idx / D;
            float4 vz[16];
#pragma unroll
            for (int z = 0; z < 16; ++z)
                vz[z] = z < S ? ld_dsmem_f32x4(dsmem_addr(op_a + (uint32_t)(idx * 4), (uint32_t)z)) : make_float4(0.f, 0.f, 0.f, 0.f);
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int z = 0; z < 16; ++z) {
                if (z < S) {
                    const float w = wts[h * 16 + z];
                    o.x = fmaf(vz[z].x, w, o.x);
                    o.y = fmaf(vz[z].y, w, o.y);
                    o.z = fmaf(vz[z].z, w, o.z);
                    o.w = fmaf(vz[z].w, w, o.w);
                }
            }
            const float inv = wts[16 * 16 + h];
            const __half2 lo = __floats2half2_rn(o.x * inv, o.y * inv), hi = __floats2half2_rn(o.z * inv, o.w * inv);
            uint2 pk;
            pk.x = *reinterpret_cast<const uint32_t *>(&lo);
            pk.y = *reinterpret_cast<const uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(out + (hq0 + h) * D + idx % D) = pk;
        }
        cluster_sync_all();   // no CTA leaves while a peer may still read its partials
    }
}

template <int D, int GP, bool CL>
w4a8_status launch_tc(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *lens, int B, int Hq,
                      int Hkv, int Lmax, int nsplit, uint16_t *out, float *ws_o, float *ws_ml, cudaStream_t stream) {
    static std::atomic<int> attr_done[w4a8_host::kDeviceSlots];
    const w4a8_status ast = w4a8_host::ensure_smem_limit(attn_tc_kernel<D, GP, CL>, ALayout<D, GP>::SMEM, attr_done);
    if (ast != W4A8_OK) return ast;
    if (CL && nsplit > 8) {
        // clusters of up to 16 CTAs (beyond the portable 8)
        static std::atomic<int> np_done[w4a8_host::kDeviceSlots];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= w4a8_host::kDeviceSlots) return W4A8_ERR_CUDA;
        if (!np_done[dev].load(std::memory_order_acquire)) {
            if (cudaFuncSetAttribute(attn_tc_kernel<D, GP, CL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                cudaSuccess) {
                cudaGetLastError();
                return W4A8_ERR_UNSUPPORTED;
            }
            np_done[dev].store(1, std::memory_order_release);
        }
    }
    int *status = w4a8_host::device_status_ptr();
    if (!status) return W4A8_ERR_CUDA;
    const uint64_t rows = (uint64_t)B * Hkv * Lmax;
    CUtensorMap tk, tv;
    if (!w4a8_host::make_tensor_map_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, k, (uint64_t)D, rows, 64, C,
                                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !w4a8_host::make_tensor_map_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, v, (uint64_t)D, rows, 64, C,
                                       CU_TENSOR_MAP_SWIZZLE_128B))
        return W4A8_ERR_CUDA;
    // programmatic dependent launch: the grid may start while the previous
    // kernel on the stream finishes; it waits for it before reading anything
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nsplit, (unsigned)Hkv, (unsigned)B);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = ALayout<D, GP>::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int na = 1;
    if (CL) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)nsplit;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        na = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (cudaLaunchKernelEx(&cfg, attn_tc_kernel<D, GP, CL>, tk, tv, q, lens, Hq, Hkv, Lmax, 1.0f / sqrtf((float)D), nsplit,
                           out, ws_o, ws_ml, status, w4a8_host::wait_budget()) != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    return w4a8_host::launch_status();
}

template <int D, bool CL>
w4a8_status launch_tc_g(int gp, const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *lens, int B,
                        int Hq, int Hkv, int Lmax, int nsplit, uint16_t *out, float *ws_o, float *ws_ml,
                        cudaStream_t stream) {
    switch (gp) {
        case 1: return launch_tc<D, 1, CL>(q, k, v, lens, B, Hq, Hkv, Lmax, nsplit, out, ws_o, ws_ml, stream);
        case 2: return launch_tc<D, 2, CL>(q, k, v, lens, B, Hq, Hkv, Lmax, nsplit, out, ws_o, ws_ml, stream);
        case 4: return launch_tc<D, 4, CL>(q, k, v, lens, B, Hq, Hkv, Lmax, nsplit, out, ws_o, ws_ml, stream);
        case 8: return launch_tc<D, 8, CL>(q, k, v, lens, B, Hq, Hkv, Lmax, nsplit, out, ws_o, ws_ml, stream);
        default: return launch_tc<D, 16, CL>(q, k, v, lens, B, Hq, Hkv, Lmax, nsplit, out, ws_o, ws_ml, stream);
    }
}

template <int D>
w4a8_status launch_tc_d(int gp, bool cl, const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *lens,
                        int B, int Hq, int Hkv, int Lmax, int nsplit, uint16_t *out, float *ws_o, float *ws_ml,
                        cudaStream_t stream) {
    return cl ? launch_tc_g<D, true>(gp, q, k, v, lens, B, Hq, Hkv, Lmax, nsplit, out, ws_o, ws_ml, stream)
              : launch_tc_g<D, false>(gp, q, k, v, lens, B, Hq, Hkv, Lmax, nsplit, out, ws_o, ws_ml, stream);
}

}  // namespace

namespace w4a8_host {

// (the cache's rows, B Hkv Lmax, are far below 2^31 on any device: 2^31 rows
// of 128 fp16 are 512 GB)
bool attention_tc_supported(int D, int Hq, int Hkv) { return (D == 128 || D == 256) && Hq / Hkv <= NH; }

int attention_tc_chunk() { return C; }

w4a8_status launch_attention_tc(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *lens, int B,
                                int Hq, int Hkv, int D, int Lmax, int nsplit, uint16_t *out, float *ws_o, float *ws_ml,
                                cudaStream_t stream, bool *merged) {
    const int G = Hq / Hkv;
    const int gp = G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : G <= 8 ? 8 : 16;
    *merged = false;
    if (nsplit >= 2 && nsplit <= 16) {
        // the sequence's chunks as one cluster, merged on chip; if the
        // cluster cannot be launched, the workspace route below takes over
        const w4a8_status st =
            D == 128 ? launch_tc_d<128>(gp, true, q, k, v, lens, B, Hq, Hkv, Lmax, nsplit, out, ws_o, ws_ml, stream)
                     : launch_tc_d<256>(gp, true, q, k, v, lens, B, Hq, Hkv, Lmax, nsplit, out, ws_o, ws_ml, stream);
        if (st == W4A8_OK) {
            *merged = true;
            return st;
        }
        cudaGetLastError();
    }
    if (D == 128) return launch_tc_d<128>(gp, false, q, k, v, lens, B, Hq, Hkv, Lmax, nsplit, out, ws_o, ws_ml, stream);
    if (D == 256) return launch_tc_d<256>(gp, false, q, k, v, lens, B, Hq, Hkv, Lmax, nsplit, out, ws_o, ws_ml, stream);
    return W4A8_ERR_UNSUPPORTED;
}

}  // namespace w4a8_host
