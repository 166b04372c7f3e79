// attention.cu -- decode attention over an fp16 KV cache.
//
// Decode reads, besides the weights, the KV cache of every sequence once per
// new token ("Що змінює ML Drift для on-device AI-інференсу на вашому
// телефоні?", tech.dede.sh, section "Stage-aware оптимізація для великих
// мовних моделей").  Layout (this library's): k and v [B][Hkv][Lmax][D] fp16,
// row t of sequence b valid for t < lens[b]; q and out [B][Hq][D] fp16;
// query head h reads KV head h / (Hq / Hkv) (grouped query heads).
//
//   out[b][h] = sum_t softmax_t(q[b][h] . k[b][g][t] / sqrt(D)) v[b][g][t]
//
// One CTA per (sequence, KV head, chunk of C = 128 cached tokens): the chunk's
// K and V rows are read once for all G query heads of the group.  The V rows
// (one contiguous range) are bulk-copied into shared memory at the start and
// land while the scores are computed; each thread issues all loads of its K
// row half before using any.  Scores are fp32 dot products (two threads per
// token, each half of D); the chunk's softmax is kept as (max m, sum l,
// unnormalised sum o); with one chunk the CTA writes the output, otherwise a
// combine kernel merges the chunks:
//   M = max m_s,  out = sum_s o_s e^(m_s - M) / sum_s l_s e^(m_s - M).
#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"

namespace {

using namespace w4a8;

constexpr int C = 128;          // cached tokens per CTA
constexpr int NT = 256;         // threads per CTA
constexpr int GMAX = 16;        // query heads per KV head, at most

size_t attn_smem(int D, int GP) {
    // V rows [C][D] fp16; q [G][D] fp32; scores [4][G][C] fp32 (four D
    // quarters, then p); the token-group fold buffer [NT/D][G][D] = NT*G fp32;
    // max and sum [2][G]; one mbarrier
    return (size_t)C * D * 2 + (size_t)GP * D * 4 + (size_t)4 * GP * C * 4 + (size_t)NT * GP * 4 + 2 * GP * 4 + 16;
}

// GP: the group size rounded up to a power of two (1..16), a compile-time
// bound for the per-head loops; heads h >= G are skipped.
template <int D, int GP>
__global__ void __launch_bounds__(NT, 2) attn_chunk_kernel(const uint16_t *__restrict__ q, const uint16_t *__restrict__ kc,
                                                        const uint16_t *__restrict__ vc, const int32_t *__restrict__ lens,
                                                        int Hq, int Hkv, int Lmax, float scale, int nsplit,
                                                        uint16_t *__restrict__ out, float *__restrict__ ws_o,
                                                        float *__restrict__ ws_ml, int *status, long long budget) {
    extern __shared__ __align__(16) float sm[];
    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int G = Hq / Hkv;
    uint16_t *vs = reinterpret_cast<uint16_t *>(sm);             // [C][D] V rows of the chunk
    float *qs = sm + C * D / 2;            // [G][D]
    float *sc = qs + GP * D;             // [4][G][C]
    float *os = sc + 4 * GP * C;         // [TH/2][G][D], TH = NT/(D/2) token groups
    float *ml = os + NT * GP;            // [G] max, [G] sum
    uint64_t *vbar = reinterpret_cast<uint64_t *>(ml + 2 * GP);
    int L = lens[b];
    L = L < 0 ? 0 : (L > Lmax ? Lmax : L);
    const int t0 = s * C;
    const int n = max(0, min(C, L - t0));
    const uint16_t *kb = kc + ((size_t)b * Hkv + g) * (size_t)Lmax * D;
    const uint16_t *vb = vc + ((size_t)b * Hkv + g) * (size_t)Lmax * D;

    if (threadIdx.x == 0) {
        mbar_init(vbar, 1);
        fence_barrier_init();
        if (n > 0) {
            // rows t0 .. t0+n-1 of this KV head are one contiguous range (16-byte multiples)
            const uint32_t bytes = (uint32_t)n * D * 2;
            mbar_arrive_expect_tx(vbar, bytes);
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                         ::"r"(smem_u32(vs)), "l"(vb + (size_t)t0 * D), "r"(bytes), "r"(smem_u32(vbar)) : "memory");
        }
    }

    // scores: thread -> tokens tp and tp + 64 of the chunk, quarter qt of D;
    // each 16-byte q load of a head feeds 16 FMAs (8 dims x 2 tokens).  The K
    // loads are issued first, together with the q loads, so that their
    // latencies overlap.
    {
        constexpr int NQ = D / 32;          // 8-dim groups per quarter row
        const int tp = threadIdx.x % 64, qt = threadIdx.x / 64;
        const int ta = tp, tb = tp + 64;
        uint4 ka[NQ], kb2[NQ];
        const uint16_t *ra = kb + (size_t)(t0 + (ta < n ? ta : 0)) * D + qt * (D / 4);
        const uint16_t *rb = kb + (size_t)(t0 + (tb < n ? tb : 0)) * D + qt * (D / 4);
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            ka[i] = ta < n ? *reinterpret_cast<const uint4 *>(ra + 8 * i) : make_uint4(0, 0, 0, 0);
            kb2[i] = tb < n ? *reinterpret_cast<const uint4 *>(rb + 8 * i) : make_uint4(0, 0, 0, 0);
        }
        // q of the group's G heads: G*D fp16 = at most 2 16-byte loads per thread
        {
            const uint16_t *qg = q + ((size_t)b * Hq + g * G) * D;
            const int items = G * D / 8;
            uint4 qv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = threadIdx.x + u * NT;
                qv[u] = i < items ? *reinterpret_cast<const uint4 *>(qg + 8 * i) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = threadIdx.x + u * NT;
                if (i < items) {
                    const __half2 *h2 = reinterpret_cast<const __half2 *>(&qv[u]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __half22float2(h2[e]);
                        qs[8 * i + 2 * e] = f.x;
                        qs[8 * i + 2 * e + 1] = f.y;
                    }
                }
            }
        }
        __syncthreads();
        float acc_a[GP], acc_b[GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) acc_a[h] = acc_b[h] = 0.0f;
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            float fa[8], fb[8];
            const __half2 *a2 = reinterpret_cast<const __half2 *>(&ka[i]);
            const __half2 *b2 = reinterpret_cast<const __half2 *>(&kb2[i]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 x = __half22float2(a2[u]), y = __half22float2(b2[u]);
                fa[2 * u] = x.x; fa[2 * u + 1] = x.y;
                fb[2 * u] = y.x; fb[2 * u + 1] = y.y;
            }
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                if (h < G) {
                    const float4 *qh = reinterpret_cast<const float4 *>(qs + h * D + qt * (D / 4) + 8 * i);
                    const float4 q0 = qh[0], q1 = qh[1];
                    const float qv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        acc_a[h] = fmaf(qv[u], fa[u], acc_a[h]);
                        acc_b[h] = fmaf(qv[u], fb[u], acc_b[h]);
                    }
                }
            }
        }
#pragma unroll
        for (int h = 0; h < GP; ++h)
            if (h < G) {
                sc[(qt * GP + h) * C + ta] = acc_a[h];
                sc[(qt * GP + h) * C + tb] = acc_b[h];
            }
    }
    __syncthreads();

    // per head: m = max, p = e^(s - m), l = sum p  (warp w takes heads w, w+8)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int h = warp; h < G; h += NT / 32) {
        float v[C / 32];
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < C / 32; ++j) {
            const int t = lane + 32 * j;
            v[j] = t < n ? ((sc[h * C + t] + sc[(GP + h) * C + t]) + (sc[(2 * GP + h) * C + t] + sc[(3 * GP + h) * C + t])) * scale
                         : -INFINITY;
            m = fmaxf(m, v[j]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.0f;
#pragma unroll
        for (int j = 0; j < C / 32; ++j) {
            const int t = lane + 32 * j;
            const float p = t < n ? expf(v[j] - m) : 0.0f;
            sc[h * C + t] = p;
            l += p;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            ml[h] = m;
            ml[GP + h] = l;
        }
    }
    __syncthreads();

    // o[h][d] = sum_t p[h][t] v[t][d]: thread -> pair of dims, half of the tokens
    {
        constexpr int PAIRS = D / 2;
        constexpr int TH = NT / PAIRS;     // token groups (2, 4 or 8)
        const int j = threadIdx.x % PAIRS, tg = threadIdx.x / PAIRS;
        float2 acc[GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) acc[h] = make_float2(0.0f, 0.0f);
        // the V rows have landed (bounded wait: on timeout the status word is
        // set and this chunk contributes nothing)
        // (polled with the non-suspending test: the copy is normally complete
        // by now, and a suspended thread may sleep past the completion)
        bool vok = n == 0 || mbar_test_wait(vbar, 0);
        if (!vok) {
            const long long c0 = clock64();
            while (!(vok = mbar_test_wait(vbar, 0)) && clock64() - c0 < budget) {
            }
            if (!vok && status) atomicExch(status, (int)W4A8_ERR_TIMEOUT);
        }
        constexpr int TPG = C / TH;        // contiguous tokens per group (multiple of 4)
        const int tbeg = tg * TPG, tend = min(n, tbeg + TPG);
        if (vok) {
            for (int t4 = tbeg; t4 < tend; t4 += 4) {
                float2 vv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    vv[u] = t4 + u < tend ? __half22float2(*reinterpret_cast<const __half2 *>(vs + (size_t)(t4 + u) * D + 2 * j))
                                          : make_float2(0.0f, 0.0f);
#pragma unroll
                for (int h = 0; h < GP; ++h) {
                    if (h < G) {
                        // p of 4 tokens in one load (p = 0 past n)
                        const float4 p = *reinterpret_cast<const float4 *>(sc + h * C + t4);
                        acc[h].x = fmaf(p.x, vv[0].x, fmaf(p.y, vv[1].x, fmaf(p.z, vv[2].x, fmaf(p.w, vv[3].x, acc[h].x))));
                        acc[h].y = fmaf(p.x, vv[0].y, fmaf(p.y, vv[1].y, fmaf(p.z, vv[2].y, fmaf(p.w, vv[3].y, acc[h].y))));
                    }
                }
            }
        }
        // fold the token groups pairwise through shared memory
        for (int step = TH; step > 1; step >>= 1) {
            const int hs = step >> 1;
            __syncthreads();
            if (tg >= hs && tg < step) {
#pragma unroll
                for (int h = 0; h < GP; ++h)
                    if (h < G) {
                        os[((tg - hs) * GP + h) * D + 2 * j] = acc[h].x;
                        os[((tg - hs) * GP + h) * D + 2 * j + 1] = acc[h].y;
                    }
            }
            __syncthreads();
            if (tg < hs) {
#pragma unroll
                for (int h = 0; h < GP; ++h)
                    if (h < G) {
                        acc[h].x += os[(tg * GP + h) * D + 2 * j];
                        acc[h].y += os[(tg * GP + h) * D + 2 * j + 1];
                    }
            }
        }
        if (tg == 0) {
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                if (h >= G) break;
                const size_t hq = (size_t)b * Hq + g * G + h;
                if (nsplit == 1) {
                    const float l = ml[GP + h];
                    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
                    *reinterpret_cast<__half2 *>(out + hq * D + 2 * j) = __floats2half2_rn(acc[h].x * inv, acc[h].y * inv);
                } else {
                    *reinterpret_cast<float2 *>(ws_o + (hq * nsplit + s) * D + 2 * j) = acc[h];
                    if (j == 0) {
                        ws_ml[(hq * nsplit + s) * 2] = ml[h];
                        ws_ml[(hq * nsplit + s) * 2 + 1] = ml[GP + h];
                    }
                }
            }
        }
    }
}

// out[b][h] from the chunks' (m, l, o): one CTA per (head, sequence), D/2
// threads.  First the split weights w_s = e^(m_s - M) and L = sum l_s w_s
// (the splits' loads spread over the threads), then each thread merges its
// pair of dims over the splits with independent loads.
constexpr int MAXS = 2048;      // splits per sequence the combine kernel takes (Lmax <= 131072 in 64-token chunks)

__global__ void attn_combine_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_ml, int Hq, int D,
                                    int nsplit, uint16_t *__restrict__ out) {
    __shared__ float wsh[MAXS];
    __shared__ float red[2][32];
    // launched as a programmatic dependent of the tensor-core chunk kernel:
    // wait for its partial results (a no-op after a plain launch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t hq = (size_t)blockIdx.y * Hq + blockIdx.x;
    const int j = threadIdx.x, nt = blockDim.x;
    const int warp = j >> 5, lane = j & 31, nw = (nt + 31) >> 5;
    float M = -INFINITY;
    for (int s = j; s < nsplit; s += nt) M = fmaxf(M, ws_ml[(hq * nsplit + s) * 2]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (lane == 0) red[0][warp] = M;
    __syncthreads();
    M = -INFINITY;
    for (int w = 0; w < nw; ++w) M = fmaxf(M, red[0][w]);
    float L = 0.0f;
    for (int s = j; s < nsplit; s += nt) {
        const float ms = ws_ml[(hq * nsplit + s) * 2];
        const float w = ms == -INFINITY ? 0.0f : expf(ms - M);      // empty chunks weigh nothing
        wsh[s] = w;
        L = fmaf(ws_ml[(hq * nsplit + s) * 2 + 1], w, L);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) red[1][warp] = L;
    __syncthreads();
    L = 0.0f;
    for (int w = 0; w < nw; ++w) L += red[1][w];
    float ox = 0.0f, oy = 0.0f;
#pragma unroll 8
    for (int s = 0; s < nsplit; ++s) {
        const float2 o = *reinterpret_cast<const float2 *>(ws_o + (hq * nsplit + s) * D + 2 * j);
        ox = fmaf(o.x, wsh[s], ox);
        oy = fmaf(o.y, wsh[s], oy);
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    *reinterpret_cast<__half2 *>(out + hq * D + 2 * j) = __floats2half2_rn(ox * inv, oy * inv);
}

template <int D, int GP>
w4a8_status launch_chunks(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *lens, int B, int Hq,
                          int Hkv, int Lmax, int nsplit, uint16_t *out, float *ws_o, float *ws_ml, cudaStream_t stream) {
    static std::atomic<int> attr_done[w4a8_host::kDeviceSlots];
    const size_t smem = attn_smem(D, GP);
    const w4a8_status ast = w4a8_host::ensure_smem_limit(attn_chunk_kernel<D, GP>, (int)smem, attr_done);
    if (ast != W4A8_OK) return ast;
    int *status = w4a8_host::device_status_ptr();
    if (!status) return W4A8_ERR_CUDA;
    dim3 grid((unsigned)nsplit, (unsigned)Hkv, (unsigned)B);
    attn_chunk_kernel<D, GP><<<grid, NT, smem, stream>>>(q, k, v, lens, Hq, Hkv, Lmax, 1.0f / sqrtf((float)D), nsplit, out,
                                                     ws_o, ws_ml, status, w4a8_host::wait_budget());
    return w4a8_host::launch_status();
}

// chunks per sequence: 64 tokens on the tensor-core kernel (D 128, 256),
// 128 on this file's kernel (D 64)
int chunk_tokens(int D) { return (D == 128 || D == 256) ? w4a8_host::attention_tc_chunk() : C; }
int nsplits(int D, int Lmax) { return (Lmax + chunk_tokens(D) - 1) / chunk_tokens(D); }

}  // namespace

namespace w4a8_host {

bool attention_shape_ok(int B, int Hq, int Hkv, int D, int Lmax) {
    return B >= 1 && Hq >= 1 && Hkv >= 1 && Hq % Hkv == 0 && Hq / Hkv <= GMAX && (D == 64 || D == 128 || D == 256) &&
           Lmax >= 1 && Lmax <= 131072 && nsplits(D, Lmax) <= MAXS;
}

size_t attention_workspace_bytes(int B, int Hq, int D, int Lmax) {
    const int ns = nsplits(D, Lmax);
    if (ns == 1) return 0;
    const size_t o = (size_t)B * Hq * ns * D * 4;
    return ((o + 255) & ~(size_t)255) + (size_t)B * Hq * ns * 2 * 4;
}

w4a8_status launch_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *lens, int B, int Hq,
                             int Hkv, int D, int Lmax, uint16_t *out, void *workspace, size_t workspace_bytes,
                             cudaStream_t stream) {
    const int ns = nsplits(D, Lmax);
    float *ws_o = nullptr, *ws_ml = nullptr;
    if (ns > 1) {
        const size_t need = attention_workspace_bytes(B, Hq, D, Lmax);
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) return W4A8_ERR_WORKSPACE;
        ws_o = static_cast<float *>(workspace);
        const size_t o = (size_t)B * Hq * ns * D * 4;
        ws_ml = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + ((o + 255) & ~(size_t)255));
    }
    const int G = Hq / Hkv;
    const int gp = G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : G <= 8 ? 8 : 16;
    w4a8_status st = W4A8_ERR_UNSUPPORTED;
    if (attention_tc_supported(D, Hq, Hkv)) {
        // head dimensions 128 and 256: both contractions on the tensor cores
        bool merged = false;
        st = launch_attention_tc(q, k, v, lens, B, Hq, Hkv, D, Lmax, ns, out, ws_o, ws_ml, stream, &merged);
        if (st != W4A8_OK || ns == 1 || merged) return st;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)Hq, (unsigned)B);
        cfg.blockDim = dim3((unsigned)(D / 2), 1, 1);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, attn_combine_kernel, (const float *)ws_o, (const float *)ws_ml, Hq, D, ns, out) !=
            cudaSuccess) {
            cudaGetLastError();
            return W4A8_ERR_CUDA;
        }
        return launch_status();
    }
#define W4A8_ATTN_CASE(DD, GG)                                                                                    \
    if (D == DD && gp == GG) st = launch_chunks<DD, GG>(q, k, v, lens, B, Hq, Hkv, Lmax, ns, out, ws_o, ws_ml, stream);
    W4A8_ATTN_CASE(64, 1) W4A8_ATTN_CASE(64, 2) W4A8_ATTN_CASE(64, 4) W4A8_ATTN_CASE(64, 8) W4A8_ATTN_CASE(64, 16)
    W4A8_ATTN_CASE(128, 1) W4A8_ATTN_CASE(128, 2) W4A8_ATTN_CASE(128, 4) W4A8_ATTN_CASE(128, 8) W4A8_ATTN_CASE(128, 16)
    W4A8_ATTN_CASE(256, 1) W4A8_ATTN_CASE(256, 2) W4A8_ATTN_CASE(256, 4) W4A8_ATTN_CASE(256, 8) W4A8_ATTN_CASE(256, 16)
#undef W4A8_ATTN_CASE
    if (st != W4A8_OK || ns == 1) return st;
    attn_combine_kernel<<<dim3((unsigned)Hq, (unsigned)B), D / 2, 0, stream>>>(ws_o, ws_ml, Hq, D, ns, out);
    return launch_status();
}

}  // namespace w4a8_host
