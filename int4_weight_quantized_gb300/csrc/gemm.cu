// gemm.cu -- prefill-phase W4A8 linear on the 5th-generation tensor cores.
//
// Prefill is compute-bound ("Що змінює ML Drift для on-device AI-інференсу на
// вашому телефоні?", tech.dede.sh, section "Stage-aware оптимізація для
// великих мовних моделей"), so the block dots run as a dense contraction on
// tcgen05.  sm_103a has no int8 MMA (tcgen05 kind::i8 is not available on
// this target), so codes are fed as fp16: every int4 weight (-8..7) and int8
// activation code (-127..127) is an exact fp16 value, each product is exact in
// fp32, and every partial sum of one 32-wide block stays below 32*8*127 =
// 32512 < 2^24, so the fp32 accumulator holds the exact integer block dot.
//
// Data flow of one CTA (128 weight rows x 128 tokens, K in stages of 64 =
// two 32-blocks):
//   - a quantisation pass (quant.cu) has already written the activation codes
//     as fp16 [M_pad][K] and the scales s_x as fp32 [K/32][M_pad];
//   - warp 0 (TMA) loads per stage the activation tile (128 tokens x 64 k,
//     128-byte swizzle) and the packed weight tile (128 rows x 32 bytes);
//     warp 2 loads s_x rows into a ring of their own;
//   - warps 3-6 expand the int4 weights to fp16 and write them into shared
//     memory in the same 128-byte-swizzled K-major layout, where the MMA
//     reads them as operand A;
//   - warp 1 issues tcgen05.mma (M=128 weight rows, N=128 tokens, K=16), two
//     per 32-block, each block into its own TMEM accumulator; the four
//     accumulators (all 512 columns) form two pairs, and the MMA and
//     epilogue hand a pair back and forth with one signal each way, so the
//     per-handshake cost is paid once per 64 k;
//   - warps 7-14 drain each block's exact integer dots from TMEM
//     (tcgen05.ld) and apply the block scales in fp32 registers:
//     acc[n][m] += d * (s_w[n,b] * s_x[m,b]); the result is stored as fp16.
//
// The contraction order inside each 8-wide group of k is [0,4,1,5,2,6,3,7]
// on both operands (the cheapest order for unpacking nibbles into fp16
// pairs); a dot product does not depend on the order of its terms.
//
// Every mbarrier wait is bounded (sync.cuh): on timeout the kernel records
// W4A8_ERR_TIMEOUT, stops issuing work, waits (bounded) for its own copies
// and MMAs in flight, frees its tensor memory and returns.
#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"
#include "tc.cuh"

namespace {

using namespace w4a8;

constexpr int BM = 128;            // weight rows per CTA: MMA M, TMEM lanes
constexpr int BN = 128;            // tokens per CTA: MMA N
constexpr int KS = 64;             // k per pipeline stage: two 32-blocks, one accumulator pair
constexpr int S_SM = 4;            // shared-memory stages
constexpr int SXG = 8;             // 32-blocks of s_x per load
constexpr int S_SX = 4;            // s_x stages (of SXG blocks each)
constexpr int NP = 2;              // accumulator pairs in TMEM (2 x 2 x 128 columns = all 512)
constexpr int TILE = 128 * 128;    // bytes of one 128-row x 64-k fp16 tile (one 128-byte-swizzle atom column)
constexpr int W_BYTES = BM * KS / 2;        // 4 KB, packed int4 of one stage
constexpr int SX_BYTES = SXG * BN * 4;      // 4 KB, SXG blocks of s_x
constexpr int EPI_WARPS = 8;          // 2 per TMEM lane quarter, 64 token columns each
constexpr int CONV_WARP0 = 3;        // warps 3..6 convert weights (32 rows each)
constexpr int EPI_WARP0 = 7;         // warps 7..14 run the epilogue
constexpr int THREADS = (EPI_WARP0 + EPI_WARPS) * 32;

constexpr int OFF_ACT = 0;                          // S_SM activation tiles (TMA, swizzled)
constexpr int OFF_A = OFF_ACT + S_SM * TILE;        // S_SM fp16 weight tiles (converter, swizzled)
constexpr int OFF_W = OFF_A + S_SM * TILE;          // S_SM packed weight tiles (TMA)
constexpr int OFF_SX = OFF_W + S_SM * W_BYTES;
constexpr int OFF_BAR = OFF_SX + S_SX * SX_BYTES;
// barriers: full, conv, empty (S_SM); sxfull, sxempty (S_SX); dfull, dempty (NP); final
constexpr int NUM_BARS = 3 * S_SM + 2 * S_SX + 2 * NP + 1;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;   // + slack to align the base to 1024

struct GemmArgs {
    const uint16_t *sw;      // [N][nb] fp16
    uint16_t *out;           // [M][N] fp16
    int32_t *dots;           // debug: [M][N][nb]
    int *status;
    long long budget;
    int M, N, K, nb;
    int splits;              // CTAs of a cluster along K (1, 2, 4 or 8); blockIdx.z is the split
    int bps;                 // 32-blocks per split (even)
};

// Instruction descriptor: fp32 accumulator, fp16 A and B, both K-major.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

// Bounded wait by every lane of a warp, with one warp-wide outcome (the
// tcgen05.ld/st that follow are warp-collective).  A failed wait raises the
// CTA's abort flag; once it is up, waits fail at once.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const GemmArgs &a, volatile uint32_t *abort_flag) {
    bool ok = (*abort_flag == 0u) && mbar_wait_bounded(bar, parity, a.budget, a.status);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && (threadIdx.x & 31) == 0) *abort_flag = 1u;
    return ok;
}

// Sum of the S partial tiles for W/2 columns of one row, in split order.
// Thread t of the 256 epilogue threads takes row t % 128 and half t / 128 of
// this CTA's W = 128/S columns.
template <int S>
__device__ __forceinline__ void reduce_splits(uint32_t red, int z, int t, int n0, int m0, const GemmArgs &a, bool ok) {
    constexpr int W = BN / S, C = W / 2;
    const int r = t & (BM - 1);
    const int c_beg = z * W + (t >> 7) * C;
    const int n = n0 + r;
    uint32_t base[S];
#pragma unroll
    for (int zz = 0; zz < S; ++zz) base[zz] = dsmem_addr(red + (uint32_t)((c_beg * BM + r) * 4), (uint32_t)zz);
#pragma unroll
    for (int j0 = 0; j0 < C; j0 += 8) {
        float v[8][S];
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int zz = 0; zz < S; ++zz) v[j][zz] = (j0 + j < C) ? ld_dsmem_f32(base[zz] + (uint32_t)((j0 + j) * BM * 4)) : 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j0 + j >= C) break;
            float s = 0.0f;
#pragma unroll
            for (int zz = 0; zz < S; ++zz) s += v[j][zz];
            const int m = m0 + c_beg + j0 + j;
            if (ok && n < a.N && m < a.M) a.out[(size_t)m * a.N + n] = __half_as_ushort(__float2half_rn(s));
        }
    }
}

template <bool DEBUG>
__global__ void __launch_bounds__(THREADS, 1)
gemm_w4a8_tc_kernel(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_w,
                    const __grid_constant__ CUtensorMap tm_sx, GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint64_t *full = bars, *conv = full + S_SM, *empty = conv + S_SM;
    uint64_t *sxfull = empty + S_SM, *sxempty = sxfull + S_SX;
    uint64_t *dfull = sxempty + S_SX, *dempty = dfull + NP, *finalb = dempty + NP;
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(smem + OFF_MISC);   // [0] tmem base, [1] abort

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BM, m0 = blockIdx.y * BN;
    const int nb = a.nb;
    // This CTA's K range: blocks [b0, b0 + nbl) of the row (all of it when
    // there is one split).
    const int b0 = blockIdx.z * a.bps;
    const int nbl = max(0, min(nb, b0 + a.bps) - b0);
    const int nst = (nbl + 1) / 2;              // stages = accumulator pairs

    if (threadIdx.x == 0) {
        for (int s = 0; s < S_SM; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&conv[s], 4);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < S_SX; ++s) {
            mbar_init(&sxfull[s], 1);
            mbar_init(&sxempty[s], EPI_WARPS);
        }
        for (int i = 0; i < NP; ++i) {
            mbar_init(&dfull[i], 1);
            mbar_init(&dempty[i], EPI_WARPS);
        }
        mbar_init(finalb, 1);
        misc[1] = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc_512(smem_u32((const void *)&misc[0]));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ TMA producers
        // warp 0: activation and packed-weight tiles; warp 2: s_x rows (own
        // ring, so the main stream never waits for the epilogue)
        if (lane == 0) {
            const bool main = warp == 0;
            const int S = main ? S_SM : S_SX;
            uint64_t *fb = main ? full : sxfull;
            uint64_t *eb = main ? empty : sxempty;
            int issued = 0;
            const int nloads = main ? nst : (nbl + SXG - 1) / SXG;
            for (int s = 0; s < nloads; ++s) {
                const int slot = s % S;
                const uint32_t ph = (uint32_t)(s / S) & 1u;
                if (misc[1] || !(mbar_test_wait(&eb[slot], ph ^ 1u) || mbar_wait_bounded(&eb[slot], ph ^ 1u, a.budget, a.status))) {
                    misc[1] = 1;
                    break;
                }
                if (main) {
                    mbar_arrive_expect_tx(&fb[slot], TILE + W_BYTES);
                    tma_load_2d(sbase + OFF_ACT + slot * TILE, &tm_act, b0 * 32 + s * KS, m0, smem_u32(&fb[slot]));
                    tma_load_2d(sbase + OFF_W + slot * W_BYTES, &tm_w, b0 * 16 + s * (KS / 2), n0, smem_u32(&fb[slot]));
                } else {
                    mbar_arrive_expect_tx(&fb[slot], SX_BYTES);
                    tma_load_2d(sbase + OFF_SX + slot * SX_BYTES, &tm_sx, m0, b0 + SXG * s, smem_u32(&fb[slot]));
                }
                issued = s + 1;
            }
            if (misc[1]) {
                // let every copy this thread issued land before the CTA exits
                for (int s = (issued > S ? issued - S : 0); s < issued; ++s)
                    mbar_wait_bounded(&fb[s % S], (uint32_t)(s / S) & 1u, a.budget, nullptr);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // One stage = one accumulator pair: two 32-blocks, each two K=16 MMAs
        // into its own accumulator; one completion signal per pair.
        if (lane == 0) {
            for (int s = 0; s < nst && !misc[1]; ++s) {
                const int slot = s % S_SM, pr = s % NP;
                const uint32_t ph = (uint32_t)(s / S_SM) & 1u, pp = (uint32_t)(s / NP) & 1u;
                const bool f_ok = mbar_test_wait(&full[slot], ph);
                const bool c_ok = mbar_test_wait(&conv[slot], ph);
                const bool d_ok = mbar_test_wait(&dempty[pr], pp ^ 1u);
                if ((!f_ok && !mbar_wait_bounded(&full[slot], ph, a.budget, a.status)) ||
                    (!c_ok && !mbar_wait_bounded(&conv[slot], ph, a.budget, a.status)) ||
                    (!d_ok && !mbar_wait_bounded(&dempty[pr], pp ^ 1u, a.budget, a.status))) {
                    misc[1] = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t abase = sbase + OFF_A + slot * TILE;
                const uint32_t bbase = sbase + OFF_ACT + slot * TILE;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if (2 * s + j >= nbl) break;
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const uint32_t off = (uint32_t)(j * 64 + kk * 32);
                        tc_mma_f16(tmem + (uint32_t)((2 * pr + j) * BN), smem_desc_sw128(abase + off),
                                  smem_desc_sw128(bbase + off), kIdesc, (uint32_t)kk);
                    }
                }
                tc_commit(smem_u32(&dfull[pr]));
                tc_commit(smem_u32(&empty[slot]));
            }
            // every MMA issued so far has completed once this barrier flips
            tc_commit(smem_u32(finalb));
            mbar_wait_bounded(finalb, 0, a.budget, nullptr);
        }
    } else if (warp >= CONV_WARP0 && warp < CONV_WARP0 + 4) {
        // ------------------------------------------------------------ int4 -> fp16 into shared memory
        // Thread r writes its row's 64 fp16 weights of the stage as 8 chunks of
        // 16 bytes, chunk c at position c ^ (r % 8) of the row's 128 bytes: the
        // 128-byte swizzled K-major layout the MMA descriptor reads.
        const int r = (warp - CONV_WARP0) * 32 + lane;
        for (int s = 0; s < nst; ++s) {
            const int slot = s % S_SM;
            const uint32_t ph = (uint32_t)(s / S_SM) & 1u;
            if (!warp_wait(&full[slot], ph, a, &misc[1])) break;
            const uint4 *src = reinterpret_cast<const uint4 *>(smem + OFF_W + slot * W_BYTES + r * (KS / 2));
            const uint4 p0 = src[0], p1 = src[1];
            const uint32_t wd[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
            uint8_t *row = smem + OFF_A + slot * TILE + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(row + ((c ^ (r & 7)) << 4)) = int4x8_to_half8(wd[c]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&conv[slot]);
        }
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------------------ epilogue
        // Per pair of blocks: one wait, four TMEM loads of 32 token columns
        // (this warp owns 64), 128 fp32 scale-multiply-adds per thread, one
        // release of the pair.
        const int e = warp - EPI_WARP0;
        const int q = warp & 3;                        // TMEM lane quarter this warp may access
        const int c0 = (e >> 2) * 64;                  // this warp's 64 token columns
        const int r = q * 32 + lane;
        const int n = n0 + r;
        const bool nok = n < a.N;
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0;
        const uint16_t *swrow = a.sw + (size_t)(nok ? n : 0) * nb + b0;
        float acc[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
        // s_w of the next pair of blocks is loaded one pair ahead and kept as
        // raw fp16 bits: converting right after the load would stall the warp
        // on the global-load latency at every block.
        unsigned short swn0 = (nok && nbl > 0) ? __ldg(swrow) : (unsigned short)0;
        unsigned short swn1 = (nok && nbl > 1) ? __ldg(swrow + 1) : (unsigned short)0;
        int sxslot = 0, gi = 0;
        uint32_t sxpar = 0u;
        for (int s = 0; s < nst; ++s) {
            const int pr = s % NP;
            const uint32_t pp = (uint32_t)(s / NP) & 1u;
            if (!(mbar_test_wait(&dfull[pr], pp) || warp_wait(&dfull[pr], pp, a, &misc[1]))) break;
            bool aborted = false;
            const unsigned short swc0 = swn0, swc1 = swn1;
            if (nok && 2 * s + 2 < nbl) swn0 = __ldg(swrow + 2 * s + 2);
            if (nok && 2 * s + 3 < nbl) swn1 = __ldg(swrow + 2 * s + 3);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int b = 2 * s + j;        // local block; b0 + b in the row
                if (b >= nbl) break;
                const float swf = __half2float(__ushort_as_half(j ? swc1 : swc0));
                if (gi == 0 && !(mbar_test_wait(&sxfull[sxslot], sxpar) || warp_wait(&sxfull[sxslot], sxpar, a, &misc[1]))) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const float *sxp = reinterpret_cast<const float *>(smem + OFF_SX + sxslot * SX_BYTES) + gi * BN + c0;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t d[32];
                    tmem_ld_cols<32>(tbase + (uint32_t)((2 * pr + j) * BN + h * 32), d);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float4 sx4 = *reinterpret_cast<const float4 *>(sxp + h * 32 + i);
                        const float sxv[4] = {sx4.x, sx4.y, sx4.z, sx4.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float dv = __uint_as_float(d[i + u]);
                            acc[h * 32 + i + u] = fmaf(dv, swf * sxv[u], acc[h * 32 + i + u]);
                            if (DEBUG) {
                                const int m = m0 + c0 + h * 32 + i + u;
                                if (nok && m < a.M) a.dots[((size_t)m * a.N + n) * nb + b0 + b] = (int32_t)dv;
                            }
                        }
                    }
                }
                if (gi == SXG - 1 || b == nbl - 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sxempty[sxslot]);
                }
                if (++gi == SXG) {
                    gi = 0;
                    if (++sxslot == S_SX) { sxslot = 0; sxpar ^= 1u; }
                }
            }
            if (aborted) break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&dempty[pr]);
        }
        if (a.splits > 1) {
            // partial tile of this K range -> shared memory, column-major
            // (the operand ring is idle now: every MMA has completed)
            float *red = reinterpret_cast<float *>(smem + OFF_ACT);
#pragma unroll
            for (int i = 0; i < 64; ++i) red[(c0 + i) * BM + r] = acc[i];
        } else if (nok && misc[1] == 0u) {
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const int m = m0 + c0 + i;
                if (m < a.M) a.out[(size_t)m * a.N + n] = __half_as_ushort(__float2half_rn(acc[i]));
            }
        }
    }

    if (a.splits > 1) {
        // Split-K: the CTAs of the cluster hold the partial tiles of their K
        // ranges; CTA z sums columns [z*W, (z+1)*W) of all of them through
        // distributed shared memory, in split order (fixed, deterministic).
        cluster_sync_all();
        if (warp >= EPI_WARP0) {
            const int t = threadIdx.x - EPI_WARP0 * 32;
            const uint32_t red = sbase + OFF_ACT;
            const bool ok = misc[1] == 0u;
            if (a.splits == 2) reduce_splits<2>(red, blockIdx.z, t, n0, m0, a, ok);
            else if (a.splits == 4) reduce_splits<4>(red, blockIdx.z, t, n0, m0, a, ok);
            else reduce_splits<8>(red, blockIdx.z, t, n0, m0, a, ok);
        }
        cluster_sync_all();   // no CTA leaves while a peer may still read its tile
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_512(tmem);
    }
}

// ------------------------------------------------------------------ host side

int m_pad(int M) { return (M + BN - 1) / BN * BN; }

constexpr int kSMs = 152;

// Split-K factor: the tile grid alone (N/128 x M_pad/128 CTAs) leaves most
// SMs idle for short sequences.  Measured on GB300, a call costs about
// 0.5 us per 32-block of a CTA plus ~8 us fixed (quantisation pass, pipeline
// fill, reduction), so pick S in {1, 2, 4, 8} minimising
// waves(tiles * S) * (blocks per split + 16); ties keep the smaller S.
int pick_splits(int tiles, int nb) {
    int best = 1;
    long best_cost = -1;
    for (int S = 1; S <= 8; S *= 2) {
        if (S > 1 && nb < 2 * S) break;
        const int bps = 2 * ((nb + 2 * S - 1) / (2 * S));
        const long waves = ((long)tiles * S + kSMs - 1) / kSMs;
        const long cost = waves * (bps + 16);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = S;
        }
    }
    return best;
}

template <bool DEBUG>
w4a8_status launch_t(const CUtensorMap &ta, const CUtensorMap &tw, const CUtensorMap &ts, const GemmArgs &a,
                     dim3 grid, cudaStream_t stream) {
    static std::atomic<int> attr_done[w4a8_host::kDeviceSlots];
    const w4a8_status ast = w4a8_host::ensure_smem_limit(gemm_w4a8_tc_kernel<DEBUG>, SMEM_BYTES, attr_done);
    if (ast != W4A8_OK) return ast;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)a.splits;
    cfg.attrs = attr;
    cfg.numAttrs = a.splits > 1 ? 1 : 0;   // one split: a plain launch
    if (cudaLaunchKernelEx(&cfg, gemm_w4a8_tc_kernel<DEBUG>, ta, tw, ts, a) != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    return w4a8_host::launch_status();
}

}  // namespace

namespace w4a8_host {

// Shapes with K % 256 == 0 run on the tensor-core kernel of gemm_mid.cu
// (128-token tiles); this file's kernel takes the others.

int prefill_splits(int M, int N, int K) {
    if (tc_supported(M, N, K)) return tc_splits(M, N, K);
    return pick_splits(((N + BM - 1) / BM) * (m_pad(M) / BN), K / 32);
}

int prefill_tokens_padded(int M, int N, int K) { return tc_supported(M, N, K) ? tc_tokens_padded(M) : m_pad(M); }

size_t prefill_workspace_bytes(int M, int N, int K) {
    const size_t mp = (size_t)prefill_tokens_padded(M, N, K);
    return mp * (size_t)K * 2 + (size_t)(K / 32) * mp * 4;
}

w4a8_status launch_prefill(const uint16_t *x, const void *packed_w, const uint16_t *scales,
                           int M, int N, int K, uint16_t *out, int32_t *dots, void *workspace,
                           cudaStream_t stream) {
    if (tc_supported(M, N, K)) return launch_tc_linear(x, packed_w, scales, M, N, K, out, dots, workspace, stream);
    const int mp = m_pad(M);
    uint16_t *q16 = static_cast<uint16_t *>(workspace);
    float *sx = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + (size_t)mp * K * 2);
    w4a8_status st = launch_quant_prefill(x, M, K, mp, q16, sx, stream);
    if (st != W4A8_OK) return st;
    return launch_prefill_gemm(q16, sx, packed_w, scales, M, N, K, out, dots, stream);
}

w4a8_status launch_prefill_gemm(const uint16_t *q16, const float *sx, const void *packed_w, const uint16_t *scales,
                                int M, int N, int K, uint16_t *out, int32_t *dots, cudaStream_t stream) {
    if (tc_supported(M, N, K)) return launch_tc_gemm(q16, sx, packed_w, scales, M, N, K, out, dots, stream);
    const int mp = m_pad(M);
    const int nb = K / 32;
    CUtensorMap ta, tw, ts;
    if (!w4a8_host::make_tensor_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, q16, (uint64_t)K, (uint64_t)mp, 64, BN,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !w4a8_host::make_tensor_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, packed_w, (uint64_t)K / 2, (uint64_t)N, KS / 2, BM,
                     CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !w4a8_host::make_tensor_map_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, sx, (uint64_t)mp, (uint64_t)nb, BN, SXG,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
        return W4A8_ERR_CUDA;

    GemmArgs a;
    a.sw = scales;
    a.out = out;
    a.dots = dots;
    a.status = device_status_ptr();
    a.budget = wait_budget();
    a.M = M;
    a.N = N;
    a.K = K;
    a.nb = nb;
    if (!a.status) return W4A8_ERR_CUDA;
    a.splits = prefill_splits(M, N, K);
    a.bps = 2 * ((nb + 2 * a.splits - 1) / (2 * a.splits));
    dim3 grid((unsigned)((N + BM - 1) / BM), (unsigned)(mp / BN), (unsigned)a.splits);
    return dots ? launch_t<true>(ta, tw, ts, a, grid, stream) : launch_t<false>(ta, tw, ts, a, grid, stream);
}

}  // namespace w4a8_host
