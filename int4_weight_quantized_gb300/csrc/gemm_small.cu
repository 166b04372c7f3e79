// gemm_small.cu -- W4A8 linear for 1 to 32 tokens on the 5th-generation
// tensor cores: weights as the 128-row MMA operand held in tensor memory,
// tokens as N (16 or 32), one synchronisation per 256 k.
//
// Stage-aware kernel choice ("Що змінює ML Drift для on-device
// AI-інференсу на вашому телефоні?", tech.dede.sh, section "Stage-aware
// оптимізація для великих мовних моделей"; "谷歌突然开源！端侧 AI 的 GPU
// 底座，要变了", m.x-techcon.com, section "对大模型，重点已经从“算得快”变成
// “数据少搬”"): a few tokens make the weight stream the whole cost, so the
// block dots go to the tensor cores and the weights are read once.
//
// With so few tokens an MMA (M = 128, N <= 32, K = 16) is a fixed ~45
// cycles, and every mbarrier test or arrival costs a warp on the order of a
// hundred cycles (measured).  So the unit of hand-off here is a quad of four
// 64-k stages (eight 32-blocks): one barrier round per quad between each
// pair of roles, against one per stage or pair of stages in gemm_mid.cu.
// The fp16 weights go to tensor memory (tcgen05.st) instead of shared
// memory, which frees shared memory for deeper copy rings and takes the
// expansion's stores and proxy fences off the shared-memory pipe.
//
// Per CTA (128 weight rows, a range of K, 16 or 32 tokens):
//   - warp 0: packed int4 weights by TMA, 128 rows x 128 bytes (one quad)
//     per copy, six copies in flight, started before the dependency wait;
//   - warp 3: activation codes (fp16, from the quantisation pass), four
//     64-k boxes per quad onto one barrier; warp 2: s_w and s_x;
//   - warps 4-7: thread r reads its row's 128 bytes of the quad, expands
//     them to exact fp16 and stores them to its tensor-memory lane (warp w
//     owns lanes 32 (w % 4) ...), two quads of 128 columns in a ring;
//   - warp 1: 16 tcgen05.mma per quad, A from tensor memory, B (tokens) from
//     shared memory, each 32-block into its own accumulator of N columns;
//     two accumulator units of 128 columns cycle with the epilogue;
//   - warps 8-15: per-block fp32 scaling of the exact dots, as in
//     gemm_mid.cu; split-K partial tiles are summed in a fixed order through
//     distributed shared memory.
//
// Every mbarrier wait is bounded; on timeout the kernel records
// W4A8_ERR_TIMEOUT, stops issuing, waits (bounded) for its own copies and
// MMAs, frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"
#include "tc.cuh"
#include "tc_pipe.cuh"

namespace {

using namespace w4a8;

constexpr int BM = 128;            // weight rows per CTA: MMA M, TMEM lanes
constexpr int QB = 8;              // 32-blocks per quad (256 k)
constexpr int W_TILE = BM * 128;   // 16 KB: 128 rows x 128 bytes (one quad), 128-byte swizzle
constexpr int WS = 6;              // packed-weight quads in flight
constexpr int AQ = 2;              // fp16 weight quads in tensor memory, 128 columns each
constexpr int ACC0 = AQ * 128;     // first accumulator column
constexpr int UNITS = 2;           // accumulator units of 128 columns
constexpr int SG = 16;             // 32-blocks per s_x load
constexpr int SS = 3;              // s_x stages
constexpr int SWG = 64;            // 32-blocks per s_w load (128 bytes of each row)
constexpr int SWS = 2;             // s_w stages
constexpr int SW_TILE = BM * SWG * 2;
constexpr int CONV_WARP0 = 4;
constexpr int CONVW = 4;
constexpr int EPI0 = CONV_WARP0 + CONVW;
constexpr int EPI_WARPS = 8;       // 2 per TMEM lane quarter, half of the tokens each
constexpr int THREADS = (EPI0 + EPI_WARPS) * 32;

template <int NT>
struct SLayout {
    static constexpr int X_BOX = NT * 64 * 2;              // NT tokens x 64 k fp16 (one TMA box)
    static constexpr int X_QUAD = 4 * X_BOX;
    static constexpr int XQ = NT == 16 ? 4 : 3;            // activation quads in flight
    static constexpr int SX_TILE = SG * NT * 4;            // 16 blocks x NT tokens fp32
    static constexpr int UB = 128 / NT;                    // blocks per accumulator unit
    static constexpr int OFF_W = 0;
    static constexpr int OFF_X = OFF_W + WS * W_TILE;
    static constexpr int OFF_SW = OFF_X + XQ * X_QUAD;
    static constexpr int OFF_SX = OFF_SW + SWS * SW_TILE;
    static constexpr int OFF_BAR = OFF_SX + SS * SX_TILE;
    // wfull, wempty; afull, aempty; xfull, xempty; sfull, sempty; swfull, swempty; accfull, accempty; final
    static constexpr int NUM_BARS = 2 * WS + 2 * AQ + 2 * XQ + 2 * SS + 2 * SWS + 2 * UNITS + 1;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;     // + slack to align the base to 1024
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(X_BOX % 1024 == 0 && OFF_X % 1024 == 0 && OFF_SW % 1024 == 0, "swizzle atoms");
    static_assert(BM * NT * 4 <= WS * W_TILE, "split-K partial tile must fit the weight ring");
};

template <int NT, bool DEBUG>
__global__ void __launch_bounds__(THREADS, 1)
gemm_small_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                  const __grid_constant__ CUtensorMap tm_sw, const __grid_constant__ CUtensorMap tm_sx, MidArgs a) {
    using LY = SLayout<NT>;
    constexpr int XQ = LY::XQ;
    constexpr int UB = LY::UB;
    constexpr int HT = NT / 2;                 // tokens per epilogue thread
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + LY::OFF_BAR);
    uint64_t *wfull = bars, *wempty = wfull + WS;
    uint64_t *afull = wempty + WS, *aempty = afull + AQ;
    uint64_t *xfull = aempty + AQ, *xempty = xfull + XQ;
    uint64_t *sfull = xempty + XQ, *sempty = sfull + SS;
    uint64_t *swfull = sempty + SS, *swempty = swfull + SWS;
    uint64_t *accfull = swempty + SWS, *accempty = accfull + UNITS;
    uint64_t *finalb = accempty + UNITS;
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(smem + LY::OFF_MISC);   // [0] tmem, [1] abort

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BM;
    const int m0 = blockIdx.y * NT;
    const int b0 = blockIdx.z * a.bps;
    const int nbl = max(0, min(a.nb, b0 + a.bps) - b0);    // this CTA's 32-blocks (multiple of 8)
    const int nq = nbl / QB;                                  // quads
    const int nunits = nbl / UB;
    const int ngroups = (nbl + SG - 1) / SG;

    if (threadIdx.x == 0) {
        for (int s = 0; s < WS; ++s) { mbar_init(&wfull[s], 1); mbar_init(&wempty[s], CONVW); }
        // a quad is ready for the MMA once the 4 expansion warps have stored
        // its weights and seen its activation boxes land
        for (int s = 0; s < AQ; ++s) { mbar_init(&afull[s], CONVW); mbar_init(&aempty[s], 1); }
        for (int s = 0; s < XQ; ++s) { mbar_init(&xfull[s], 1); mbar_init(&xempty[s], 1); }
        for (int s = 0; s < SS; ++s) { mbar_init(&sfull[s], 1); mbar_init(&sempty[s], EPI_WARPS); }
        for (int s = 0; s < SWS; ++s) { mbar_init(&swfull[s], 1); mbar_init(&swempty[s], EPI_WARPS); }
        for (int s = 0; s < UNITS; ++s) { mbar_init(&accfull[s], 1); mbar_init(&accempty[s], EPI_WARPS); }
        mbar_init(finalb, 1);
        misc[1] = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc_512(smem_u32((const void *)&misc[0]));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        // ---------------------------------------------------------- weights (TMA), before the dependency wait
        if (lane == 0) {
            int issued = 0;
            for (int q = 0; q < nq; ++q) {
                const int slot = q % WS;
                if (!one_wait(&wempty[slot], ((uint32_t)(q / WS) & 1u) ^ 1u, a, misc + 1)) break;
                mbar_arrive_expect_tx(&wfull[slot], W_TILE);
                tma_load_2d(sbase + LY::OFF_W + slot * W_TILE, &tm_w, (b0 + QB * q) * 16, n0, smem_u32(&wfull[slot]));
                issued = q + 1;
            }
            for (int q = (issued > WS ? issued - WS : 0); q < issued; ++q)
                mbar_wait_bounded(&wfull[q % WS], (uint32_t)(q / WS) & 1u, a.budget, nullptr);
        }
    } else if (warp == 2 || warp == 3) {
        // ---------------------------------------------------------- scales (warp 2), activation codes (warp 3)
        pdl_wait();
        if (lane == 0 && warp == 3) {
            int issued = 0;
            for (int q = 0; q < nq; ++q) {
                const int slot = q % XQ;
                if (!one_wait(&xempty[slot], ((uint32_t)(q / XQ) & 1u) ^ 1u, a, misc + 1)) break;
                mbar_arrive_expect_tx(&xfull[slot], LY::X_QUAD);
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    tma_load_2d(sbase + LY::OFF_X + slot * LY::X_QUAD + h * LY::X_BOX, &tm_x, (b0 + QB * q + 2 * h) * 32,
                                m0, smem_u32(&xfull[slot]));
                issued = q + 1;
            }
            for (int q = (issued > XQ ? issued - XQ : 0); q < issued; ++q)
                mbar_wait_bounded(&xfull[q % XQ], (uint32_t)(q / XQ) & 1u, a.budget, nullptr);
        } else if (lane == 0) {
            // s_x in groups of SG blocks; s_w (128-byte rows) once every SWG / SG groups
            int issued = 0, swissued = 0;
            for (int g = 0; g < ngroups; ++g) {
                if (g % (SWG / SG) == 0) {
                    const int w = g / (SWG / SG), slot = w % SWS;
                    if (!one_wait(&swempty[slot], ((uint32_t)(w / SWS) & 1u) ^ 1u, a, misc + 1)) break;
                    mbar_arrive_expect_tx(&swfull[slot], SW_TILE);
                    tma_load_2d(sbase + LY::OFF_SW + slot * SW_TILE, &tm_sw, b0 + SWG * w, n0, smem_u32(&swfull[slot]));
                    swissued = w + 1;
                }
                const int slot = g % SS;
                if (!one_wait(&sempty[slot], ((uint32_t)(g / SS) & 1u) ^ 1u, a, misc + 1)) break;
                mbar_arrive_expect_tx(&sfull[slot], LY::SX_TILE);
                tma_load_2d(sbase + LY::OFF_SX + slot * LY::SX_TILE, &tm_sx, m0, b0 + SG * g, smem_u32(&sfull[slot]));
                issued = g + 1;
            }
            for (int g = (issued > SS ? issued - SS : 0); g < issued; ++g)
                mbar_wait_bounded(&sfull[g % SS], (uint32_t)(g / SS) & 1u, a.budget, nullptr);
            for (int w = (swissued > SWS ? swissued - SWS : 0); w < swissued; ++w)
                mbar_wait_bounded(&swfull[w % SWS], (uint32_t)(w / SWS) & 1u, a.budget, nullptr);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        // The whole warp runs the loop, so every address and descriptor is
        // warp-uniform (uniform registers, computed once per quad; per block
        // only compile-time offsets are added) and lane 0 issues.  The MMA
        // warp shares its sub-partition with an expansion warp and two
        // epilogue warps, so its instruction count per MMA sets its rate.
        constexpr uint32_t idesc = (1u << 4) | ((uint32_t)(NT >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
        constexpr int UPQ = QB / UB;                  // accumulator units per quad (1 or 2)
        const uint64_t xdesc0 = smem_desc_sw128(sbase + LY::OFF_X);
        for (int q = 0; q < nq; ++q) {
            const int as = q % AQ, xs = q % XQ;
            if (!warp_wait(&afull[as], (uint32_t)(q / AQ) & 1u, a, misc + 1)) break;
            tc_fence_after();
            const uint32_t abase = tmem + (uint32_t)(as * 128);
            const uint64_t xq = xdesc0 + (uint64_t)((xs * LY::X_QUAD) >> 4);
            bool ok = true;
#pragma unroll
            for (int h = 0; h < UPQ; ++h) {
                const int u = q * UPQ + h;
                if (!warp_wait(&accempty[u % UNITS], ((uint32_t)(u / UNITS) & 1u) ^ 1u, a, misc + 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dbase = tmem + (uint32_t)(ACC0 + (u % UNITS) * 128);
#pragma unroll
                for (int jj = 0; jj < UB; ++jj) {
                    const int j = h * UB + jj;            // block of the quad
                    // block j: box j / 2, bytes (j % 2) * 64 of each 128-byte token row
                    const uint64_t xo = (uint64_t)((((j >> 1) * LY::X_BOX) + (j & 1) * 64) >> 4);
                    if (lane == 0) {
                        tc_mma_f16_ta(dbase + (uint32_t)(jj * NT), abase + (uint32_t)(j * 16), xq + xo, idesc, 0u);
                        tc_mma_f16_ta(dbase + (uint32_t)(jj * NT), abase + (uint32_t)(j * 16 + 8), xq + xo + 2, idesc, 1u);
                    }
                }
                if (lane == 0) tc_commit(smem_u32(&accfull[u % UNITS]));
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) {
                tc_commit(smem_u32(&aempty[as]));
                tc_commit(smem_u32(&xempty[xs]));
            }
            __syncwarp();
        }
        // every MMA issued so far has completed once this barrier flips
        if (lane == 0) {
            tc_commit(smem_u32(finalb));
            mbar_wait_bounded(finalb, 0, a.budget, nullptr);
        }
        __syncwarp();
    } else if (warp >= CONV_WARP0 && warp < EPI0) {
        // ---------------------------------------------------------- int4 -> fp16 weights into tensor memory
        // Thread r holds row r: the 8 chunks of 16 bytes of its 128-byte row
        // (chunk c at position c ^ (r % 8): 128-byte swizzle), i.e. the 8
        // blocks of the quad; block j becomes 16 columns (32 fp16, two
        // consecutive k per column) at column 16 j of the quad's 128.
        const int qtr = warp & 3;                     // TMEM lane quarter of this warp
        const int r = qtr * 32 + lane;
        const uint32_t tlane = tmem + ((uint32_t)(qtr * 32) << 16);
        for (int q = 0; q < nq; ++q) {
            const int ws = q % WS, as = q % AQ, xs = q % XQ;
            if (!warp_wait(&wfull[ws], (uint32_t)(q / WS) & 1u, a, misc + 1)) break;
            const uint8_t *wrow = smem + LY::OFF_W + ws * W_TILE + r * 128;
            uint32_t wd[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 pk = *reinterpret_cast<const uint4 *>(wrow + ((c ^ (r & 7)) << 4));
                wd[4 * c] = pk.x; wd[4 * c + 1] = pk.y; wd[4 * c + 2] = pk.z; wd[4 * c + 3] = pk.w;
            }
            if (!warp_wait(&aempty[as], ((uint32_t)(q / AQ) & 1u) ^ 1u, a, misc + 1)) break;
            tc_fence_after();
#pragma unroll
            for (int p = 0; p < 4; ++p) {                 // one 64-k stage (two blocks) per store
                uint32_t v[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 h = int4x8_to_half8(wd[8 * p + c]);
                    v[4 * c] = h.x; v[4 * c + 1] = h.y; v[4 * c + 2] = h.z; v[4 * c + 3] = h.w;
                }
                tmem_st_cols32(tlane + (uint32_t)(as * 128 + 32 * p), v);
            }
            tmem_st_wait();
            // the packed slot is released only now: every value read from it
            // has been used (a release right after issuing the loads could
            // let the next copy into the slot overtake them)
            __syncwarp();
            if (lane == 0) mbar_arrive(&wempty[ws]);
            // the quad's activation boxes must have landed too before it is handed on
            if (!warp_wait(&xfull[xs], (uint32_t)(q / XQ) & 1u, a, misc + 1)) break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[as]);
        }
    } else if (warp >= EPI0) {
        // ---------------------------------------------------------- epilogue
        const int e = warp - EPI0;
        const int q = warp & 3;                       // TMEM lane quarter this warp may access
        const int t0 = (e >> 2) * HT;                 // this warp's first token
        const int r = q * 32 + lane;
        const int n = n0 + r;
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ACC0 + t0);
        float2 acc[HT / 2];
#pragma unroll
        for (int i = 0; i < HT / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);
        bool ok = true;
        pdl_wait();                                   // outputs are written below
        for (int u = 0; u < nunits && ok; ++u) {
            const int bu = u * UB;                    // first local block of the unit
            const int g = bu / SG, gw = bu / SWG;
            if (bu % SWG == 0 && !warp_wait(&swfull[gw % SWS], (uint32_t)(gw / SWS) & 1u, a, misc + 1)) {
                ok = false;
                break;
            }
            if (bu % SG == 0 && !warp_wait(&sfull[g % SS], (uint32_t)(g / SS) & 1u, a, misc + 1)) {
                ok = false;
                break;
            }
            // this row's s_w of the unit's UB blocks (fp16 pairs), one vector load
            // from the 128-byte-swizzled s_w tile (16-byte chunk c at c ^ (r % 8))
            uint32_t swu[UB / 2];
            {
                const int bo = bu % SWG;
                const uint8_t *sp = smem + LY::OFF_SW + (gw % SWS) * SW_TILE + r * 128 + (((bo >> 3) ^ (r & 7)) << 4) +
                                    (bo & 7) * 2;
                if constexpr (UB == 8) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(sp);
                    swu[0] = v.x; swu[1] = v.y; swu[2] = v.z; swu[3] = v.w;
                } else {
                    const uint2 v = *reinterpret_cast<const uint2 *>(sp);
                    swu[0] = v.x; swu[1] = v.y;
                }
            }
            if (!warp_wait(&accfull[u % UNITS], (uint32_t)(u / UNITS) & 1u, a, misc + 1)) { ok = false; break; }
            tc_fence_after();
            const float *sxt = reinterpret_cast<const float *>(smem + LY::OFF_SX + (g % SS) * LY::SX_TILE);
            const uint32_t tu = tbase + (uint32_t)((u % UNITS) * 128);
            // all UB blocks of the unit in one batch of loads (UB * HT = 64 columns)
            uint32_t d[UB][HT];
#pragma unroll
            for (int j = 0; j < UB; ++j) tmem_ld_cols<HT>(tu + (uint32_t)(j * NT), d[j]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&accempty[u % UNITS]);
#pragma unroll
            for (int j = 0; j < UB; ++j) {
                const int bl = bu + j;
                const uint32_t pr = swu[j >> 1];
                const float sw = __half2float(__ushort_as_half((uint16_t)((j & 1) ? (pr >> 16) : (pr & 0xffffu))));
                scale_acc<HT, DEBUG>(acc, d[j], sw, sxt + (bl % SG) * NT + t0, n, m0 + t0, b0 + bl, a);
            }
            const int bl_last = bu + UB - 1;
            if (bl_last % SG == SG - 1 || bl_last == nbl - 1) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&sempty[g % SS]);
            }
            if (bl_last % SWG == SWG - 1 || bl_last == nbl - 1) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&swempty[gw % SWS]);
            }
        }
        if (a.splits > 1) {
            // partial tile of this K range -> shared memory, [token][row]
            // (the weight ring is idle: every quad has been expanded and every
            // MMA has completed)
            float *red = reinterpret_cast<float *>(smem + LY::OFF_W);
#pragma unroll
            for (int i = 0; i < HT / 2; ++i) {
                red[(t0 + 2 * i) * BM + r] = acc[i].x;
                red[(t0 + 2 * i + 1) * BM + r] = acc[i].y;
            }
        } else if (ok && misc[1] == 0u && n < a.N) {
#pragma unroll
            for (int i = 0; i < HT / 2; ++i) {
                const int m = m0 + t0 + 2 * i;
                if (m < a.M) a.out[(size_t)m * a.N + n] = __half_as_ushort(__float2half_rn(acc[i].x));
                if (m + 1 < a.M) a.out[(size_t)(m + 1) * a.N + n] = __half_as_ushort(__float2half_rn(acc[i].y));
            }
        }
    }

    if (a.splits > 1) {
        // CTA z sums tokens [z*NT/S, (z+1)*NT/S) of every peer's partial tile
        // through distributed shared memory, in split order (deterministic).
        cluster_sync_all();
        if (warp >= EPI0) {
            const int t = threadIdx.x - EPI0 * 32;
            const uint32_t red = sbase + LY::OFF_W;
            const int S = a.splits;
            const int w = NT / S;                      // tokens reduced by this CTA
            const int c0 = (int)blockIdx.z * w;
            const bool okk = misc[1] == 0u;
            for (int idx = t; idx < w * BM; idx += EPI_WARPS * 32) {
                const int rr = idx % BM, c = c0 + idx / BM;
                const uint32_t off = (uint32_t)((c * BM + rr) * 4);
                float v[8];
#pragma unroll
                for (int z = 0; z < 8; ++z) v[z] = z < S ? ld_dsmem_f32(dsmem_addr(red + off, (uint32_t)z)) : 0.0f;
                float sum = 0.0f;
#pragma unroll
                for (int z = 0; z < 8; ++z)
                    if (z < S) sum += v[z];
                const int nn = n0 + rr, m = m0 + c;
                if (okk && nn < a.N && m < a.M) a.out[(size_t)m * a.N + nn] = __half_as_ushort(__float2half_rn(sum));
            }
        }
        cluster_sync_all();   // no CTA leaves while a peer may still read its tile
    }

    if (threadIdx.x == 0) pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_512(tmem);
    }
}

template <int NT, bool DEBUG>
w4a8_status launch_small(const CUtensorMap &tw, const CUtensorMap &tx, const CUtensorMap &tsw, const CUtensorMap &tsx,
                         const MidArgs &a, dim3 grid, cudaStream_t stream) {
    static std::atomic<int> attr_done[w4a8_host::kDeviceSlots];
    const w4a8_status ast = w4a8_host::ensure_smem_limit(gemm_small_kernel<NT, DEBUG>, SLayout<NT>::SMEM, attr_done);
    if (ast != W4A8_OK) return ast;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SLayout<NT>::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (a.splits > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = (unsigned)a.splits;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (cudaLaunchKernelEx(&cfg, gemm_small_kernel<NT, DEBUG>, tw, tx, tsw, tsx, a) != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    return w4a8_host::launch_status();
}

}  // namespace

namespace w4a8_host {

w4a8_status launch_small_gemm(int nt, const CUtensorMap &tw, const CUtensorMap &tx, const CUtensorMap &tsw,
                              const CUtensorMap &tsx, const w4a8::MidArgs &a, dim3 grid, cudaStream_t stream) {
    const bool dbg = a.dots != nullptr;
    switch (nt) {
        case 16: return dbg ? launch_small<16, true>(tw, tx, tsw, tsx, a, grid, stream)
                            : launch_small<16, false>(tw, tx, tsw, tsx, a, grid, stream);
        case 32: return dbg ? launch_small<32, true>(tw, tx, tsw, tsx, a, grid, stream)
                            : launch_small<32, false>(tw, tx, tsw, tsx, a, grid, stream);
        default: return W4A8_ERR_UNSUPPORTED;
    }
}

}  // namespace w4a8_host
