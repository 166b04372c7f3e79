// gemm_mid.cu -- W4A8 linear on the 5th-generation tensor cores with the
// weights as the 128-row operand, for tiles of 64 tokens (33 to 64 tokens)
// and of 128 tokens (prefill, K a multiple of 256); 1 to 32 tokens run in
// gemm_small.cu.
//
// Stage-aware kernel choice ("Що змінює ML Drift для on-device
// AI-інференсу на вашому телефоні?", tech.dede.sh, section "Stage-aware
// оптимізація для великих мовних моделей"; "谷歌突然开源！端侧 AI 的 GPU
// 底座，要变了", m.x-techcon.com, section "对大模型，重点已经从“算得快”变成
// “数据少搬”"): between one-token decode (a memory-bound GEMV) and long
// prefill (a compute-bound GEMM) lies a range of token counts where the
// weight stream still sets the time but dp4a per token costs too many
// instructions.  Here the tokens are the MMA's N dimension (a tile of 64 or
// 128) and every CTA streams 128 weight rows through a deep ring, so the
// tensor cores do the block dots and the weights are read once.
//
// Per CTA (128 weight rows, a range of K, all tokens):
//   - warp 0 streams the packed int4 weight tiles by TMA, 128 rows x 128
//     bytes (four 64-k stages) per load, into a ring of 2-4 such tiles; it
//     starts before the kernel waits for the quantisation pass (programmatic
//     dependent launch).  Tiles of 32-byte rows stream at well under half the
//     rate of 128-byte rows (measured), hence the wide loads;
//   - warps 4-7 expand them into fp16 (exact: -8..7) in the 128-byte-swizzled
//     K-major layout of the MMA's A operand;
//   - warp 3 loads the activation codes (fp16, written by the quantisation
//     pass) as the B operand, warp 2 the block scales s_w (64 blocks of each
//     row per load) and s_x;
//   - warp 1 issues tcgen05.mma (M = 128 rows, N = tokens, K = 16), two per
//     32-block, each block into its own TMEM accumulator of N columns; the
//     accumulator units (four of 128 columns, or two of 256 at 128 tokens)
//     cycle between it and the epilogue;
//   - warps 8 and up (8 of them at 128 tokens, 16 at 64) read each block's
//     exact integer dots (tcgen05.ld) and apply
//     acc += d * (s_w * s_x) in fp32 (pairs of tokens per instruction);
//   - with several CTAs along K (a thread-block cluster), the fp32 partial
//     tiles are summed in a fixed order through distributed shared memory.
//
// Every mbarrier wait is bounded (sync.cuh): on timeout the kernel records
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

constexpr int BM = 128;           // weight rows per CTA: MMA M, TMEM lanes
constexpr int KS = 64;            // k per stage: two 32-blocks
constexpr int AS = 4;             // fp16 weight (A operand) stages
constexpr int PS = AS / 2;        // stage pairs of A tiles in flight (one barrier per pair)
constexpr int WSTG = 4;           // pipeline stages per packed-weight load (128 bytes of each row)
constexpr int SG = 16;            // 32-blocks per s_x load
constexpr int SS = 3;             // s_x stages
constexpr int SWG = 64;           // 32-blocks per s_w load (128 bytes of each row)
constexpr int SWS = 2;            // s_w stages
constexpr int A_TILE = BM * KS * 2;            // 16 KB
constexpr int W_TILE = BM * 128;               // 16 KB: 128 rows x 128 bytes (4 stages), 128-byte swizzle
constexpr int SW_TILE = BM * SWG * 2;          // 16 KB: 128 rows x 64 fp16, 128-byte swizzle
constexpr int CONV_WARP0 = 4;

template <int NT>
struct Layout {
    static constexpr int WS = NT == 128 ? 2 : 4;           // packed-weight slots (4 pipeline stages each)
    static constexpr int X_TILE = NT * KS * 2;            // NT tokens x 64 k fp16
    // activation stages: a ring of its own, deep enough to hide the load
    // latency (about a microsecond) behind the MMAs of several stages
    static constexpr int XS = NT == 64 ? 6 : 4;
    static constexpr int XP = XS / 2;                      // activation stage pairs (one barrier each)
    static constexpr int SX_TILE = SG * NT * 4;            // 16 blocks x NT tokens fp32
    // accumulator units handed between the MMA and the epilogue: UB blocks
    // of NT columns each, NU of them in the 512 TMEM columns (at 128 tokens
    // two blocks per unit, so the epilogue's per-unit waits, scale loads and
    // arrivals are paid once per two blocks)
    static constexpr int UB = NT == 128 ? 2 : 128 / NT;
    static constexpr int UCOLS = UB * NT;
    static constexpr int NU = 512 / UCOLS;
    // int4 -> fp16 expansion warps (one thread per weight row; 8 warps with
    // two threads per row measured no faster)
    static constexpr int CONVW = 4;
    static constexpr int EPI0 = CONV_WARP0 + CONVW;        // first epilogue warp (a multiple of 4)
    // epilogue warps, a multiple of 4 (one group per TMEM lane quarter, each
    // warp of a group a share of the tokens): 16 measured faster than 8 at
    // 64 tokens, slower at 128
    static constexpr int EPI_WARPS = NT == 128 ? 8 : 16;
    static constexpr int THREADS = (EPI0 + EPI_WARPS) * 32;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_X = OFF_A + AS * A_TILE;
    static constexpr int OFF_W = OFF_X + XS * X_TILE;
    static constexpr int OFF_SW = OFF_W + WS * W_TILE;
    static constexpr int OFF_SX = OFF_SW + SWS * SW_TILE;
    static constexpr int OFF_BAR = OFF_SX + SS * SX_TILE;
    // wfull, wempty; pfull, pempty; xfull, xempty; sfull, sempty (s_x); swfull, swempty; accfull, accempty; final
    static constexpr int NUM_BARS = 2 * WS + 2 * PS + 2 * XP + 2 * SS + 2 * SWS + 2 * NU + 1;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;     // + slack to align the base to 1024
    static_assert(128 * NT * 4 <= AS * A_TILE, "split-K partial tile must fit the A ring");
};

template <int NT, bool DEBUG>
__global__ void __launch_bounds__(Layout<NT>::THREADS, 1)
gemm_mid_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                const __grid_constant__ CUtensorMap tm_sw, const __grid_constant__ CUtensorMap tm_sx, MidArgs a) {
    using LY = Layout<NT>;
    constexpr int WS = LY::WS;
    constexpr int XS = LY::XS, XP = LY::XP;
    constexpr int UB = LY::UB;
    constexpr int UNITS = LY::NU;
    constexpr int EPI_WARPS = LY::EPI_WARPS;
    constexpr int HT = NT / (EPI_WARPS / 4);   // tokens per epilogue thread
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + LY::OFF_BAR);
    uint64_t *wfull = bars, *wempty = wfull + WS;
    uint64_t *pfull = wempty + WS, *pempty = pfull + PS;
    uint64_t *xfull = pempty + PS, *xempty = xfull + XP;
    uint64_t *sfull = xempty + XP, *sempty = sfull + SS;
    uint64_t *swfull = sempty + SS, *swempty = swfull + SWS;
    uint64_t *accfull = swempty + SWS, *accempty = accfull + UNITS;
    uint64_t *finalb = accempty + UNITS;
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(smem + LY::OFF_MISC);   // [0] tmem, [1] abort

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BM;
    const int m0 = blockIdx.y * NT;
    const int b0 = blockIdx.z * a.bps;
    const int nbl = max(0, min(a.nb, b0 + a.bps) - b0);    // this CTA's 32-blocks (multiple of 8)
    const int nst = nbl / 2;                                 // stages
    const int nunits = nbl / UB;
    const int ngroups = (nbl + SG - 1) / SG;

    if (threadIdx.x == 0) {
        for (int s = 0; s < WS; ++s) { mbar_init(&wfull[s], 1); mbar_init(&wempty[s], LY::CONVW); }
        // a pair is ready for the MMA once the 4 expansion warps have written
        // its A tiles and seen its activation tiles land
        for (int s = 0; s < PS; ++s) { mbar_init(&pfull[s], LY::CONVW); mbar_init(&pempty[s], 1); }
        for (int s = 0; s < XP; ++s) { mbar_init(&xfull[s], 1); mbar_init(&xempty[s], 1); }
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
        // each load brings 128 bytes (256 k, four stages) of all 128 rows:
        // tiles of wide rows stream at the full rate, narrow ones do not
        if (lane == 0) {
            int issued = 0;
            const int nw = nst / WSTG;
            for (int w = 0; w < nw; ++w) {
                const int slot = w % WS;
                if (!one_wait(&wempty[slot], ((uint32_t)(w / WS) & 1u) ^ 1u, a, misc + 1)) break;
                mbar_arrive_expect_tx(&wfull[slot], W_TILE);
                tma_load_2d(sbase + LY::OFF_W + slot * W_TILE, &tm_w, (b0 + 2 * WSTG * w) * 16, n0, smem_u32(&wfull[slot]));
                issued = w + 1;
            }
            for (int w = (issued > WS ? issued - WS : 0); w < issued; ++w)
                mbar_wait_bounded(&wfull[w % WS], (uint32_t)(w / WS) & 1u, a.budget, nullptr);
        }
    } else if (warp == 2 || warp == 3) {
        // ---------------------------------------------------------- scales (warp 2), activation codes (warp 3)
        pdl_wait();
        if (lane == 0 && warp == 3) {
            int issued = 0;
            for (int p = 0; p < nst / 2; ++p) {
                const int slot = p % XP;
                if (!one_wait(&xempty[slot], ((uint32_t)(p / XP) & 1u) ^ 1u, a, misc + 1)) break;
                mbar_arrive_expect_tx(&xfull[slot], 2 * LY::X_TILE);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int st = 2 * p + h;
                    tma_load_2d(sbase + LY::OFF_X + (st % XS) * LY::X_TILE, &tm_x, (b0 + 2 * st) * 32, m0,
                                smem_u32(&xfull[slot]));
                }
                issued = p + 1;
            }
            for (int p = (issued > XP ? issued - XP : 0); p < issued; ++p)
                mbar_wait_bounded(&xfull[p % XP], (uint32_t)(p / XP) & 1u, a.budget, nullptr);
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
        // One barrier test and one commit per pair of stages (8 MMAs): each
        // mbarrier round trip costs the issuing thread about as much as two
        // MMAs of this size (measured), so they are amortised.  Descriptors
        // are formed once; per MMA only the start-address field advances.
        if (lane == 0) {
            constexpr uint32_t idesc = (1u << 4) | ((uint32_t)(NT >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
            const uint64_t adesc0 = smem_desc_sw128(sbase + LY::OFF_A);
            const uint64_t xdesc0 = smem_desc_sw128(sbase + LY::OFF_X);
            for (int p = 0; p < nst / 2; ++p) {
                const int slot = p % PS;
                if (!one_wait(&pfull[slot], (uint32_t)(p / PS) & 1u, a, misc + 1)) break;
                tc_fence_after();
                bool ok = true;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int st = 2 * p + (j >> 1);           // stage of this block
                    const int b = 2 * st + (j & 1), u = b / UB, jj = b - u * UB;
                    if (jj == 0 && !one_wait(&accempty[u % UNITS], ((uint32_t)(u / UNITS) & 1u) ^ 1u, a, misc + 1)) {
                        ok = false;
                        break;
                    }
                    if (jj == 0) tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)((u % UNITS) * LY::UCOLS + jj * NT);
                    const uint64_t ao = (uint64_t)(((st % AS) * A_TILE + (j & 1) * 64) >> 4);
                    const uint64_t xo = (uint64_t)(((st % XS) * LY::X_TILE + (j & 1) * 64) >> 4);
                    tc_mma_f16(d, adesc0 + ao, xdesc0 + xo, idesc, 0u);
                    tc_mma_f16(d, adesc0 + ao + 2, xdesc0 + xo + 2, idesc, 1u);
                    if (jj == UB - 1) tc_commit(smem_u32(&accfull[u % UNITS]));
                }
                if (!ok) break;
                tc_commit(smem_u32(&pempty[slot]));
                tc_commit(smem_u32(&xempty[p % XP]));
            }
            // every MMA issued so far has completed once this barrier flips
            tc_commit(smem_u32(finalb));
            mbar_wait_bounded(finalb, 0, a.budget, nullptr);
        }
    } else if (warp >= CONV_WARP0 && warp < LY::EPI0) {
        // ---------------------------------------------------------- int4 -> fp16 A tiles
        // Thread r expands its row's 64 weights of the stage into 8 chunks of
        // 16 bytes, chunk c at position c ^ (r % 8) of the row's 128 bytes.
        // The packed slot is released only after the values read from it
        // have been used (the fp16 stores depend on them): a release right
        // after issuing the loads could let the next TMA copy into the slot
        // overtake them.
        // The weight tile is 128-byte swizzled (chunk c of row r at c ^ (r % 8)),
        // so a warp's reads of its 32 rows' 32 bytes spread over all banks.
        constexpr int HALVES = LY::CONVW / 4;              // threads per weight row
        constexpr int CW = 8 / HALVES;                     // 16-byte output chunks per thread and stage
        const int ct = (warp - CONV_WARP0) * 32 + lane;
        const int r = ct % 128, h = ct / 128;
        for (int s = 0; s < nst; ++s) {
            const int w = s / WSTG, sub = s % WSTG, ws = w % WS, as = s % AS, p = s / 2;
            // barrier tests cost the warp about as much as converting a
            // stage, so each is made once per slot (weights: 4 stages) or
            // pair (A tiles)
            if (sub == 0 && !warp_wait(&wfull[ws], (uint32_t)(w / WS) & 1u, a, misc + 1)) break;
            if ((s & 1) == 0 && !warp_wait(&pempty[p % PS], ((uint32_t)(p / PS) & 1u) ^ 1u, a, misc + 1)) break;
            const uint8_t *wrow = smem + LY::OFF_W + ws * W_TILE + r * 128;
            uint32_t wd[CW];
#pragma unroll
            for (int i = 0; i < CW / 4; ++i) {
                const uint4 pk = *reinterpret_cast<const uint4 *>(wrow + (((2 * sub + h + i) ^ (r & 7)) << 4));
                wd[4 * i] = pk.x; wd[4 * i + 1] = pk.y; wd[4 * i + 2] = pk.z; wd[4 * i + 3] = pk.w;
            }
            uint8_t *row = smem + LY::OFF_A + as * A_TILE + r * 128;
#pragma unroll
            for (int c = 0; c < CW; ++c) {
                const int cc = h * CW + c;                 // output chunk (8 weights) of the row
                *reinterpret_cast<uint4 *>(row + ((cc ^ (r & 7)) << 4)) = int4x8_to_half8(wd[c]);
            }
            if (s & 1) fence_proxy_async_smem();       // both stages' tiles written: make them visible to the MMA
            // the pair's activation tiles must have landed too before the pair is handed on
            if ((s & 1) && !warp_wait(&xfull[p % XP], (uint32_t)(p / XP) & 1u, a, misc + 1)) break;
            __syncwarp();
            if (lane == 0) {
                if (s & 1) mbar_arrive(&pfull[p % PS]);
                if (sub == WSTG - 1) mbar_arrive(&wempty[ws]);
            }
        }
    } else if (warp >= LY::EPI0) {
        // ---------------------------------------------------------- epilogue
        const int e = warp - LY::EPI0;
        const int q = warp & 3;                       // TMEM lane quarter this warp may access
        const int t0 = (e >> 2) * HT;                 // this warp's first token
        const int r = q * 32 + lane;
        const int n = n0 + r;
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)t0;
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
            uint32_t swu[UB > 1 ? UB / 2 : 1];
            {
                const int bo = bu % SWG;
                const uint8_t *sp = smem + LY::OFF_SW + (gw % SWS) * SW_TILE + r * 128 + (((bo >> 3) ^ (r & 7)) << 4) +
                                    (bo & 7) * 2;
                if constexpr (UB == 8) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(sp);
                    swu[0] = v.x; swu[1] = v.y; swu[2] = v.z; swu[3] = v.w;
                } else if constexpr (UB == 4) {
                    const uint2 v = *reinterpret_cast<const uint2 *>(sp);
                    swu[0] = v.x; swu[1] = v.y;
                } else if constexpr (UB == 2) {
                    swu[0] = *reinterpret_cast<const uint32_t *>(sp);
                } else {
                    swu[0] = *reinterpret_cast<const uint16_t *>(sp);
                }
            }
            if (!warp_wait(&accfull[u % UNITS], (uint32_t)(u / UNITS) & 1u, a, misc + 1)) { ok = false; break; }
            tc_fence_after();
            const float *sxt = reinterpret_cast<const float *>(smem + LY::OFF_SX + (g % SS) * LY::SX_TILE);
            const uint32_t tu = tbase + (uint32_t)((u % UNITS) * LY::UCOLS);
            if constexpr (NT <= 64) {
                // all UB blocks of the unit in one batch of loads (UB * HT columns)
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
            } else {
                // UB blocks of 128 tokens: this thread's HT columns of each in
                // chunks of 16, the next chunk's load in flight while the
                // current one is scaled (tcgen05.wait::ld waits for all of a
                // thread's loads, so the buffers alternate); the accumulator
                // unit is released as soon as its last chunk has landed
                constexpr int CHB = HT / 16;             // chunks per block
                constexpr int CH = UB * CHB;
                const int mb = m0 + t0;
                uint32_t dbuf[2][16];
                tmem_ld_cols<16>(tu, dbuf[0]);
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    const int j = c / CHB, cc = c % CHB;
                    tmem_ld_wait();
                    if (c + 1 < CH) {
                        const int j1 = (c + 1) / CHB, cc1 = (c + 1) % CHB;
                        tmem_ld_cols<16>(tu + (uint32_t)(j1 * NT + 16 * cc1), dbuf[(c + 1) & 1]);
                    } else {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&accempty[u % UNITS]);
                    }
                    const uint32_t pr = swu[j >> 1];
                    const float sw = __half2float(__ushort_as_half((uint16_t)((j & 1) ? (pr >> 16) : (pr & 0xffffu))));
                    scale_acc<16, DEBUG>(acc + 8 * cc, dbuf[c & 1], sw, sxt + ((bu + j) % SG) * NT + t0 + 16 * cc, n,
                                         mb + 16 * cc, b0 + bu + j, a);
                }
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
            // (the A ring is idle: every MMA has completed)
            float *red = reinterpret_cast<float *>(smem + LY::OFF_A);
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
        if (warp >= LY::EPI0) {
            const int t = threadIdx.x - LY::EPI0 * 32;
            const uint32_t red = sbase + LY::OFF_A;
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

// ------------------------------------------------------------------ host side

constexpr int kSMs = 152;

int nt_for(int M) { return M <= 16 ? 16 : (M <= 32 ? 32 : 64); }

// CTAs along K per 128-row tile: the tile count alone leaves SMs idle for
// narrow layers, so K is split over S CTAs (S in 1..8, 16-block multiples)
// minimising the waves of one-CTA-per-SM launches times the blocks per CTA,
// plus a per-CTA fixed cost of about 24 blocks (pipeline fill, reduction).
int pick_mid_splits(int tiles, int nb) {
    int best = 1;
    long best_cost = -1;
    for (int S = 1; S <= 8; S *= 2) {
        const int bps = SG * ((nb + SG * S - 1) / (SG * S));
        if (S > 1 && (S - 1) * bps >= nb) break;          // a split would be empty
        const long waves = ((long)tiles * S + kSMs - 1) / kSMs;
        const long cost = waves * (bps + 24);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = S;
        }
    }
    return best;
}

template <int NT, bool DEBUG>
w4a8_status launch_nt(const CUtensorMap &tw, const CUtensorMap &tx, const CUtensorMap &tsw, const CUtensorMap &tsx,
                      const MidArgs &a, dim3 grid, cudaStream_t stream) {
    static std::atomic<int> attr_done[w4a8_host::kDeviceSlots];
    const w4a8_status ast = w4a8_host::ensure_smem_limit(gemm_mid_kernel<NT, DEBUG>, Layout<NT>::SMEM, attr_done);
    if (ast != W4A8_OK) return ast;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(Layout<NT>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Layout<NT>::SMEM;
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
    if (cudaLaunchKernelEx(&cfg, gemm_mid_kernel<NT, DEBUG>, tw, tx, tsw, tsx, a) != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    return w4a8_host::launch_status();
}

}  // namespace

namespace w4a8_host {

bool tc_supported(int M, int N, int K) { return M >= 1 && N >= 1 && K >= 256 && K % 256 == 0; }

bool mid_supported(int M, int N, int K) { return M <= 64 && tc_supported(M, N, K); }

int tc_tokens_padded(int M) { return M <= 64 ? nt_for(M) : (M + 127) / 128 * 128; }

int tc_splits(int M, int N, int K) {
    const int mp = tc_tokens_padded(M);
    const int nt = M <= 64 ? mp : 128;
    return pick_mid_splits(((N + BM - 1) / BM) * (mp / nt), K / 32);
}

size_t tc_workspace_bytes(int M, int N, int K) {
    (void)N;
    const size_t mp = (size_t)tc_tokens_padded(M);
    return mp * (size_t)K * 2 + (size_t)(K / 32) * mp * 4;
}

w4a8_status launch_tc_gemm(const uint16_t *q16, const float *sx, const void *packed_w, const uint16_t *scales, int M,
                           int N, int K, uint16_t *out, int32_t *dots, cudaStream_t stream) {
    if (!tc_supported(M, N, K)) return W4A8_ERR_UNSUPPORTED;
    const int mp = tc_tokens_padded(M);
    const int NT = M <= 64 ? mp : 128;
    const int nb = K / 32;
    CUtensorMap tw, tx, tsw, tsx;
    if (!make_tensor_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, packed_w, (uint64_t)K / 2, (uint64_t)N, 128, BM,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, q16, (uint64_t)K, (uint64_t)mp, KS, NT,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_2d(&tsw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, scales, (uint64_t)nb, (uint64_t)N, SWG, BM,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_2d(&tsx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, sx, (uint64_t)mp, (uint64_t)nb, NT, SG,
                            CU_TENSOR_MAP_SWIZZLE_NONE))
        return W4A8_ERR_CUDA;

    MidArgs a;
    a.out = out;
    a.dots = dots;
    a.status = device_status_ptr();
    a.budget = wait_budget();
    a.M = M;
    a.N = N;
    a.nb = nb;
    if (!a.status) return W4A8_ERR_CUDA;
    a.splits = tc_splits(M, N, K);
    a.bps = SG * ((nb + SG * a.splits - 1) / (SG * a.splits));
    const dim3 grid((unsigned)((N + BM - 1) / BM), (unsigned)(mp / NT), (unsigned)a.splits);
    if (NT <= 32) return launch_small_gemm(NT, tw, tx, tsw, tsx, a, grid, stream);
    switch (NT) {
        case 64: return dots ? launch_nt<64, true>(tw, tx, tsw, tsx, a, grid, stream)
                             : launch_nt<64, false>(tw, tx, tsw, tsx, a, grid, stream);
        default: return dots ? launch_nt<128, true>(tw, tx, tsw, tsx, a, grid, stream)
                             : launch_nt<128, false>(tw, tx, tsw, tsx, a, grid, stream);
    }
}

w4a8_status launch_tc_linear(const uint16_t *x, const void *packed_w, const uint16_t *scales, int M, int N, int K,
                             uint16_t *out, int32_t *dots, void *workspace, cudaStream_t stream) {
    if (!tc_supported(M, N, K)) return W4A8_ERR_UNSUPPORTED;
    const int mp = tc_tokens_padded(M);
    uint16_t *q16 = static_cast<uint16_t *>(workspace);
    float *sx = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + (size_t)mp * K * 2);
    w4a8_status st = launch_quant_prefill(x, M, K, mp, q16, sx, stream);
    if (st != W4A8_OK) return st;
    return launch_tc_gemm(q16, sx, packed_w, scales, M, N, K, out, dots, stream);
}

}  // namespace w4a8_host
