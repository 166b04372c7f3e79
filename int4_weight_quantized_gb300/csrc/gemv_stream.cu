// gemv_stream.cu -- decode-phase W4A8 linear that streams each CTA's weight
// rows through a shared-memory ring with bulk asynchronous copies.
//
// Decode is memory-bound: the time is the weight stream ("Що змінює ML Drift
// для on-device AI-інференсу на вашому телефоні?", tech.dede.sh, section
// "Stage-aware оптимізація для великих мовних моделей").  This kernel keeps
// that stream busy:
//   - each CTA owns a contiguous range of output rows; since the packed
//     layout is row-major, the range is one contiguous byte range, copied in
//     chunks of CR whole rows (weights and their fp16 block scales) by one
//     producer warp with cp.async.bulk into an S-deep ring;
//   - the first S chunks, and an L2 prefetch of the activations, are
//     requested before the kernel waits for the previous kernel on the
//     stream (programmatic dependent launch), so a call's weight reads
//     overlap the tail of the call before it; only the activations and the
//     output depend on earlier work;
//   - activations are then quantised in the kernel (the pages' in-kernel
//     activation quantisation) into shared memory, and every lane keeps the
//     codes of its K blocks (l, l+32, l+64, ...) in registers;
//   - one warp computes one whole row at a time: lane l reads its BPL
//     16-byte blocks of the row from the ring (32 int4 weights each), does
//     8 dp4a per block and token and one fp32 multiply-add with s_w * s_x,
//     and the 32 lanes are summed with shuffles; the warp then stores the
//     row's outputs itself, so no cross-warp reduction is needed;
//   - for one token with long rows the K blocks form 2 or 4 groups and as
//     many warps share each row, one group each; their partial sums meet in
//     shared memory and are added in group order.
// Packed weights are stored as w + 8: dp4a of the unsigned nibbles gives
// d + 8*sum(q), and starting the integer accumulator at 0x4B400000 - 8*sum(q)
// leaves the float 1.5*2^23 + d, from which d follows exactly by one fp32
// subtraction.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"

namespace {

using namespace w4a8;

// Consumer warps per CTA, and CTAs per SM the registers are capped for.
// When a lane holds few activation-code words in registers (tokens x code
// slices x weight rows per output <= 2), registers are capped so that three
// launches' CTAs fit on an SM at once: each CTA's weight copies are then
// issued two launches before its rows are needed.  Heavier footprints keep
// their registers (capping them for two CTAs per SM measured slower: the
// rows lose their loads in flight).  (More consumer warps do not help: the
// work after the dependency wait is issue-bound.)
constexpr bool light_cfg(int MT, int BPL, int NV) { return MT * (BPL > 0 ? BPL : 1) * NV <= 2; }
template <int MT, int BPL, int NV>
struct Warps {
    static constexpr bool LIGHT = light_cfg(MT, BPL, NV);
    static constexpr int CW = 8;
    static constexpr int THREADS = (CW + 1) * 32;   // + one producer warp
    static constexpr int MIN_CTAS = LIGHT ? 3 : 1;
};
constexpr int STAGES = 8;
constexpr int STAGE_TARGET = 65536;         // weight bytes per chunk (at least; fewer, larger chunks
                                            // shorten the work after the dependency wait)
constexpr int SMEM_COTENANT = 110 * 1024;   // two CTAs per SM: the next launch's copies start early
constexpr int SMEM_ALONE = 200 * 1024;      // one CTA per SM, for long rows or many tokens
constexpr int SMEM_WHOLE = 224 * 1024;      // one CTA per SM whose rows all fit the ring at once
constexpr int RG_MAX = 4;                   // rows reduced together per warp (compile-time bound)

struct StreamArgs {
    const uint16_t *x;
    const uint8_t *pw;
    const uint16_t *sw;
    uint16_t *out;
    int32_t *dots;       // debug instantiation only
    int *status;
    long long budget;
    int M, N, K, nb;
    int rows_per_cta;    // R
    int cr;              // rows per chunk
    int rg;              // rows per warp and pass, <= RG_MAX and <= 8 / MT
    int sw_bulk;         // scales copied with the weights (nb % 8 == 0)
    size_t stage_bytes;  // weights + scales per stage, 16-byte multiple
    int nslots;          // ring slots (<= STAGES)
    int act;             // gated kernel: 1 = SiLU, 2 = GELU (tanh form)
    const int8_t *xq;    // Q8 input: activation codes [M][K] (natural k order) ...
    const float *xs;     // ... and their block scales [M][K/32]
};

// Activation of the gated kernel's gate branch, from its definition:
// SiLU g / (1 + e^-g); GELU (tanh form) g/2 (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))).
__device__ __forceinline__ float gate_act(int act, float g) {
    if (act == 1) return g / (1.0f + expf(-g));
    const float c = 0.7978845608028654f;    // sqrt(2/pi)
    return 0.5f * g * (1.0f + tanhf(c * (g + 0.044715f * g * g * g)));
}

struct Layout {
    size_t ring, act_codes, act_sx, act_cb, part, bars, total;
};

constexpr int PART_FLOATS = 16;    // >= the partial sums a lane holds per pass (RG * MT * NV, rounded up)

__host__ __device__ inline Layout layout(int MT, int nb, size_t stage_bytes, int nslots, int kg) {
    Layout L;
    size_t o = 0;
    L.ring = o;
    o += (size_t)nslots * stage_bytes;
    L.act_codes = o;
    o += (size_t)MT * nb * 32;
    L.act_sx = o;
    o += (size_t)MT * nb * 4;
    L.act_cb = o;
    o += (size_t)MT * nb * 4;
    o = (o + 15) & ~(size_t)15;
    L.part = o;                     // K-group partial sums: [2 passes][consumer warps][PART_FLOATS]
    if (kg > 1) o += 2 * 8 * PART_FLOATS * 4;
    L.bars = o;
    o += 2 * STAGES * 8;
    L.total = o;
    return L;
}

// Bulk copy global -> shared, marked evict-first in L2: weights are read once
// per call, and should not push the (re-used) activations out of L2.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <int CW>
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(CW * 32) : "memory"); }

// The warps of one row slot (ids 2.. are free: 0 is __syncthreads, 1 the consumers).
__device__ __forceinline__ void slot_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }
constexpr int pow2ceil(int v) { return v <= 1 ? 1 : 2 * pow2ceil((v + 1) / 2); }

// Sums P per-lane values over the 32 lanes of a warp in P - 1 + 5 - log2(P)
// shuffles: each halving step keeps one half of the lane's values (chosen by
// the lane's bit) and sends the other half to the partner lane, which keeps
// the opposite half; the remaining steps are plain butterflies.  Afterwards
// every lane holds the total of value index lane >> (5 - log2(P)).
template <int P>
__device__ __forceinline__ float warp_reduce_halving(float (&v)[P], int lane) {
    constexpr int L = ilog2(P);
#pragma unroll
    for (int l = 0; l < L; ++l) {
        const int bit = 16 >> l;
        const bool up = (lane & bit) != 0;
        const int half = P >> (l + 1);
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float keep = up ? v[i + half] : v[i];
            const float send = up ? v[i] : v[i + half];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
    }
    float t = v[0];
#pragma unroll
    for (int bit = 16 >> L; bit > 0; bit >>= 1) t += __shfl_xor_sync(0xffffffffu, t, bit);
    return t;
}

// BPL > 0: K has BPL slices of 32 blocks and each lane keeps the activation
// codes of its BPL blocks in registers.  BPL == 0: any K; the codes are read
// from shared memory next to each weight block.
// GATED: the weights stack N gate rows over N up rows; every chunk carries
// the gate rows of the CTA's range and the matching up rows, and output row
// n is act(gate_n . x) * (up_n . x) -- the element-wise operators of two
// branches fused into the fully connected operator.
// Q8: the activations arrive already quantised (int8 codes and fp32 block
// scales, e.g. from the RMS-normalisation operator) instead of as fp16 x.
// KG > 1 (codes in registers, one token): the K blocks form KG groups of 32
// BPL blocks, and KG consumer warps share each row, one group each.
template <int MT, int BPL, int KG, bool DEBUG, bool GATED, bool Q8>
__global__ void __launch_bounds__(Warps<MT, BPL, GATED ? 2 : 1>::THREADS, Warps<MT, BPL, GATED ? 2 : 1>::MIN_CTAS)
    gemv_stream_kernel(StreamArgs a) {
    static_assert(!(DEBUG && GATED) && !(DEBUG && Q8), "the debug instantiation is the plain linear");
    constexpr int NV = GATED ? 2 : 1;         // weight rows per output row
    constexpr int CWARPS = Warps<MT, BPL, NV>::CW;
    constexpr int RG = (8 / MT) < RG_MAX ? (8 / MT) : RG_MAX;
    static_assert(CWARPS == 8, "the partial-sum region is sized for 8 consumer warps");
    static_assert(KG == 1 || (BPL > 0 && CWARPS % KG == 0), "K groups need register codes and whole row slots");
    const int rgr = a.rg;
    extern __shared__ __align__(16) uint8_t smem[];
    const Layout L = layout(MT, a.nb, a.stage_bytes, a.nslots, KG);
    const int NS = a.nslots;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + NS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = blockIdx.x * a.rows_per_cta;
    const int r1 = min(a.N, r0 + a.rows_per_cta);
    const int nrows = max(0, r1 - r0);
    const int nchunks = (nrows + a.cr - 1) / a.cr;
    const size_t row_bytes = (size_t)a.K / 2;
    const size_t w_stage = (size_t)a.cr * row_bytes;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CWARPS);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == CWARPS) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // The activations into L2 ahead of the dependency wait: L2 is the
            // point of coherence, so lines the previous kernel writes later
            // are updated there, and the loads after the wait (which do not
            // hit this SM's L1 before it) see its results.  When x comes from
            // a host copy or an older kernel this takes an HBM round trip off
            // the post-wait chain.
            if constexpr (!Q8) {
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.x), "r"((uint32_t)(a.M * a.K * 2))
                             : "memory");
            } else {
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.xq), "r"((uint32_t)(a.M * a.K))
                             : "memory");
            }
            const uint64_t pol = policy_evict_first();
            int issued = 0;
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % NS;
                const uint32_t ph = (uint32_t)(c / NS) & 1u;
                if (!mbar_wait_bounded(&empty[s], ph ^ 1u, a.budget, a.status)) break;
                const int rows = min(a.cr, nrows - c * a.cr);
                const int rr = r0 + c * a.cr;
                const uint32_t wbytes = (uint32_t)(rows * row_bytes);
                const uint32_t sbytes = a.sw_bulk ? (uint32_t)(rows * a.nb * 2) : 0u;
                const uint32_t dst = smem_u32(smem + L.ring + (size_t)s * a.stage_bytes);
                mbar_arrive_expect_tx(&full[s], NV * (wbytes + sbytes));
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const size_t src_row = (size_t)rr + (size_t)v * a.N;     // up rows follow the N gate rows
                    bulk_g2s(dst + (uint32_t)(v * w_stage), a.pw + src_row * row_bytes, wbytes, smem_u32(&full[s]), pol);
                    if (sbytes)
                        bulk_g2s(dst + (uint32_t)(NV * w_stage + (size_t)v * a.cr * a.nb * 2), a.sw + src_row * a.nb,
                                 sbytes, smem_u32(&full[s]), pol);
                }
                if (c == NS - 1 || c == nchunks - 1) pdl_launch_dependents();
                issued = c + 1;
            }
            if (nchunks == 0) pdl_launch_dependents();
            // the CTA must not retire while its copies are still landing
            for (int c = (issued > NS ? issued - NS : 0); c < issued; ++c)
                mbar_wait_bounded(&full[c % NS], (uint32_t)(c / NS) & 1u, a.budget, nullptr);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // Activations may be produced by the previous kernel on the stream.
    pdl_wait();
    uint32_t *codes = reinterpret_cast<uint32_t *>(smem + L.act_codes);
    float *sxs = reinterpret_cast<float *>(smem + L.act_sx);
    int *cbs = reinterpret_cast<int *>(smem + L.act_cb);
    const int tid = threadIdx.x;
    {
        // When all of x takes two rounds of the consumer threads, both
        // rounds' loads are issued before either is quantised (one load
        // latency instead of two); in the four-group instantiation (one
        // token, K > 8192) x of more than four rounds goes four rounds at a
        // time; otherwise longer x keeps one load per round (batched, three
        // or four rounds measured slower, and a four-wide batch in the code
        // slowed the other instantiations).
        const int items = MT * a.nb * 4;
        constexpr int XB = Warps<MT, BPL, NV>::LIGHT ? 1 : (KG >= 4 ? 4 : 2);
        constexpr int STRIDE = CWARPS * 32;
        const int xb = XB == 1 ? 1 : (items <= 2 * STRIDE ? 2 : (XB == 4 && items > 4 * STRIDE ? 4 : 1));
        for (int base0 = 0; base0 < items; base0 += xb * STRIDE) {
            uint4 xv[XB];
            uint2 cv[XB];
            float sxq[XB];
#pragma unroll
            for (int u = 0; u < XB; ++u) {
                const int i = base0 + u * STRIDE + tid;
                xv[u] = make_uint4(0u, 0u, 0u, 0u);
                cv[u] = make_uint2(0u, 0u);
                sxq[u] = 0.0f;
                if (u < xb && i < items) {
                    const int m = i / (a.nb * 4);
                    const int rem = i - m * a.nb * 4;
                    const int b = rem >> 2, t = rem & 3;
                    if constexpr (Q8) {
                        // codes and scale in flight together: the scale does not wait for the code sums
                        cv[u] = *reinterpret_cast<const uint2 *>(a.xq + (size_t)m * a.K + (size_t)b * kBlock + t * 8);
                        if (t == 0) sxq[u] = a.xs[(size_t)m * a.nb + b];
                    } else if (m < a.M) {
                        xv[u] = *reinterpret_cast<const uint4 *>(a.x + (size_t)m * a.K + (size_t)b * kBlock + t * 8);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < XB; ++u) {
                const int ib = base0 + u * STRIDE;
                if (u >= xb || ib >= items) break;   // the same for every consumer thread
                const int i = ib + tid;
                const bool act = i < items;
                int m = 0, b = 0, t = 0;
                if (act) {
                    m = i / (a.nb * 4);
                    const int rem = i - m * a.nb * 4;
                    b = rem >> 2;
                    t = rem & 3;
                }
                if constexpr (Q8) {
                    // 8 codes of this block: even k to one word, odd k to the
                    // other, as the quantiser below packs them; the block's code
                    // sum for the unsigned-weight offset comes from two dp4a with ones
                    int sum = __dp4a((int)cv[u].x, 0x01010101, __dp4a((int)cv[u].y, 0x01010101, 0));
                    sum += __shfl_xor_sync(0xffffffffu, sum, 1, 4);
                    sum += __shfl_xor_sync(0xffffffffu, sum, 2, 4);
                    if (act) {
                        uint32_t *cw = codes + ((size_t)m * a.nb + b) * 8;
                        cw[2 * t] = __byte_perm(cv[u].x, cv[u].y, 0x6420);
                        cw[2 * t + 1] = __byte_perm(cv[u].x, cv[u].y, 0x7531);
                        if (t == 0) {
                            sxs[m * a.nb + b] = sxq[u];
                            cbs[m * a.nb + b] = kMagicBits - 8 * sum;
                        }
                    }
                } else {
                    Quant8 r = quant8_group4(xv[u]);
                    if (act) {
                        uint32_t *cw = codes + ((size_t)m * a.nb + b) * 8;
                        cw[2 * t] = pack_bytes4(r.q[0], r.q[2], r.q[4], r.q[6]);
                        cw[2 * t + 1] = pack_bytes4(r.q[1], r.q[3], r.q[5], r.q[7]);
                        if (t == 0) {
                            sxs[m * a.nb + b] = r.s;
                            cbs[m * a.nb + b] = kMagicBits - 8 * r.sum;
                        }
                    }
                }
            }
        }
    }
    consumer_sync<CWARPS>();

    // Row slots: the KG warps w with equal w / KG compute the same rows, warp
    // w over the K blocks of group w % KG (32 BPL consecutive blocks), and
    // their partial sums meet in shared memory.  Warps past the last whole
    // slot only take part in the chunk hand-offs.
    const int kgi = warp % KG, slot = warp / KG;
    constexpr int nslot = CWARPS / KG;
    // this lane's K blocks (g0 + lane + 32 j) and their activation codes, in registers
    constexpr int BR = BPL > 0 ? BPL : 1;
    const int g0 = kgi * 32 * BR;
    uint32_t qa[MT][BR][8];
    float sxr[MT][BR];
    int cbr[MT][BR];
    if constexpr (BPL > 0) {
#pragma unroll
        for (int j = 0; j < BPL; ++j) {
            const int b = g0 + lane + 32 * j;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (b < a.nb) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(codes + ((size_t)m * a.nb + b) * 8);
                    const uint4 c0 = src[0], c1 = src[1];
                    qa[m][j][0] = c0.x; qa[m][j][1] = c0.y; qa[m][j][2] = c0.z; qa[m][j][3] = c0.w;
                    qa[m][j][4] = c1.x; qa[m][j][5] = c1.y; qa[m][j][6] = c1.z; qa[m][j][7] = c1.w;
                    sxr[m][j] = sxs[m * a.nb + b];
                    cbr[m][j] = cbs[m * a.nb + b];
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) qa[m][j][i] = 0u;
                    sxr[m][j] = 0.0f;
                    cbr[m][j] = kMagicBits;
                }
            }
        }
    }

    const bool reuse = nchunks > NS;         // ring slots are refilled: release them
    // A warp whose wait ran out leaves at once when it computes rows alone;
    // in a slot of several warps it stops waiting but keeps meeting its
    // partners at every slot barrier, so none of them waits forever (the
    // status word already holds the error).
    bool alive = true;
    int pp = 0;                              // pass parity: which half of the partial-sum region
    for (int c = 0; c < nchunks; ++c) {
        const int s = c % NS;
        const uint32_t ph = (uint32_t)(c / NS) & 1u;
        if (alive) {
            bool ok = mbar_wait_bounded(&full[s], ph, a.budget, a.status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if constexpr (KG == 1) return;
                alive = false;
            }
        }
        const uint8_t *wst = smem + L.ring + (size_t)s * a.stage_bytes;
        const uint16_t *sst = reinterpret_cast<const uint16_t *>(wst + NV * w_stage);
        const int rows = min(a.cr, nrows - c * a.cr);
        // RG consecutive rows per warp at a time: their shuffle reductions
        // are independent and overlap
        for (int base = 0; base < rows;) {
            // rows per warp in this pass: at most rgr, and no more than the
            // remaining rows need, so the last pass spreads over all warps
            const int rgp = min(rgr, (rows - base + nslot - 1) / nslot);
            const int rb = base + slot * rgp;
            base += nslot * rgp;
            if (slot >= nslot || rb >= rows) continue;
            // partial sums of this lane: value (g * MT + m) * NV + br is output
            // row rb + g, token m, branch br (0 gate or plain, 1 up)
            constexpr int NVAL = RG * MT * NV;
            constexpr int P = pow2ceil(NVAL);
            float v[P];
#pragma unroll
            for (int i = 0; i < P; ++i) v[i] = 0.0f;
            // one 32-block of a weight row (weights at wp, scale swh) against
            // every token.  Even k sit in the low nibbles, odd k in the high
            // nibbles: masking the high nibbles in place gives 16x the odd
            // weights, so they run in their own dp4a chain, divided by 16
            // (exactly) when the block is done.
            auto block = [&](int g, int br, int n, int b, const uint8_t *wp, uint16_t swh, const uint32_t (*q)[8],
                             const float *sxv, const int *cbv, bool valid) {
                const uint4 w = *reinterpret_cast<const uint4 *>(wp);
                const float swf = __half2float(__ushort_as_half(swh));
                const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    int de = cbv[m], d16 = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        de = dp4a_us(w4[i] & 0x0F0F0F0Fu, q[m][2 * i], de);
                        d16 = dp4a_us(w4[i] & 0xF0F0F0F0u, q[m][2 * i + 1], d16);
                    }
                    const int d = de + (d16 >> 4);
                    if (DEBUG && valid && m < a.M) a.dots[((size_t)m * a.N + n) * a.nb + b] = d - kMagicBits;
                    float &acc = v[(g * MT + m) * NV + br];
                    acc = fmaf(__int_as_float(d) - kMagic, swf * sxv[m], acc);
                }
            };
            // A pass whose RG rows all exist runs without branches, so the
            // compiler can interleave the rows' loads and dp4a chains; a
            // shorter pass stops at its last row.  A block past the row's end
            // reads the last block with zero codes (contributing nothing).
            auto rows_pass = [&](auto full_tag) {
                constexpr bool FULL = decltype(full_tag)::value;
#pragma unroll
                for (int gv = 0; gv < RG * NV; ++gv) {
                    const int g = gv / NV, br = gv % NV;
                    const int rr = rb + g;
                    if constexpr (!FULL) {
                        if (g >= rgp || rr >= rows) break;
                    }
                    const bool rvalid = true;
                    const int n = r0 + c * a.cr + rr;
                    const uint8_t *wrow = wst + (size_t)br * w_stage + (size_t)rr * row_bytes;
                    const uint16_t *srow = sst + (size_t)br * a.cr * a.nb + (size_t)rr * a.nb;
                    const uint16_t *sglob = a.sw + ((size_t)n + (size_t)br * a.N) * a.nb;
                    if constexpr (BPL > 0) {
    #pragma unroll
                        for (int j = 0; j < BPL; ++j) {
                            const int b = g0 + lane + 32 * j;
                            const bool bvalid = b < a.nb;          // codes of such blocks are zero
                            const int bc = bvalid ? b : a.nb - 1;
                            const uint16_t swh = a.sw_bulk ? srow[bc] : __ldg(sglob + bc);
                            uint32_t q[MT][8];
                            float sxv[MT];
                            int cbv[MT];
    #pragma unroll
                            for (int m = 0; m < MT; ++m) {
    #pragma unroll
                                for (int i = 0; i < 8; ++i) q[m][i] = qa[m][j][i];
                                sxv[m] = sxr[m][j];
                                cbv[m] = cbr[m][j];
                            }
                            block(g, br, n, bc, wrow + (size_t)bc * 16, swh, q, sxv, cbv, rvalid && bvalid);
                        }
                    } else {
                        for (int b = lane; b < a.nb; b += 32) {
                            const uint16_t swh = a.sw_bulk ? srow[b] : __ldg(sglob + b);
                            uint32_t q[MT][8];
                            float sxv[MT];
                            int cbv[MT];
    #pragma unroll
                            for (int m = 0; m < MT; ++m) {
                                const uint4 *src = reinterpret_cast<const uint4 *>(codes + ((size_t)m * a.nb + b) * 8);
                                const uint4 c0 = src[0], c1 = src[1];
                                q[m][0] = c0.x; q[m][1] = c0.y; q[m][2] = c0.z; q[m][3] = c0.w;
                                q[m][4] = c1.x; q[m][5] = c1.y; q[m][6] = c1.z; q[m][7] = c1.w;
                                sxv[m] = sxs[m * a.nb + b];
                                cbv[m] = cbs[m * a.nb + b];
                            }
                            block(g, br, n, b, wrow + (size_t)b * 16, swh, q, sxv, cbv, rvalid);
                        }
                    }
                }
            };
            if (rgp == RG && rb + RG <= rows) rows_pass(std::true_type{});
            else rows_pass(std::false_type{});
            float t = warp_reduce_halving<P>(v, lane);
            constexpr int SH = 5 - ilog2(P);             // lanes per value after the reduction: 1 << SH
            static_assert(P <= PART_FLOATS, "partial-sum region too small");
            const int vi = lane >> SH;
            if constexpr (KG > 1) {
                // the slot's partial sums, added in K-group order by its first warp
                float *part = reinterpret_cast<float *>(smem + L.part) + (size_t)pp * CWARPS * PART_FLOATS;
                if ((lane & ((1 << SH) - 1)) == 0) part[warp * PART_FLOATS + vi] = t;
                slot_sync(2 + slot, KG * 32);
                pp ^= 1;
                if (kgi != 0 || !alive) continue;
                for (int g2 = 1; g2 < KG; ++g2) t += part[(slot * KG + g2) * PART_FLOATS + vi];
            }
            if constexpr (GATED) t = gate_act(a.act, t) * __shfl_xor_sync(0xffffffffu, t, 1 << SH);
            const int br = vi % NV, g = (vi / NV) / MT, m = (vi / NV) % MT;
            if ((lane & ((1 << SH) - 1)) == 0 && vi < NVAL && br == 0 && g < rgp && rb + g < rows && m < a.M)
                a.out[(size_t)m * a.N + r0 + c * a.cr + rb + g] = __half_as_ushort(__float2half_rn(t));
        }
        if (reuse) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }
}

struct Plan {
    int MT, BPL, KG, R, cr, rg, sw_bulk, nslots;
    size_t stage_bytes, smem;
    int grid;
    bool ok;
};

constexpr int kSMs = 152;

// Where the activation codes live: BPL blocks per lane (1, 2, 4 or 8) in
// each of KG K groups of 32 BPL blocks (KG warps per row slot).  Several
// tokens keep one group: BPL = K/32 slices rounded up to a power of two
// while tokens x BPL <= 8, else the codes stay in shared memory (BPL = 0).
// One token with rows of more than 4 slices (K > 4096) takes 4 slices per
// lane in 2 or 4 groups (up to K = 16384): the codes of 8 slices, or codes
// read from shared memory, measured slower.
void pick_codes(int MT, int nb, int &bpl, int &kg) {
    const int need = (nb + 31) / 32;
    int b = 1;
    while (b < need) b *= 2;
    kg = 1;
    bpl = (b <= 8 && MT * b <= 8) ? b : 0;
    if (MT == 1 && b > 4 && need <= 16) {
        bpl = 4;
        kg = need <= 8 ? 2 : 4;
    }
}

// Launch plan: each of (up to) 152 CTAs owns R consecutive rows, streamed in
// chunks of cr rows through an nslots-deep ring.  Chunks aim at about a
// quarter of the CTA's bytes (at least 64 KB, so a CTA of up to 64 KB is one
// chunk).  A CTA that needs several fills wants at least three slots, so a
// slot is always being filled while another is read; the ring is sized, in
// this order, for co-resident CTAs (the lightest register footprints: the
// next launches' copies then start during this one) with three slots, for
// one CTA per SM holding all of its rows at once in up to three chunks (up
// to 224 KB), for one CTA
// per SM with three slots (200 KB), and the last two with two.  Within each
// budget the largest chunk wins, but not one below a row per row slot while
// another budget remains.
Plan make_plan(int M, int N, int K, int nv = 1) {
    // nv = weight rows per output row (2 for the gated kernel)
    Plan p{};
    const int nb = K / 32;
    p.MT = M < 8 ? M : 8;
    pick_codes(p.MT, nb, p.BPL, p.KG);
    const size_t row_bytes = (size_t)nv * K / 2;
    p.sw_bulk = (nb % 8) == 0;
    p.R = (N + kSMs - 1) / kSMs;
    p.grid = (N + p.R - 1) / p.R;
    const size_t cta_bytes = (size_t)p.R * row_bytes;
    size_t target = (cta_bytes + 3) / 4;
    if (target < (size_t)STAGE_TARGET) target = STAGE_TARGET;
    int cr0 = (int)(target / row_bytes);
    if (cr0 < 1) cr0 = 1;
    if (cr0 > p.R) cr0 = p.R;
    auto fit = [&](int cr, size_t limit, int min_slots) {
        p.cr = cr;
        p.stage_bytes = ((size_t)cr * row_bytes + (p.sw_bulk ? (size_t)nv * cr * nb * 2 : 0) + 15) & ~(size_t)15;
        const int nch = (p.R + cr - 1) / cr;
        p.nslots = nch < STAGES ? nch : STAGES;
        const int floor_slots = nch < min_slots ? nch : min_slots;
        for (;;) {
            p.smem = layout(p.MT, nb, p.stage_bytes, p.nslots, p.KG).total;
            if (p.smem <= limit || p.nslots <= floor_slots) break;
            --p.nslots;
        }
        return p.smem <= limit;
    };
    const int row_slots = Warps<1, 1, 1>::CW / p.KG;
    const bool share = light_cfg(p.MT, p.BPL, nv);
    struct Budget {
        size_t limit;
        int min_slots;
    };
    // min_slots STAGES + 1: every chunk of the CTA in flight at once
    const Budget budgets[] = {{(size_t)SMEM_COTENANT, 3}, {(size_t)SMEM_WHOLE, STAGES + 1}, {(size_t)SMEM_ALONE, 3},
                              {(size_t)SMEM_COTENANT, 2}, {(size_t)SMEM_ALONE, 2}};
    bool ok = false;
    for (const Budget &b : budgets) {
        if (b.limit == (size_t)SMEM_COTENANT && !share) continue;
        for (int cr = cr0; cr >= 1 && !ok; --cr) {
            ok = fit(cr, b.limit, b.min_slots);
            if (ok && cr < row_slots && cr < cr0) ok = false;
            // all in flight: at most three chunks (more, smaller ones measured slower)
            if (ok && b.min_slots > STAGES && (p.nslots < (p.R + cr - 1) / cr || p.nslots > 3)) ok = false;
        }
        if (ok) break;
    }
    if (!ok) {   // last resort: the largest chunk that fits alone
        for (int cr = cr0; cr >= 1 && !ok; --cr) ok = fit(cr, SMEM_ALONE, 2);
    }
    // rows per warp and pass: the kernel spreads each pass's rows over all
    // row slots (at most this many per slot)
    p.rg = (8 / p.MT) < RG_MAX ? (8 / p.MT) : RG_MAX;
    p.ok = ok;
    return p;
}

template <int MT, int BPL, int KG, bool DEBUG, bool GATED, bool Q8>
w4a8_status launch_t(const Plan &p, const StreamArgs &a, cudaStream_t stream) {
    auto kern = gemv_stream_kernel<MT, BPL, KG, DEBUG, GATED, Q8>;
    static std::atomic<int> attr_done[w4a8_host::kDeviceSlots];
    const w4a8_status ast = w4a8_host::ensure_smem_limit(kern, SMEM_WHOLE, attr_done);
    if (ast != W4A8_OK) return ast;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid, 1, 1);
    cfg.blockDim = dim3(Warps<MT, BPL, GATED ? 2 : 1>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    return w4a8_host::launch_status();
}

template <bool DEBUG, bool GATED, bool Q8>
w4a8_status dispatch(const Plan &p, const StreamArgs &a, cudaStream_t stream) {
    if (p.KG == 2 && p.MT == 1 && p.BPL == 4) return launch_t<1, 4, 2, DEBUG, GATED, Q8>(p, a, stream);
    if (p.KG == 4 && p.MT == 1 && p.BPL == 4) return launch_t<1, 4, 4, DEBUG, GATED, Q8>(p, a, stream);
    if (p.KG != 1) return W4A8_ERR_UNSUPPORTED;
    switch (p.MT * 16 + p.BPL) {
        case 1 * 16 + 1: return launch_t<1, 1, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 1 * 16 + 2: return launch_t<1, 2, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 1 * 16 + 4: return launch_t<1, 4, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 1 * 16 + 8: return launch_t<1, 8, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 2 * 16 + 1: return launch_t<2, 1, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 2 * 16 + 2: return launch_t<2, 2, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 2 * 16 + 4: return launch_t<2, 4, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 3 * 16 + 1: return launch_t<3, 1, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 3 * 16 + 2: return launch_t<3, 2, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 4 * 16 + 1: return launch_t<4, 1, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 4 * 16 + 2: return launch_t<4, 2, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 5 * 16 + 1: return launch_t<5, 1, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 6 * 16 + 1: return launch_t<6, 1, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 7 * 16 + 1: return launch_t<7, 1, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 8 * 16 + 1: return launch_t<8, 1, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 1 * 16 + 0: return launch_t<1, 0, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 2 * 16 + 0: return launch_t<2, 0, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 3 * 16 + 0: return launch_t<3, 0, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 4 * 16 + 0: return launch_t<4, 0, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 5 * 16 + 0: return launch_t<5, 0, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 6 * 16 + 0: return launch_t<6, 0, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 7 * 16 + 0: return launch_t<7, 0, 1, DEBUG, GATED, Q8>(p, a, stream);
        case 8 * 16 + 0: return launch_t<8, 0, 1, DEBUG, GATED, Q8>(p, a, stream);
        default: return W4A8_ERR_UNSUPPORTED;
    }
}

}  // namespace

namespace w4a8_host {

bool gemv_stream_supported(int M, int N, int K) { return make_plan(M < 8 ? M : 8, N, K).ok; }

bool gemv_stream_plan_info(int M, int N, int K, int nv, int *out) {
    const Plan p = make_plan(M < 8 ? M : 8, N, K, nv);
    if (out) {
        const int v[kPlanFields] = {p.MT, p.BPL, p.KG, p.R, p.cr, p.nslots, (int)p.stage_bytes, (int)p.smem, p.grid, p.rg};
        for (int i = 0; i < kPlanFields; ++i) out[i] = v[i];
    }
    return p.ok;
}

bool gemv_stream_preferred(int M, int N, int K) {
    const Plan p = make_plan(M < 8 ? M : 8, N, K);
    return p.ok && (p.BPL > 0 || p.MT <= 2);
}

namespace {

w4a8_status run_stream(const uint16_t *x, const void *packed_w, const uint16_t *scales, int M, int N, int K,
                       uint16_t *out, int32_t *dots, int act, cudaStream_t stream,
                       const int8_t *xq = nullptr, const float *xs = nullptr) {
    int *status = device_status_ptr();
    if (!status) return W4A8_ERR_CUDA;
    const bool gated = act != 0;
    for (int m0 = 0; m0 < M; m0 += 8) {
        const int mc = (M - m0) < 8 ? (M - m0) : 8;
        Plan p = make_plan(mc, N, K, gated ? 2 : 1);
        if (!p.ok) return W4A8_ERR_UNSUPPORTED;
        StreamArgs a;
        a.x = x ? x + (size_t)m0 * K : nullptr;
        a.xq = xq ? xq + (size_t)m0 * K : nullptr;
        a.xs = xs ? xs + (size_t)m0 * (K / 32) : nullptr;
        a.pw = static_cast<const uint8_t *>(packed_w);
        a.sw = scales;
        a.out = out + (size_t)m0 * N;
        a.dots = dots ? dots + (size_t)m0 * N * (K / 32) : nullptr;
        a.status = status;
        a.budget = wait_budget();
        a.M = mc;
        a.N = N;
        a.K = K;
        a.nb = K / 32;
        a.rows_per_cta = p.R;
        a.cr = p.cr;
        a.rg = p.rg;
        a.sw_bulk = p.sw_bulk;
        a.stage_bytes = p.stage_bytes;
        a.nslots = p.nslots;
        a.act = act;
        w4a8_status st = gated ? dispatch<false, true, false>(p, a, stream)
                         : xq ? dispatch<false, false, true>(p, a, stream)
                         : (dots ? dispatch<true, false, false>(p, a, stream) : dispatch<false, false, false>(p, a, stream));
        if (st != W4A8_OK) return st;
    }
    return W4A8_OK;
}

}  // namespace

w4a8_status launch_gemv_stream(const uint16_t *x, const void *packed_w, const uint16_t *scales,
                               int M, int N, int K, uint16_t *out, int32_t *dots, cudaStream_t stream) {
    return run_stream(x, packed_w, scales, M, N, K, out, dots, 0, stream);
}

w4a8_status launch_gemv_stream_q8(const int8_t *codes, const float *sx, const void *packed_w, const uint16_t *scales,
                                  int M, int N, int K, uint16_t *out, cudaStream_t stream) {
    return run_stream(nullptr, packed_w, scales, M, N, K, out, nullptr, 0, stream, codes, sx);
}

bool gemv_stream_gated_supported(int M, int N, int K) { return make_plan(M < 8 ? M : 8, N, K, 2).ok; }

bool gemv_stream_gated_preferred(int M, int N, int K) {
    const Plan p = make_plan(M < 8 ? M : 8, N, K, 2);
    return p.ok && (p.BPL > 0 || p.MT <= 2);
}

w4a8_status launch_gemv_stream_gated(const uint16_t *x, const void *packed_gu, const uint16_t *scales_gu,
                                     int M, int N, int K, uint16_t *out, int act, cudaStream_t stream) {
    if (act != 1 && act != 2) return W4A8_ERR_INVALID_VALUE;
    return run_stream(x, packed_gu, scales_gu, M, N, K, out, nullptr, act, stream);
}

}  // namespace w4a8_host
