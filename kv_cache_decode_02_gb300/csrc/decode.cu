// Split-KV single-query decode attention: one CTA per (split, KV head, sequence).
//
// The computation is flash-decoding as the pages describe it ("Rolling-KV -- overflow
// throughput evaluations", sections 1 and 3: a decode op that emits its own LSE channel;
// "KVARN KV Performance optimizations", items 2, 4, 6 and 9: GQA rows padded to eight
// physical rows, record-contiguous compact plans, fully masked splits skipped, query
// rows sharing every decoded K/V byte, partials merged by max/numerator/denominator).
// The kernel design is our own for sm_103a:
//
//  * warp 2 is the producer.  A 32-cell tile whose valid entries form one physical run
//    (every contiguous cache, and every tile of a compact plan, whose records are
//    positional) is fetched with 3-D tensor-map TMA boxes {128 bytes, 1 head, 32 cells}
//    under the 128-byte swizzle: for f16 head_dim 128, K low/high halves and V
//    low/high halves.  Cells inside the box that are not valid (plan holes, cells past
//    the length) are loaded too and masked.  A tile whose entries are not one run falls
//    back to one 1-D bulk copy per row into a plain row layout.  A ring of n_stages
//    stages, each guarded by a full and an empty mbarrier, keeps up to n_stages tiles
//    in flight per CTA.
//  * warps 0 and 1 each consume 16 cells of every tile.  Masked V rows are zeroed first
//    so that P = 0 never meets a NaN; then S = q K^T on the tensor cores (mma
//    m16n8k16, the G <= 8 query rows of this KV head in M), an online softmax in fp32
//    on exp2-scaled scores, and O^T += V^T P^T (head_dim in M, query rows in N).  Each
//    K/V byte is read from HBM once for all G query heads.
//  * Q8_0 is dequantised as it is consumed: int8 lanes become exact f16 with the
//    magic-number byte permutation, per-32 K scales multiply fp32 block dot products,
//    per-32 V scales are folded into the f16 P operand of each block.  Scales arrive by
//    8/16-byte cp.async per valid cell.
//  * the two consumer warps merge their (m, l, O) through shared memory and write the
//    split's normalised partial O_p and its natural-log LSE_p.
//
// All waits are bounded; a wait that gives up sets a sticky status bit in the workspace
// and the CTA finishes without writing results.
#include <climits>
#include <cmath>
#include <mutex>

#include "kvattn_internal.cuh"

namespace kvattn {

namespace {

constexpr int kMaxStages = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kHeaderBytes = 1024;  // barriers + tile flags; stages start 1024-B aligned
constexpr int kPlaneBytes = kTileCells * 128;  // one 128-B-wide swizzled plane of a tile

constexpr int cmax(int a, int b) { return a > b ? a : b; }

template <int KVT, int D>
struct Geom {
    static constexpr int kRowBytes = KVT == KVATTN_KV_F16 ? 2 * D : D;  // per (cell, KV head)
    static constexpr int kPlanes = kRowBytes / 128;
    static constexpr int kPadRow = kRowBytes;        // per-cell fallback layout: plain rows
    static constexpr int kSclBytes = KVT == KVATTN_KV_Q8_0 ? D / 16 : 0;  // D/32 half scales
    static constexpr int kSwzSection = kPlanes * kPlaneBytes;
    static constexpr int kPadSection = kTileCells * kPadRow;
    static constexpr int kKvArea = cmax(2 * kSwzSection, 2 * kPadSection);
    static constexpr int kKsOff = kKvArea;
    static constexpr int kVsOff = kKsOff + kTileCells * kSclBytes;
    static constexpr int kBytes = (kVsOff + kTileCells * kSclBytes + 1023) / 1024 * 1024;
    static constexpr int kArrivals = KVT == KVATTN_KV_Q8_0 ? 64 : 32;  // + cp.async arrivals
    // end-of-unit exchange area: warp 1's O fragments ([D/16][32 lanes] float4), max, sum
    static constexpr int kXchgBytes = ((D / 16) * 32 * 16 + 64 + 1023) / 1024 * 1024;
    // multi-query: two O tiles per lane, max and sum of 16 rows
    static constexpr int kXchgBytesMQ = (2 * (D / 16) * 32 * 16 + 128 + 1023) / 1024 * 1024;
};

// Byte address of (row r, byte b) of a K or V section in either layout.
// PLANE: bytes between the 128-byte-wide planes of a section (rows per box x 128).
template <bool SWZ, int PAD_ROW, int PLANE = kPlaneBytes>
__device__ __forceinline__ uint32_t sec_addr(uint32_t base, int r, int b) {
    if (SWZ)
        return base + (b >> 7) * PLANE + r * 128 + ((((b >> 4) & 7) ^ (r & 7)) << 4) + (b & 15);
    return base + r * PAD_ROW + b;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// TMA load of one 3-D tensor-map box, completing on an mbarrier, with an L2 cache-policy
// hint (a policy made by createpolicy).  The K/V boxes are read once per call: marking them
// evict-first keeps the L2 for what is read again soon -- the partials the merge reads back
// (a four-sequence GQA-6 decode at split 128 writes 25 MB of them: 101.2 -> 94.8 us per op
// with the hint) and the next call's prefetched tiles.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                                 uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// TMA load of one 4-D tensor-map box (8-bit rows of 256 bytes: both 128-byte planes of the
// box's cells in one copy).
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                                 uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(policy)
        : "memory");
}

// TMA load of one 2-D tensor-map box (the scale planes of the quantised caches).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// L2 prefetch of one tensor-map box (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map), "r"(x), "r"(y),
                 "r"(z)
                 : "memory");
}

__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* map, int x, int y, int z, int w) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(map), "r"(x),
                 "r"(y), "r"(z), "r"(w)
                 : "memory");
}
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Output head_dim index of accumulator slot (m-tile mt, upper half hi) for thread row gq.
template <int KVT>
__device__ __forceinline__ int out_dim(int mt, int hi, int gq) {
    if (KVT == KVATTN_KV_F16) return 16 * mt + 8 * hi + gq;
    // Q8_0: m-tile 2b+hb covers dims 32b + 4*gq + 2*hb + hi (block-aligned permutation)
    return 32 * (mt >> 1) + 4 * gq + 2 * (mt & 1) + hi;
}

// Online-softmax step shared by the consumer paths.  Masks the 2x2 scores a thread holds
// for query row gq and turns them into probabilities against the running reference max
// m_run (log2 units).  The reference only moves when some row's new max exceeds it by more
// than kRescaleSlack, so most tiles skip the rescale of O and l entirely; probabilities
// then stay below 2^kRescaleSlack, which f16 P and the fp32 accumulators hold exactly as
// well as values below 1.  Returns true (warp-uniform) when O and l must be scaled by alpha.
constexpr float kRescaleSlack = 8.f;

__device__ __forceinline__ bool softmax_step(const float (&sacc)[2][4], uint32_t mask, int tq, float scale_log2,
                                             float& m_run, float& alpha, float (&pf)[2][2]) {
    float x[2][2];
    float tmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int c = 8 * j + 2 * tq + e;
            x[j][e] = ((mask >> c) & 1u) ? sacc[j][e] * scale_log2 : -INFINITY;
            tmax = fmaxf(tmax, x[j][e]);
        }
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
    const bool grow = __any_sync(0xffffffffu, tmax > m_run + kRescaleSlack);
    alpha = 1.f;
    if (grow) {
        const float m_new = fmaxf(m_run, tmax);
        alpha = fast_exp2(m_run - ((m_new == -INFINITY) ? 0.f : m_new));
        m_run = m_new;
    }
    const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) pf[j][e] = fast_exp2(x[j][e] - m_use);
    return grow;
}

// O^T accumulators hold rows 2tq, 2tq+1; their alphas come from lanes 8tq and 8tq+4.
template <int D>
__device__ __forceinline__ void rescale_o(float (&oacc)[D / 16][4], float alpha, int tq) {
    const float alpha0 = __shfl_sync(0xffffffffu, alpha, 8 * tq);
    const float alpha1 = __shfl_sync(0xffffffffu, alpha, 8 * tq + 4);
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        oacc[mt][0] *= alpha0;
        oacc[mt][1] *= alpha1;
        oacc[mt][2] *= alpha0;
        oacc[mt][3] *= alpha1;
    }
}

// Q8_0 q.K of one 32-element block b for the two 8-cell n-tiles: exact f16 K lanes, one
// fresh fp32 accumulator per block, then the block's K scale multiplies it into the scores.
__device__ __forceinline__ void q8_qk_block(float (&sacc)[2][4], const uint32_t (&qa0)[2], const uint32_t (&qa1)[2],
                                            const uint32_t (&kw)[2][2], const float (&ksc)[2][2]) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        float cb[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t w0 = kw[j][0] ^ 0x80808080u, w1 = kw[j][1] ^ 0x80808080u;
        mma_16816(cb, qa0[0], 0u, qa0[1], 0u, i8x2_lo(w0), i8x2_hi(w0));
        mma_16816(cb, qa1[0], 0u, qa1[1], 0u, i8x2_lo(w1), i8x2_hi(w1));
        sacc[j][0] = fmaf(cb[0], ksc[j][0], sacc[j][0]);
        sacc[j][1] = fmaf(cb[1], ksc[j][1], sacc[j][1]);
    }
}

// Q8_0 O^T += V^T P'^T for block b (m-tiles 2b, 2b+1).  vw holds the block's 4 bytes of
// head dims 32b + 4gq .. +3 for cells 2tq, 2tq+1, 2tq+8, 2tq+9; pb0/pb1 hold P times the
// cells' V scales.
__device__ __forceinline__ void q8_pv_block(float (&o0)[4], float (&o1)[4], const uint32_t (&vw)[4], uint32_t pb0,
                                            uint32_t pb1) {
    const uint32_t f0 = vw[0] ^ 0x80808080u, f1 = vw[1] ^ 0x80808080u;
    const uint32_t f2 = vw[2] ^ 0x80808080u, f3 = vw[3] ^ 0x80808080u;
    // interleave the two cells of each pair: bytes 0,1 (m-tile 2b) and bytes 2,3 (2b+1)
    const uint32_t u00 = prmt_b32(f0, f1, 0x5140u), u01 = prmt_b32(f0, f1, 0x7362u);
    const uint32_t u10 = prmt_b32(f2, f3, 0x5140u), u11 = prmt_b32(f2, f3, 0x7362u);
    mma_16816(o0, i8x2_lo(u00), i8x2_hi(u00), i8x2_lo(u10), i8x2_hi(u10), pb0, pb1);
    mma_16816(o1, i8x2_lo(u01), i8x2_hi(u01), i8x2_lo(u11), i8x2_hi(u11), pb0, pb1);
}

// Q8_0 scale word (two half scales) of cell `cell` holding block blk; SROW bytes between
// two cells' scale rows.
template <int SROW>
__device__ __forceinline__ uint32_t scale_word(const unsigned char* sc, int cell, int blk) {
    return reinterpret_cast<const uint32_t*>(sc + cell * SROW)[blk >> 1];
}

// One warp's 16 cells of a tile: scores, online softmax, P V (f16 head_dim 256, Q8_0).
// SROW: bytes between two cells' scale rows (Q8_0).
template <int KVT, int D, bool SWZ, int PLANE = kPlaneBytes, int SROW = Geom<KVT, D>::kSclBytes>
__device__ __forceinline__ void consume_tile(uint32_t kb, uint32_t vb, const unsigned char* ks,
                                             const unsigned char* vs, uint32_t mask, int warp, int lane,
                                             const uint32_t (&qa)[D / 16][2], float (&oacc)[D / 16][4], float& m_run, float& l_run,
                                             float scale_log2) {
    using G = Geom<KVT, D>;
    const int gq = lane >> 2;
    const int tq = lane & 3;
    const int r0 = warp * kWarpCells;  // first row of this warp within the tile
    float sacc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;

    // ---- S = q K^T ----
    if (KVT == KVATTN_KV_F16) {
#pragma unroll
        for (int kk = 0; kk < D / 16; kk += 2) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sec_addr<SWZ, G::kPadRow, PLANE>(kb, r0 + 8 * j + (lane & 7), (kk * 16 + 8 * (lane >> 3)) * 2),
                        b0, b1, b2, b3);
                mma_16816(sacc[j], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
                mma_16816(sacc[j], qa[kk + 1][0], 0u, qa[kk + 1][1], 0u, b2, b3);
            }
        }
    } else {
#pragma unroll
        for (int b = 0; b < D / 32; ++b) {
            uint32_t kw[2][2];
            float ksc[2][2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int r = r0 + 8 * j + gq;
                // block b, half hb: d = 32b + 16hb + 4tq + {0,1 | 2,3}
                kw[j][0] = lds32(sec_addr<SWZ, G::kPadRow, PLANE>(kb, r, 32 * b + 4 * tq));
                kw[j][1] = lds32(sec_addr<SWZ, G::kPadRow, PLANE>(kb, r, 32 * b + 16 + 4 * tq));
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    ksc[j][e] = __half2float(
                        reinterpret_cast<const __half*>(ks + (r0 + 8 * j + 2 * tq + e) * SROW)[b]);
            }
            q8_qk_block(sacc, qa[2 * b], qa[2 * b + 1], kw, ksc);
        }
    }

    float alpha, pf[2][2];
    const bool grow = softmax_step(sacc, mask, tq, scale_log2, m_run, alpha, pf);
    if (grow) {
        rescale_o<D>(oacc, alpha, tq);
        l_run *= alpha;
    }

    // ---- O^T += V^T P^T ----
    if (KVT == KVATTN_KV_F16) {
        // l sums the fp32 probabilities (the LSE stays exact to fp32 even over a handful of
        // cells); the MMA weights are their f16 roundings
        uint32_t pb[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) pb[j] = pack_half2(pf[j][0], pf[j][1]);
        l_run += (pf[0][0] + pf[0][1]) + (pf[1][0] + pf[1][1]);
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(sec_addr<SWZ, G::kPadRow, PLANE>(vb, r0 + (lane & 7) + 8 * (lane >> 4),
                                                    (16 * mt + 8 * ((lane >> 3) & 1)) * 2),
                          a0, a1, a2, a3);
            mma_16816(oacc[mt], a0, a1, a2, a3, pb[0], pb[1]);
        }
    } else {
        l_run += (pf[0][0] + pf[0][1]) + (pf[1][0] + pf[1][1]);
        const uint32_t ph0 = pack_half2(pf[0][0], pf[0][1]);
        const uint32_t ph1 = pack_half2(pf[1][0], pf[1][1]);
        const int c0 = r0 + 2 * tq;
#pragma unroll
        for (int b = 0; b < D / 32; ++b) {
            const uint32_t s01 = prmt_b32(scale_word<SROW>(vs, c0, b), scale_word<SROW>(vs, c0 + 1, b),
                                          (b & 1) ? 0x7632u : 0x5410u);
            const uint32_t s89 = prmt_b32(scale_word<SROW>(vs, c0 + 8, b), scale_word<SROW>(vs, c0 + 9, b),
                                          (b & 1) ? 0x7632u : 0x5410u);
            const int off = 32 * b + 4 * gq;
            const uint32_t vw[4] = {lds32(sec_addr<SWZ, G::kPadRow, PLANE>(vb, c0, off)),
                                    lds32(sec_addr<SWZ, G::kPadRow, PLANE>(vb, c0 + 1, off)),
                                    lds32(sec_addr<SWZ, G::kPadRow, PLANE>(vb, c0 + 8, off)),
                                    lds32(sec_addr<SWZ, G::kPadRow, PLANE>(vb, c0 + 9, off))};
            q8_pv_block(oacc[2 * b], oacc[2 * b + 1], vw, hmul2_u32(ph0, s01), hmul2_u32(ph1, s89));
        }
    }
}

// f16 head_dim 128: the warp copies every K/V fragment of its 16 cells into registers,
// releases the stage to the producer at once, and only then computes, so the stage is
// refilled while the tensor-core work runs.
template <bool SWZ>
__device__ __forceinline__ void consume_tile_staged(uint32_t kb, uint32_t vb, uint32_t mask, int warp, int lane,
                                                    uint32_t empty_bar, const uint32_t (&qa)[8][2],
                                                    float (&oacc)[8][4], float& m_run, float& l_run,
                                                    float scale_log2) {
    constexpr int D = 128;
    using G = Geom<KVATTN_KV_F16, D>;
    const int tq = lane & 3;
    const int r0 = warp * kWarpCells;
    float sacc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;

    uint32_t kf[2][4][4];
    uint32_t vf[8][4];
#pragma unroll
    for (int kp = 0; kp < 4; ++kp)
#pragma unroll
        for (int j = 0; j < 2; ++j)
            ldsm_x4(sec_addr<SWZ, G::kPadRow>(kb, r0 + 8 * j + (lane & 7), (2 * kp * 16 + 8 * (lane >> 3)) * 2),
                    kf[j][kp][0], kf[j][kp][1], kf[j][kp][2], kf[j][kp][3]);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
        ldsm_x4_trans(sec_addr<SWZ, G::kPadRow>(vb, r0 + (lane & 7) + 8 * (lane >> 4),
                                                (16 * mt + 8 * ((lane >> 3) & 1)) * 2),
                      vf[mt][0], vf[mt][1], vf[mt][2], vf[mt][3]);
    __syncwarp();
    mbar_arrive(empty_bar);  // every lane: its shared-memory reads are done
#pragma unroll
    for (int kp = 0; kp < 4; ++kp)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            mma_16816(sacc[j], qa[2 * kp][0], 0u, qa[2 * kp][1], 0u, kf[j][kp][0], kf[j][kp][1]);
            mma_16816(sacc[j], qa[2 * kp + 1][0], 0u, qa[2 * kp + 1][1], 0u, kf[j][kp][2], kf[j][kp][3]);
        }
    float alpha, pf[2][2];
    if (softmax_step(sacc, mask, tq, scale_log2, m_run, alpha, pf)) {
        rescale_o<D>(oacc, alpha, tq);
        l_run *= alpha;
    }
    // l sums the fp32 probabilities; the MMA weights are their f16 roundings
    uint32_t pb[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) pb[j] = pack_half2(pf[j][0], pf[j][1]);
    l_run += (pf[0][0] + pf[0][1]) + (pf[1][0] + pf[1][1]);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) mma_16816(oacc[mt], vf[mt][0], vf[mt][1], vf[mt][2], vf[mt][3], pb[0], pb[1]);
}

// Query row of lane row gq: single-query (rg < 0) the query head g G + gq of sequence s; in
// the 8-row multi-query units of the quantised head_dim-256 kernels, row r = 8 rg + gq of
// the unit's KV head, token r / G, query head g G + r % G.  ok: the row exists.
template <int D>
__device__ __forceinline__ const uint32_t* q_row_ptr(const SplitDecodeParams& p, int s, int g, int gq, int rg,
                                                     bool& ok) {
    if (rg < 0) {
        ok = gq < p.group;
        const int h = g * p.group + (ok ? gq : 0);
        return reinterpret_cast<const uint32_t*>(p.q + ((int64_t)s * p.n_head + h) * D);
    }
    const int r = 8 * rg + gq;
    ok = r < p.group * p.n_q;
    const int t = ok ? r / p.group : 0;
    const int h = g * p.group + (ok ? r % p.group : 0);
    return reinterpret_cast<const uint32_t*>(p.q + (((int64_t)s * p.n_q + t) * p.n_head + h) * D);
}

// Loads the query fragments of (sequence s, KV head g): the GQA rows of the head fill the
// first `group` rows of the m16n8k16 A operand (rows 8-15 and rows >= group stay zero).
template <int KVT, int D>
__device__ __forceinline__ void load_q_frags(const SplitDecodeParams& p, int s, int g, int gq, int tq,
                                             uint32_t (&qa)[D / 16][2], int rg = -1) {
    bool row_ok;
    const uint32_t* qrow = q_row_ptr<D>(p, s, g, gq, rg, row_ok);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        int d0, d1;
        if (KVT == KVATTN_KV_F16) {
            d0 = 16 * kk + 2 * tq;
            d1 = d0 + 8;
        } else {
            d0 = 32 * (kk >> 1) + 16 * (kk & 1) + 4 * tq;
            d1 = d0 + 2;
        }
        qa[kk][0] = row_ok ? __ldg(qrow + d0 / 2) : 0u;
        qa[kk][1] = row_ok ? __ldg(qrow + d1 / 2) : 0u;
    }
}

// Query fragments in the element order of the Q4_0 key path (q4_qk_block): for the MMA of
// block b, half h, the k pairs (2tq, 2tq+1) and (2tq+8, 2tq+9) hold elements (e, e+2) and
// (e+1, e+3) with e = 32b + 16h + 4tq.
template <int D>
__device__ __forceinline__ void load_q_frags_q4k(const SplitDecodeParams& p, int s, int g, int gq, int tq,
                                                 uint32_t (&qa)[D / 16][2], int rg = -1) {
    bool row_ok;
    const uint32_t* qrow = q_row_ptr<D>(p, s, g, gq, rg, row_ok);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const int e = 32 * (kk >> 1) + 16 * (kk & 1) + 4 * tq;
        const uint32_t w0 = row_ok ? __ldg(qrow + e / 2) : 0u;      // elements e, e+1
        const uint32_t w1 = row_ok ? __ldg(qrow + e / 2 + 1) : 0u;  // elements e+2, e+3
        qa[kk][0] = prmt_b32(w0, w1, 0x5410u);  // (e, e+2)
        qa[kk][1] = prmt_b32(w0, w1, 0x7632u);  // (e+1, e+3)
    }
}

// Query fragments of a head-pair unit (the head_dim-256 kernels reading a head_dim-128 cache
// as 256-byte rows of KV heads 2g2 and 2g2+1): rows gq < G are query heads 2 g2 G + gq of the
// first head and fill dims 0-127, rows G .. 2G-1 belong to the second head and fill dims
// 128-255; the other half of every row is zero, so each score is its own head's q.K.  The
// element order is load_q_frags' (8-bit keys) or load_q_frags_q4k's (4-bit keys).
template <bool KQ4>
__device__ __forceinline__ void load_q_frags_pair(const SplitDecodeParams& p, int s, int g2, int gq, int tq,
                                                  uint32_t (&qa)[16][2]) {
    const int G = p.group >> 1;
    const bool ok = gq < p.group;
    const int hi = gq >= G ? 1 : 0;
    const int h = g2 * p.group + (ok ? gq : 0);
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + ((int64_t)s * p.n_head + h) * 128);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
        const bool mine = ok && (kk >= 8) == (hi != 0);
        const int e = (32 * (kk >> 1) + 16 * (kk & 1) + 4 * tq) & 127;  // element within the row's half
        if (KQ4) {
            const uint32_t w0 = mine ? __ldg(qrow + e / 2) : 0u;
            const uint32_t w1 = mine ? __ldg(qrow + e / 2 + 1) : 0u;
            qa[kk][0] = prmt_b32(w0, w1, 0x5410u);
            qa[kk][1] = prmt_b32(w0, w1, 0x7632u);
        } else {
            qa[kk][0] = mine ? __ldg(qrow + e / 2) : 0u;
            qa[kk][1] = mine ? __ldg(qrow + (e + 2) / 2) : 0u;
        }
    }
}

// One work unit = (sequence, split, KV head).  Units are numbered with the KV head fastest,
// so the CTAs that run side by side read the rows of every head of the same cells.
struct Unit {
    int s, g;
    int rg;           // multi-query row group (0 without row groups)
    int64_t split_idx;
    int64_t len;      // the sequence's clamped length
    int64_t i0, i1;   // plan entries / cells [i0, i1) of the split
    int n_tiles;      // 0: nothing to read
    bool write_empty; // an empty unit still reports (0, -inf)
};

__device__ __forceinline__ Unit unit_at(const SplitDecodeParams& p, int64_t u) {
    Unit x;
    // unit counts fit in 32 bits (checked on the host): 32-bit division is far cheaper
    const uint32_t uu = (uint32_t)u, us = (uint32_t)p.unit_splits;
    uint32_t r;
    if (p.n_rg > 1) {
        const uint32_t nrg = (uint32_t)p.n_rg, hkv = (uint32_t)p.n_head_kv * nrg;
        r = uu / hkv;
        const uint32_t gv = uu - r * hkv;
        x.g = (int)(gv / nrg);
        x.rg = (int)(gv - (uint32_t)x.g * nrg);
    } else {
        const uint32_t hk = (uint32_t)p.n_head_kv;
        r = uu / hk;
        x.g = (int)(uu - r * hk);
        x.rg = 0;
    }
    const uint32_t si = r / us;
    x.split_idx = (int64_t)(r - si * us);
    x.s = (int)si;
    const int64_t cap = p.plan ? p.plan_stride : p.n_cells;
    // (the length and the descriptor are independent loads: issue both before using either)
    int64_t L = p.seq_lens != nullptr ? (int64_t)__ldg(p.seq_lens + x.s) : p.fixed_len;
    const int desc_valid = p.desc != nullptr ? __ldg(&p.desc[(int64_t)x.s * p.n_split + x.split_idx].x) : 1;
    L = L < 0 ? 0 : L;
    L = L < p.max_len ? L : p.max_len;
    L = L < cap ? L : cap;
    x.i0 = x.split_idx * p.split;
    x.len = L;
    x.i1 = (x.i0 + p.split < L) ? x.i0 + p.split : L;
    const bool empty = x.i0 >= x.i1 || desc_valid == 0;
    x.n_tiles = empty ? 0 : (int)((x.i1 - x.i0 + kTileCells - 1) / kTileCells);
    // A fully masked split inside the length reports (0, -inf) for the merge; a split past
    // the length writes only when the caller asked for every partial slot.
    x.write_empty = empty && (x.i0 < x.i1 || p.write_beyond);
    return x;
}

// The query rows a unit reads are those of its (sequence, KV head, row group): units with the
// same key share their query fragments, so a warp reloads them only when the key changes
// (a CTA's successive units mostly keep the sequence and KV head).
__device__ __forceinline__ int64_t q_key(const SplitDecodeParams& p, const Unit& x) {
    return ((int64_t)x.s * p.n_head_kv + x.g) * 256 + x.rg;
}

// ---------------------------------------------------------------------------------------
// Causal multi-query decode (f16, head_dim 128).  The G x n_q query rows of a KV head
// (row r = token r / G, query head g*G + r % G) fill the whole M of the q.K^T MMA -- a
// lane holds rows gq and gq + 8 -- and two N = 8 tiles of the P V MMA.  Each row keeps its
// own running max and sum; row r sees the cells at logical positions below
// L - n_q + 1 + r / G (its token's own position and everything before it).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void load_q_frags_mq(const SplitDecodeParams& p, int s, int g, int gq, int tq,
                                                int row0, uint32_t (&qa)[8][4]) {
    constexpr int D = 128;
    const int rows = p.group * p.n_q;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = row0 + gq + 8 * half;
        const bool ok = r < rows;
        const int t = ok ? r / p.group : 0;
        const int h = g * p.group + (ok ? r % p.group : 0);
        const uint32_t* qrow =
            reinterpret_cast<const uint32_t*>(p.q + (((int64_t)s * p.n_q + t) * p.n_head + h) * D);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int d0 = 16 * kk + 2 * tq;
            qa[kk][2 * half] = ok ? __ldg(qrow + d0 / 2) : 0u;
            qa[kk][2 * half + 1] = ok ? __ldg(qrow + (d0 + 8) / 2) : 0u;
        }
    }
}

// One warp's 16 cells of a tile for the 16 query rows.  lim[hh]: cells c < lim[hh] of the
// warp's 16 are inside the causal window of the lane's row gq + 8 hh.
template <bool SWZ>
__device__ __forceinline__ void mq_tile(uint32_t kb, uint32_t vb, uint32_t mask, int warp, int lane,
                                        const int (&lim)[2], const uint32_t (&qa)[8][4], float (&oacc)[2][8][4],
                                        float (&m_run)[2], float (&l_run)[2], float scale_log2) {
    constexpr int D = 128;
    using G = Geom<KVATTN_KV_F16, D>;
    const int tq = lane & 3;
    const int r0 = warp * kWarpCells;
    float sacc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; kk += 2) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(sec_addr<SWZ, G::kPadRow>(kb, r0 + 8 * j + (lane & 7), (kk * 16 + 8 * (lane >> 3)) * 2), b0,
                    b1, b2, b3);
            mma_16816(sacc[j], qa[kk][0], qa[kk][2], qa[kk][1], qa[kk][3], b0, b1);
            mma_16816(sacc[j], qa[kk + 1][0], qa[kk + 1][2], qa[kk + 1][1], qa[kk + 1][3], b2, b3);
        }
    }
    // online softmax, one (max, sum) per row: hh = 0 -> row gq, hh = 1 -> row gq + 8
    float x[2][2][2];
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int c = 8 * j + 2 * tq + e;
                const bool ok = ((mask >> c) & 1u) && c < lim[hh];
                x[hh][j][e] = ok ? sacc[j][2 * hh + e] * scale_log2 : -INFINITY;
                tmax[hh] = fmaxf(tmax[hh], x[hh][j][e]);
            }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        tmax[hh] = fmaxf(tmax[hh], __shfl_xor_sync(0xffffffffu, tmax[hh], 1));
        tmax[hh] = fmaxf(tmax[hh], __shfl_xor_sync(0xffffffffu, tmax[hh], 2));
    }
    const bool grow = __any_sync(0xffffffffu, tmax[0] > m_run[0] + kRescaleSlack || tmax[1] > m_run[1] + kRescaleSlack);
    if (grow) {
        float alpha[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const float m_new = fmaxf(m_run[hh], tmax[hh]);
            alpha[hh] = fast_exp2(m_run[hh] - ((m_new == -INFINITY) ? 0.f : m_new));
            m_run[hh] = m_new;
            l_run[hh] *= alpha[hh];
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const float a0 = __shfl_sync(0xffffffffu, alpha[nt], 8 * tq);
            const float a1 = __shfl_sync(0xffffffffu, alpha[nt], 8 * tq + 4);
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                oacc[nt][mt][0] *= a0;
                oacc[nt][mt][1] *= a1;
                oacc[nt][mt][2] *= a0;
                oacc[nt][mt][3] *= a1;
            }
        }
    }
    uint32_t pb[2][2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const float m_use = (m_run[hh] == -INFINITY) ? 0.f : m_run[hh];
        float psum = 0.f;  // over the fp32 probabilities (the MMA weights are their f16 roundings)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float p0 = fast_exp2(x[hh][j][0] - m_use), p1 = fast_exp2(x[hh][j][1] - m_use);
            pb[hh][j] = pack_half2(p0, p1);
            psum += p0 + p1;
        }
        l_run[hh] += psum;
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(sec_addr<SWZ, G::kPadRow>(vb, r0 + (lane & 7) + 8 * (lane >> 4), (16 * mt + 8 * ((lane >> 3) & 1)) * 2),
                      a0, a1, a2, a3);
        mma_16816(oacc[0][mt], a0, a1, a2, a3, pb[0][0], pb[0][1]);
        mma_16816(oacc[1][mt], a0, a1, a2, a3, pb[1][0], pb[1][1]);
    }
}

// A whole 32-cell tile for the warp's 16 query rows (the row-split layouts): four
// independent q.K^T accumulator chains instead of two per 16-cell half, one max and sum
// reduction per row and tile, and P V over k = 32 cells.  lim[hh]: cells c < lim[hh] of the
// tile are inside the causal window of the lane's row gq + 8 hh.  The caller has zeroed the
// V rows of masked cells that came in with a TMA box.
template <bool SWZ>
__device__ __forceinline__ void mq_tile32(uint32_t kb, uint32_t vb, uint32_t mask, int lane, const int (&lim)[2],
                                          const uint32_t (&qa)[8][4], float (&oacc)[2][8][4], float (&m_run)[2],
                                          float (&l_run)[2], float scale_log2) {
    constexpr int D = 128;
    using G = Geom<KVATTN_KV_F16, D>;
    const int tq = lane & 3;
    float sacc[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; kk += 2) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(sec_addr<SWZ, G::kPadRow>(kb, 8 * j + (lane & 7), (kk * 16 + 8 * (lane >> 3)) * 2), b0, b1, b2, b3);
            mma_16816(sacc[j], qa[kk][0], qa[kk][2], qa[kk][1], qa[kk][3], b0, b1);
            mma_16816(sacc[j], qa[kk + 1][0], qa[kk + 1][2], qa[kk + 1][1], qa[kk + 1][3], b2, b3);
        }
    }
    float x[2][4][2];
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int c = 8 * j + 2 * tq + e;
                const bool ok = ((mask >> c) & 1u) && c < lim[hh];
                x[hh][j][e] = ok ? sacc[j][2 * hh + e] * scale_log2 : -INFINITY;
                tmax[hh] = fmaxf(tmax[hh], x[hh][j][e]);
            }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        tmax[hh] = fmaxf(tmax[hh], __shfl_xor_sync(0xffffffffu, tmax[hh], 1));
        tmax[hh] = fmaxf(tmax[hh], __shfl_xor_sync(0xffffffffu, tmax[hh], 2));
    }
    const bool grow = __any_sync(0xffffffffu, tmax[0] > m_run[0] + kRescaleSlack || tmax[1] > m_run[1] + kRescaleSlack);
    if (grow) {
        float alpha[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const float m_new = fmaxf(m_run[hh], tmax[hh]);
            alpha[hh] = fast_exp2(m_run[hh] - ((m_new == -INFINITY) ? 0.f : m_new));
            m_run[hh] = m_new;
            l_run[hh] *= alpha[hh];
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const float a0 = __shfl_sync(0xffffffffu, alpha[nt], 8 * tq);
            const float a1 = __shfl_sync(0xffffffffu, alpha[nt], 8 * tq + 4);
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                oacc[nt][mt][0] *= a0;
                oacc[nt][mt][1] *= a1;
                oacc[nt][mt][2] *= a0;
                oacc[nt][mt][3] *= a1;
            }
        }
    }
    uint32_t pb[2][4];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const float m_use = (m_run[hh] == -INFINITY) ? 0.f : m_run[hh];
        float psum = 0.f;  // over the fp32 probabilities (the MMA weights are their f16 roundings)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float p0 = fast_exp2(x[hh][j][0] - m_use), p1 = fast_exp2(x[hh][j][1] - m_use);
            pb[hh][j] = pack_half2(p0, p1);
            psum += p0 + p1;
        }
        l_run[hh] += psum;
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(sec_addr<SWZ, G::kPadRow>(vb, 16 * ks + (lane & 7) + 8 * (lane >> 4),
                                                    (16 * mt + 8 * ((lane >> 3) & 1)) * 2),
                          a0, a1, a2, a3);
            mma_16816(oacc[0][mt], a0, a1, a2, a3, pb[0][2 * ks], pb[0][2 * ks + 1]);
            mma_16816(oacc[1][mt], a0, a1, a2, a3, pb[1][2 * ks], pb[1][2 * ks + 1]);
        }
}

// The consumer warps of the multi-query kernel: the same ring and unit walk as the
// single-query consumers (partial row of (token t, head h) = t * n_head + h).  Up to 16 query
// rows per KV head, each warp attends to its 16 cells of every tile for all rows and the
// two warps meet in the doubled end-of-unit exchange; with 17 to 32 rows, warp w takes rows
// 16w .. 16w+15 over all 32 cells of every tile and writes them itself (no exchange); with
// 33 to 128 rows, each group of 32 rows is a unit of its own in the same way (the groups of
// a split are neighbouring units, so the second reads the split's K/V from L2).  Beyond 16
// rows the tcgen05 kernel (decode_tc.cu) takes most calls; these layouts serve the others.
__device__ __forceinline__ void mq_consumers(const SplitDecodeParams& p, uint64_t* full_bar, uint64_t* empty_bar,
                                             const uint32_t* tile_mask, const uint32_t* tile_swz,
                                             volatile int* abort_flag, uint64_t* xchg_bar, unsigned char* xchg,
                                             unsigned char* stages, int n_stages, int64_t n_units, int warp,
                                             int lane) {
    constexpr int D = 128;
    using G = Geom<KVATTN_KV_F16, D>;
    const int gq = lane >> 2;
    const int tq = lane & 3;
    const int H = p.n_head, GQ = p.group, NQ = p.n_q;
    const int rows = GQ * NQ;
    const int grp = p.n_rg > 1 ? p.rg_rows : rows;  // rows of one unit (a row group's, or all)
    const bool rsplit = grp > 16;  // the warps split the rows instead of the cells
    // first row of this warp in a unit
    auto first_row = [&](const Unit& y) { return p.rg_rows * y.rg + (rsplit ? 16 * warp : 0); };
    const int64_t HR = (int64_t)NQ * H;  // partial rows per (sequence, split)
    float4* xo = reinterpret_cast<float4*>(xchg);      // [2][D/16][32 lanes]
    float* xm = reinterpret_cast<float*>(xo + 2 * (D / 16) * 32);  // [16] max
    float* xl = xm + 16;                                            // [16] sum
    constexpr float kLn2 = 0.69314718055994530942f;
    uint32_t qa[8][4];
    int64_t qa_key = -1;  // q_key of the rows whose query fragments qa holds
    uint32_t T = 0, X = 0;
    bool stop = false;
    for (int64_t u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
        const Unit x = unit_at(p, u);
        const int64_t part = (int64_t)x.s * p.part_stride + p.part_base + x.split_idx;
        const int row0 = first_row(x);
        if (x.n_tiles == 0) {
            if (warp == 0 && x.write_empty) {
                // the unit's rows: its row group's, or every row without row groups
                const int rb = p.rg_rows * x.rg;
                const int n_rows = rows - rb < grp ? rows - rb : grp;
                for (int idx = lane; idx < n_rows * D; idx += 32) {
                    const int r = rb + idx / D;
                    const int d = idx % D;
                    const int64_t row = (int64_t)(r / GQ) * H + x.g * GQ + r % GQ;
                    p.part_o[(part * HR + row) * D + d] = 0.f;
                    if (d == 0) p.part_lse[part * HR + row] = -INFINITY;
                }
            }
            continue;
        }
        if (qa_key != q_key(p, x)) {
            load_q_frags_mq(p, x.s, x.g, gq, tq, row0, qa);
            qa_key = q_key(p, x);
        }
        float oacc[2][8][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 8; ++i) oacc[nt][i][0] = oacc[nt][i][1] = oacc[nt][i][2] = oacc[nt][i][3] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
        // causal limit (logical position, exclusive) of the lane's rows row0 + gq and row0 + gq + 8
        const int64_t lim_row[2] = {x.len - NQ + 1 + (row0 + gq) / GQ, x.len - NQ + 1 + (row0 + gq + 8) / GQ};
        for (int t = 0; t < x.n_tiles; ++t, ++T) {
            const int st = (int)(T % (uint32_t)n_stages);
            const uint32_t use = T / (uint32_t)n_stages;
            const bool ok = mbar_wait_bounded(smem_addr(&full_bar[st]), use & 1u, abort_flag, p.wait_limit_ns);
            if (!__all_sync(0xffffffffu, ok)) {
                stop = true;
                break;
            }
            const bool swz = tile_swz[st] != 0u;
            unsigned char* stage = stages + st * G::kBytes;
            // hw: the 16-cell half of the tile
            auto half = [&](int hw) {
                const uint32_t mask = (tile_mask[st] >> (hw * kWarpCells)) & 0xffffu;
                if (mask == 0u) return;
                const int64_t p0 = x.i0 + (int64_t)t * kTileCells + hw * kWarpCells;
                int lim[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int64_t rel = lim_row[hh] - p0;
                    lim[hh] = rel < 0 ? 0 : (rel > kWarpCells ? kWarpCells : (int)rel);
                }
                if (swz) {
                    const uint32_t kb = smem_addr(stage);
                    if (mask != 0xffffu) {
                        // masked rows came in with the box: zero their V rows (with split rows
                        // both warps write the same zeros, each before its own reads)
                        const int r = hw * kWarpCells + (lane & 15);
                        if (lane < 16 && !((mask >> lane) & 1u)) {
#pragma unroll
                            for (int pl = 0; pl < G::kPlanes; ++pl) {
                                uint4* z = reinterpret_cast<uint4*>(stage + G::kSwzSection + pl * kPlaneBytes + r * 128);
#pragma unroll
                                for (int k = 0; k < 8; ++k) z[k] = make_uint4(0, 0, 0, 0);
                            }
                            fence_proxy_async();
                        }
                        __syncwarp();
                    }
                    mq_tile<true>(kb, kb + G::kSwzSection, mask, hw, lane, lim, qa, oacc, m_run, l_run, p.scale_log2);
                } else {
                    const uint32_t kb = smem_addr(stage);
                    mq_tile<false>(kb, kb + G::kPadSection, mask, hw, lane, lim, qa, oacc, m_run, l_run,
                                   p.scale_log2);
                }
            };
            if (rsplit) {
                // the whole tile: zero the V rows of masked cells that came with the box (every
                // warp writes the same zeros, each before its own reads), then one 32-cell pass
                const uint32_t mask = tile_mask[st];
                if (mask != 0u) {
                    const int64_t p0 = x.i0 + (int64_t)t * kTileCells;
                    int lim[2];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int64_t rel = lim_row[hh] - p0;
                        lim[hh] = rel < 0 ? 0 : (rel > kTileCells ? kTileCells : (int)rel);
                    }
                    const uint32_t kb = smem_addr(stage);
                    if (swz) {
                        if (mask != 0xffffffffu) {
                            if (!((mask >> lane) & 1u)) {
#pragma unroll
                                for (int pl = 0; pl < G::kPlanes; ++pl) {
                                    uint4* z = reinterpret_cast<uint4*>(stage + G::kSwzSection + pl * kPlaneBytes +
                                                                        lane * 128);
#pragma unroll
                                    for (int k = 0; k < 8; ++k) z[k] = make_uint4(0, 0, 0, 0);
                                }
                                fence_proxy_async();
                            }
                            __syncwarp();
                        }
                        mq_tile32<true>(kb, kb + G::kSwzSection, mask, lane, lim, qa, oacc, m_run, l_run, p.scale_log2);
                    } else {
                        mq_tile32<false>(kb, kb + G::kPadSection, mask, lane, lim, qa, oacc, m_run, l_run,
                                         p.scale_log2);
                    }
                }
            } else {
                half(warp);
            }
            __syncwarp();
            mbar_arrive(smem_addr(&empty_bar[st]));
        }
        if (stop) break;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 1);
            l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 2);
        }
        const int64_t un = u + gridDim.x;
        if (un < n_units) {
            const Unit y = unit_at(p, un);
            if (y.n_tiles > 0 && q_key(p, y) != qa_key) {
                load_q_frags_mq(p, y.s, y.g, gq, tq, first_row(y), qa);
                qa_key = q_key(p, y);
            }
        }
        if (rsplit) {
            // this warp's 16 rows are complete: normalise and write them
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = row0 + 8 * nt + 2 * tq + e;
                    const float m = __shfl_sync(0xffffffffu, m_run[nt], 8 * tq + 4 * e);
                    const float l = __shfl_sync(0xffffffffu, l_run[nt], 8 * tq + 4 * e);
                    const bool have = m != -INFINITY && l > 0.f;
                    const float inv = have ? 1.f / l : 0.f;
                    if (r < rows) {
                        const int64_t row = (int64_t)(r / GQ) * H + x.g * GQ + r % GQ;
                        float* orow = p.part_o + (part * HR + row) * D;
#pragma unroll
                        for (int mt = 0; mt < 8; ++mt) {
                            orow[16 * mt + gq] = oacc[nt][mt][e] * inv;
                            orow[16 * mt + 8 + gq] = oacc[nt][mt][2 + e] * inv;
                        }
                        if (gq == 0) p.part_lse[part * HR + row] = have ? (m + fast_log2(l)) * kLn2 : -INFINITY;
                    }
                }
            continue;
        }
        if (warp == 1) {
            if (X > 0) {
                const bool ok = mbar_wait_bounded(smem_addr(&xchg_bar[1]), (X - 1) & 1u, abort_flag, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, ok)) break;
            }
            if (tq == 0) {
                xm[gq] = m_run[0];
                xm[8 + gq] = m_run[1];
                xl[gq] = l_run[0];
                xl[8 + gq] = l_run[1];
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int mt = 0; mt < 8; ++mt)
                    xo[(nt * 8 + mt) * 32 + lane] =
                        make_float4(oacc[nt][mt][0], oacc[nt][mt][1], oacc[nt][mt][2], oacc[nt][mt][3]);
            __syncwarp();
            mbar_arrive(smem_addr(&xchg_bar[0]));
        } else {
            const bool ok = mbar_wait_bounded(smem_addr(&xchg_bar[0]), X & 1u, abort_flag, p.wait_limit_ns);
            if (!__all_sync(0xffffffffu, ok)) break;
            float f0[2][2], f1[2][2], inv[2][2], lse[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = 8 * nt + 2 * tq + e;
                    const float m0 = __shfl_sync(0xffffffffu, m_run[nt], 8 * tq + 4 * e);
                    const float l0 = __shfl_sync(0xffffffffu, l_run[nt], 8 * tq + 4 * e);
                    const float m1 = xm[r], l1 = xl[r];
                    const float M = fmaxf(m0, m1);
                    f0[nt][e] = (m0 == -INFINITY) ? 0.f : fast_exp2(m0 - M);
                    f1[nt][e] = (m1 == -INFINITY) ? 0.f : fast_exp2(m1 - M);
                    const float den = l0 * f0[nt][e] + l1 * f1[nt][e];
                    const bool have = M != -INFINITY && den > 0.f;
                    inv[nt][e] = have ? 1.f / den : 0.f;
                    lse[nt][e] = have ? (M + fast_log2(den)) * kLn2 : -INFINITY;
                }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    const float4 o1 = xo[(nt * 8 + mt) * 32 + lane];
                    oacc[nt][mt][0] = (oacc[nt][mt][0] * f0[nt][0] + o1.x * f1[nt][0]) * inv[nt][0];
                    oacc[nt][mt][1] = (oacc[nt][mt][1] * f0[nt][1] + o1.y * f1[nt][1]) * inv[nt][1];
                    oacc[nt][mt][2] = (oacc[nt][mt][2] * f0[nt][0] + o1.z * f1[nt][0]) * inv[nt][0];
                    oacc[nt][mt][3] = (oacc[nt][mt][3] * f0[nt][1] + o1.w * f1[nt][1]) * inv[nt][1];
                }
            __syncwarp();
            mbar_arrive(smem_addr(&xchg_bar[1]));
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = row0 + 8 * nt + 2 * tq + e;
                    if (r < rows) {
                        const int64_t row = (int64_t)(r / GQ) * H + x.g * GQ + r % GQ;
                        float* orow = p.part_o + (part * HR + row) * D;
#pragma unroll
                        for (int mt = 0; mt < 8; ++mt) {
                            orow[16 * mt + gq] = oacc[nt][mt][e];
                            orow[16 * mt + 8 + gq] = oacc[nt][mt][2 + e];
                        }
                        if (gq == 0) p.part_lse[part * HR + row] = lse[nt][e];
                    }
                }
        }
        ++X;
    }
}

// Multi-query consumers at head_dim 256 (up to 16 query rows per KV head; beyond that, row
// groups of 16 that are units of their own): warp w takes rows 8w .. 8w+7 of its unit's
// group (M = 16 of the q.K^T MMA with rows 8-15 zero, N = 8 of the P V MMA, as the
// single-query kernel) over both 16-cell halves of every tile, folding each row's causal
// limit into its lanes' cell mask, and writes its rows at the unit's end (no exchange).
template <int D>
__device__ __forceinline__ void mq_consumers_rows8(const SplitDecodeParams& p, uint64_t* full_bar, uint64_t* empty_bar,
                                                   const uint32_t* tile_mask, const uint32_t* tile_swz,
                                                   volatile int* abort_flag, unsigned char* stages, int n_stages,
                                                   int64_t n_units, int warp, int lane) {
    using G = Geom<KVATTN_KV_F16, D>;
    const int gq = lane >> 2;
    const int tq = lane & 3;
    const int H = p.n_head, GQ = p.group, NQ = p.n_q;
    const int rows = GQ * NQ;
    const int64_t HR = (int64_t)NQ * H;
    // first row of this warp in a unit: 16 rows per row group (more than 16 rows per KV head)
    auto first_row = [&](const Unit& y) { return p.rg_rows * y.rg + 8 * warp; };
    constexpr float kLn2 = 0.69314718055994530942f;
    auto load_q = [&](int s, int g, int row0, uint32_t (&qa)[D / 16][2]) {
        const int r = row0 + gq;
        const bool ok = r < rows;
        const int t = ok ? r / GQ : 0;
        const int h = g * GQ + (ok ? r % GQ : 0);
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + (((int64_t)s * NQ + t) * H + h) * D);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int d0 = 16 * kk + 2 * tq;
            qa[kk][0] = ok ? __ldg(qrow + d0 / 2) : 0u;
            qa[kk][1] = ok ? __ldg(qrow + (d0 + 8) / 2) : 0u;
        }
    };
    uint32_t qa[D / 16][2];
    int64_t qa_key = -1;  // q_key of the rows whose query fragments qa holds
    uint32_t T = 0;
    bool stop = false;
    for (int64_t u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
        const Unit x = unit_at(p, u);
        const int64_t part = (int64_t)x.s * p.part_stride + p.part_base + x.split_idx;
        const int row0 = first_row(x);
        if (x.n_tiles == 0) {
            if (x.write_empty) {
                for (int idx = lane; idx < 8 * D; idx += 32) {
                    const int r = row0 + idx / D;
                    const int d = idx % D;
                    if (r < rows) {
                        const int64_t row = (int64_t)(r / GQ) * H + x.g * GQ + r % GQ;
                        p.part_o[(part * HR + row) * D + d] = 0.f;
                        if (d == 0) p.part_lse[part * HR + row] = -INFINITY;
                    }
                }
            }
            continue;
        }
        if (qa_key != q_key(p, x)) {
            load_q(x.s, x.g, row0, qa);
            qa_key = q_key(p, x);
        }
        float oacc[D / 16][4];
        float m_run = -INFINITY, l_run = 0.f;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
        // causal limit (logical position, exclusive) of the lane's row row0 + gq
        const int64_t lim_row = x.len - NQ + 1 + (row0 + gq) / GQ;
        for (int t = 0; t < x.n_tiles; ++t, ++T) {
            const int st = (int)(T % (uint32_t)n_stages);
            const uint32_t use = T / (uint32_t)n_stages;
            const bool ok = mbar_wait_bounded(smem_addr(&full_bar[st]), use & 1u, abort_flag, p.wait_limit_ns);
            if (!__all_sync(0xffffffffu, ok)) {
                stop = true;
                break;
            }
            const bool swz = tile_swz[st] != 0u;
            unsigned char* stage = stages + st * G::kBytes;
#pragma unroll 1
            for (int hw = 0; hw < 2; ++hw) {
                const uint32_t mask = (tile_mask[st] >> (hw * kWarpCells)) & 0xffffu;
                if (mask == 0u) continue;
                const int64_t rel = lim_row - (x.i0 + (int64_t)t * kTileCells + hw * kWarpCells);
                const int lim = rel < 0 ? 0 : (rel > kWarpCells ? kWarpCells : (int)rel);
                const uint32_t lane_mask = mask & ((lim >= 32 ? 0xffffffffu : (1u << lim)) - 1u);
                if (swz) {
                    const uint32_t kb = smem_addr(stage);
                    if (mask != 0xffffu) {
                        // masked rows came in with the box: zero their V rows (both warps write
                        // the same zeros, each before its own reads)
                        const int r = hw * kWarpCells + (lane & 15);
                        if (lane < 16 && !((mask >> lane) & 1u)) {
#pragma unroll
                            for (int pl = 0; pl < G::kPlanes; ++pl) {
                                uint4* z = reinterpret_cast<uint4*>(stage + G::kSwzSection + pl * kPlaneBytes + r * 128);
#pragma unroll
                                for (int k = 0; k < 8; ++k) z[k] = make_uint4(0, 0, 0, 0);
                            }
                            fence_proxy_async();
                        }
                        __syncwarp();
                    }
                    consume_tile<KVATTN_KV_F16, D, true>(kb, kb + G::kSwzSection, nullptr, nullptr, lane_mask, hw,
                                                         lane, qa, oacc, m_run, l_run, p.scale_log2);
                } else {
                    const uint32_t kb = smem_addr(stage);
                    consume_tile<KVATTN_KV_F16, D, false>(kb, kb + G::kPadSection, nullptr, nullptr, lane_mask, hw,
                                                          lane, qa, oacc, m_run, l_run, p.scale_log2);
                }
            }
            __syncwarp();
            mbar_arrive(smem_addr(&empty_bar[st]));
        }
        if (stop) break;
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
        const int64_t un = u + gridDim.x;
        if (un < n_units) {
            const Unit y = unit_at(p, un);
            if (y.n_tiles > 0 && q_key(p, y) != qa_key) {
                load_q(y.s, y.g, first_row(y), qa);
                qa_key = q_key(p, y);
            }
        }
        // this lane's O rows are 8w + 2tq + e; their max / sum sit in lanes 8tq + 4e
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = row0 + 2 * tq + e;
            const float m = __shfl_sync(0xffffffffu, m_run, 8 * tq + 4 * e);
            const float l = __shfl_sync(0xffffffffu, l_run, 8 * tq + 4 * e);
            const bool have = m != -INFINITY && l > 0.f;
            const float inv = have ? 1.f / l : 0.f;
            if (r < rows) {
                const int64_t row = (int64_t)(r / GQ) * H + x.g * GQ + r % GQ;
                float* orow = p.part_o + (part * HR + row) * D;
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    orow[out_dim<KVATTN_KV_F16>(mt, 0, gq)] = oacc[mt][e] * inv;
                    orow[out_dim<KVATTN_KV_F16>(mt, 1, gq)] = oacc[mt][2 + e] * inv;
                }
                if (gq == 0) p.part_lse[part * HR + row] = have ? (m + fast_log2(l)) * kLn2 : -INFINITY;
            }
        }
    }
}

// Persistent split-decode kernel (f16 KV; Q8_0 runs in q8_self_body below).  Each CTA walks
// the units blockIdx.x, blockIdx.x + grid,
// ...; warp 2 streams the 32-cell tiles of those units through a ring of shared-memory
// stages without stopping between units, warps 0 and 1 attend to 16 cells of every tile.
// At the end of a unit warp 1 hands its running max, sum and unnormalised O to warp 0
// through an exchange area guarded by two mbarriers, and warp 0 writes the unit's partial
// (normalised O and LSE), so no CTA-wide barrier stalls the ring between units.
// MQ8: multi-query units of up to 8 query rows on the single-query consumers (row r = 8 rg +
// gq of the unit's KV head, token r / G, head g G + r % G; each lane's cells cut at its row's
// causal limit), for small verification batches.
// NCW: consumer warps (warp NCW produces).  Two, except the multi-query kernel for 33 to 48
// rows per KV head at head_dim 128, whose three consumer warps take 16 rows each.
template <int KVT, int D, bool MQ = false, bool MQ8 = false, int NCW = kConsumerWarps>
__device__ __forceinline__ void split_decode_body(const SplitDecodeParams& p) {
    static_assert(KVT == KVATTN_KV_F16, "Q8_0 runs in q8_self_body");
    static_assert(!MQ || D == 128 || D == 256, "multi-query decode: head_dim 128 or 256");
    using G = Geom<KVT, D>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment of the stage ring (the 128-B swizzle repeats every 8 rows)
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty_bar = full_bar + kMaxStages;
    uint64_t* xchg_bar = empty_bar + kMaxStages;  // [0] warp 1's result is posted, [1] area free
    uint32_t* tile_mask = reinterpret_cast<uint32_t*>(xchg_bar + 2);
    uint32_t* tile_swz = tile_mask + kMaxStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tile_swz + kMaxStages);
    float4* xo = reinterpret_cast<float4*>(smem + kHeaderBytes);  // [D/16][32 lanes] of warp 1's O
    float* xm = reinterpret_cast<float*>(xo + (D / 16) * 32);      // [8] warp 1's running max
    float* xl = xm + 8;                                             // [8] warp 1's running sum
    // (the head_dim-256 multi-query consumers split the rows and exchange nothing)
    unsigned char* stages = smem + kHeaderBytes + (MQ && D == 128 ? G::kXchgBytesMQ : G::kXchgBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_stages = p.n_stages;
    const int64_t n_units = (int64_t)p.n_seq * p.unit_splits * p.n_head_kv * (p.n_rg > 1 ? p.n_rg : 1);

    if (threadIdx.x == 0) {
        for (int i = 0; i < n_stages; ++i) {
            mbar_init(smem_addr(&full_bar[i]), p.src_lsu ? 64 : G::kArrivals);
            mbar_init(smem_addr(&empty_bar[i]), NCW * 32);
        }
        mbar_init(smem_addr(&xchg_bar[0]), 32);
        mbar_init(smem_addr(&xchg_bar[1]), 32);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    __syncthreads();
    // One wave (a unit per CTA): dependent launches (the merge, the next call) may be
    // scheduled at once -- they still wait for this grid to complete before reading
    // anything it writes -- and this CTA pulls its first tiles into L2 while the previous
    // kernel drains.  Grids of several units per CTA trigger only at exit: their
    // dependents, placed as slots free up, would otherwise crowd the CTAs that own an
    // extra unit onto the SMs that freed first (measured slower on GB300), and prefetched
    // tiles would wait long enough behind the tail to be evicted from L2.
    const bool one_wave = (int64_t)gridDim.x >= n_units;
    if (one_wave) pdl_launch_dependents();
    if (one_wave && warp == NCW && lane == 0 && p.use_tma && p.plan == nullptr && !p.src_lsu &&
        (int64_t)blockIdx.x < n_units) {
        // The lengths read here may still change before the dependency wait below; they
        // only steer these hints, never the loads (boxes outside the cache are not fetched).
        // Two tiles beyond the ring's depth: the previous call's merge leaves HBM idle for a
        // few microseconds (Qwen3-8B-shaped layer, 36-layer graph: 14.88 us per op with the
        // ring's depth of 3, 14.69 with 5, 14.62 with 6 but the kernel alone then slower,
        // 12.11 -> 12.6 us; 8 slower on both).
        const Unit x = unit_at(p, blockIdx.x);
        const int n_pre = x.n_tiles < n_stages + 2 ? x.n_tiles : n_stages + 2;
        for (int t = 0; t < n_pre; ++t) {
            const int64_t base = (int64_t)x.s * p.n_cells + x.i0 + (int64_t)t * kTileCells;
            if (base >= INT_MAX / 2) break;
#pragma unroll
            for (int pl = 0; pl < G::kPlanes; ++pl) {
                const int xx = pl * (KVT == KVATTN_KV_F16 ? 64 : 128);
                tma_prefetch_3d(&p.tmap_k, xx, x.g, (int)base);
                tma_prefetch_3d(&p.tmap_v, xx, x.g, (int)base);
            }
        }
    }
    if (!p.no_dep_wait) pdl_wait();

    const int gq = lane >> 2;
    const int tq = lane & 3;
    const int H = p.n_head;

    if (warp == NCW) {
        // ------------------------------- producer -------------------------------
        const int64_t Hk = p.n_head_kv;
        bool bad = false, stop = false;
        uint32_t T = 0;  // tiles issued by this CTA (ring position)
        for (int64_t u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
            const Unit x = unit_at(p, u);
            // The split's descriptor (the same for every KV head) is written by its head-0 unit
            // from the plan entries this warp reads anyway: count, smallest and largest valid
            // cell, the (cell - position) range, out-of-range entries seen.
            const bool emit_desc = p.desc_out != nullptr && x.g == 0 && x.rg == 0;
            if (x.n_tiles == 0) {
                if (emit_desc && lane == 0)
                    p.desc_out[(int64_t)x.s * p.n_split + x.split_idx] = make_int4(0, -1, -1, x.i0 >= x.len ? 9 : 1);
                continue;
            }
            int d_lo = INT_MAX, d_hi = -1, d_count = 0;
            long long d_off_lo = LLONG_MAX, d_off_hi = LLONG_MIN;
            bool d_bad = false;
            const int s = x.s, g = x.g, n_tiles = x.n_tiles;
            const int64_t i0 = x.i0, i1 = x.i1;
            // plan entries of this lane's cell, prefetched four tiles ahead
            const int32_t* prow = p.plan != nullptr ? p.plan + (int64_t)s * p.plan_stride : nullptr;
            auto plan_entry = [&](int tt) -> int32_t {
                const int64_t i = i0 + (int64_t)tt * kTileCells + lane;
                return (prow != nullptr && tt < n_tiles && i < i1) ? __ldg(prow + i) : -1;
            };
            int32_t e0 = plan_entry(0), e1 = plan_entry(1), e2 = plan_entry(2), e3 = plan_entry(3);
            for (int t = 0; t < n_tiles; ++t, ++T) {
                const int32_t e = e0;
                e0 = e1;
                e1 = e2;
                e2 = e3;
                e3 = plan_entry(t + 4);
                const int st = (int)(T % (uint32_t)n_stages);
                const uint32_t use = T / (uint32_t)n_stages;
                if (use > 0) {
                    const bool ok =
                        mbar_wait_bounded(smem_addr(&empty_bar[st]), (use - 1) & 1u, abort_flag, p.wait_limit_ns);
                    if (!__all_sync(0xffffffffu, ok)) {  // the whole warp agrees before any collective
                        stop = true;
                        break;
                    }
                }
                const int64_t tile0 = i0 + (int64_t)t * kTileCells;
                const int64_t i = tile0 + lane;
                bool valid = i < i1;
                int64_t cell = 0;
                if (valid) {
                    if (p.plan != nullptr) {
                        if (e < -1 || (int64_t)e >= p.n_cells) {
                            bad = true;
                            d_bad = true;
                            valid = false;
                        } else {
                            valid = e >= 0;
                            cell = e;
                        }
                    } else {
                        cell = (int64_t)s * p.n_cells + i;
                    }
                }
                const uint32_t mask = __ballot_sync(0xffffffffu, valid);
                // One physical run?  offset = cell - entry position must be the same for every
                // valid lane; the box then starts at the cell of the tile's first entry.
                int64_t base = (int64_t)s * p.n_cells + tile0;  // no plan: always one run
                bool run = true;
                if (p.plan != nullptr) {
                    long long off_lo = valid ? (long long)(cell - i) : LLONG_MAX;
                    long long off_hi = valid ? (long long)(cell - i) : LLONG_MIN;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        off_lo = min(off_lo, __shfl_xor_sync(0xffffffffu, off_lo, o));
                        off_hi = max(off_hi, __shfl_xor_sync(0xffffffffu, off_hi, o));
                    }
                    run = mask != 0u && off_lo == off_hi;
                    base = off_lo + tile0;
                    if (emit_desc) {
                        d_off_lo = min(d_off_lo, off_lo);
                        d_off_hi = max(d_off_hi, off_hi);
                        d_count += __popc(mask);
                        if (valid) {
                            d_lo = min(d_lo, (int)cell);
                            d_hi = max(d_hi, (int)cell);
                        }
                    }
                }
                const bool use_tma = run && p.use_tma != 0 && mask != 0u && base > INT_MIN / 2 &&
                                     base < INT_MAX / 2;
                unsigned char* stage = stages + st * G::kBytes;
                const uint32_t bar = smem_addr(&full_bar[st]);
                if (lane == 0) {
                    tile_mask[st] = mask;
                    tile_swz[st] = use_tma ? 1u : 0u;
                    const uint32_t bytes = use_tma     ? (uint32_t)(2 * G::kSwzSection)
                                           : p.src_lsu ? 0u  // cp.async completions arrive instead
                                                       : (uint32_t)__popc(mask) * 2u * (uint32_t)G::kRowBytes;
                    mbar_expect_tx(bar, bytes + (T == 0 ? p.stall_tx : 0u));
                }
                __syncwarp();
                if (use_tma) {
                    if (lane == 0) {
                        const uint32_t kdst = smem_addr(stage);
                        const uint32_t vdst = kdst + G::kSwzSection;
#pragma unroll
                        for (int pl = 0; pl < G::kPlanes; ++pl) {
                            const int xx = pl * (KVT == KVATTN_KV_F16 ? 64 : 128);  // elements of 128 B
                            const uint64_t pol = l2_evict_first_policy();
                            tma_load_3d_hint(kdst + pl * kPlaneBytes, &p.tmap_k, xx, g, (int)base, bar, pol);
                            tma_load_3d_hint(vdst + pl * kPlaneBytes, &p.tmap_v, xx, g, (int)base, bar, pol);
                        }
                    }
                }
                bool wrote = false;  // generic-proxy writes into the stage by this lane
                if (!use_tma) {
                    unsigned char* krow = stage + lane * G::kPadRow;
                    unsigned char* vrow = stage + G::kPadSection + lane * G::kPadRow;
                    if (p.src_lsu) {
                        // 16-byte asynchronous loads, a whole row per group of lanes, so every
                        // request covers full lines (the source may sit across the host link)
                        constexpr int kLanesPerRow = G::kRowBytes / 16 < 32 ? G::kRowBytes / 16 : 32;
                        constexpr int kRowsPerPass = 32 / kLanesPerRow;
                        constexpr int kChunksPerLane = G::kRowBytes / 16 / kLanesPerRow;
                        const int sub = lane % kLanesPerRow;
                        for (int r0 = 0; r0 < kTileCells; r0 += kRowsPerPass) {
                            const int c = r0 + lane / kLanesPerRow;
                            const bool cv = __shfl_sync(0xffffffffu, valid, c);
                            const int64_t ccell = __shfl_sync(0xffffffffu, cell, c);
                            if (cv) {
                                const int64_t row = ccell * Hk + g;
                                const char* ksrc = static_cast<const char*>(p.k) + row * G::kRowBytes;
                                const char* vsrc = static_cast<const char*>(p.v) + row * G::kRowBytes;
                                unsigned char* kd = stage + c * G::kPadRow;
                                unsigned char* vd = stage + G::kPadSection + c * G::kPadRow;
#pragma unroll
                                for (int j = 0; j < kChunksPerLane; ++j) {
                                    const int off = 16 * (sub + j * kLanesPerRow);
                                    cp_async_16_cg(smem_addr(kd + off), ksrc + off);
                                    cp_async_16_cg(smem_addr(vd + off), vsrc + off);
                                }
                            }
                        }
                    }
                    if (valid) {
                        if (!p.src_lsu) {
                            const int64_t row = cell * Hk + g;
                            bulk_g2s(smem_addr(krow), static_cast<const char*>(p.k) + row * G::kRowBytes,
                                     G::kRowBytes, bar);
                            bulk_g2s(smem_addr(vrow), static_cast<const char*>(p.v) + row * G::kRowBytes,
                                     G::kRowBytes, bar);
                        }
                    } else {
                        uint4* z = reinterpret_cast<uint4*>(vrow);
#pragma unroll
                        for (int k = 0; k < G::kRowBytes / 16; ++k) z[k] = make_uint4(0, 0, 0, 0);
                        wrote = true;
                    }
                }
                if (p.src_lsu) cp_async_arrive_noinc(bar);
                if (wrote) fence_proxy_async();  // zero-fills before later async writes to this stage
                mbar_arrive(bar);
            }
            if (emit_desc && !stop) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    d_lo = min(d_lo, __shfl_xor_sync(0xffffffffu, d_lo, o));
                    d_hi = max(d_hi, __shfl_xor_sync(0xffffffffu, d_hi, o));
                }
                const bool any_bad = __any_sync(0xffffffffu, d_bad);
                if (lane == 0) {
                    const int flags = (d_count == 0 ? 1 : (d_off_lo == d_off_hi ? 2 : 0)) | (any_bad ? 4 : 0);
                    p.desc_out[(int64_t)s * p.n_split + x.split_idx] =
                        make_int4(d_count, d_count ? d_lo : -1, d_count ? d_hi : -1, flags);
                }
            }
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, KVATTN_DEVICE_BAD_PLAN_ENTRY);
    } else {
        // ------------------------------- consumers -------------------------------
        if constexpr (MQ && D == 256) {
            mq_consumers_rows8<D>(p, full_bar, empty_bar, tile_mask, tile_swz, abort_flag, stages, n_stages, n_units,
                                  warp, lane);
        } else if constexpr (MQ) {
            mq_consumers(p, full_bar, empty_bar, tile_mask, tile_swz, abort_flag, xchg_bar,
                         reinterpret_cast<unsigned char*>(xo), stages, n_stages, n_units, warp, lane);
        } else {
        uint32_t qa[D / 16][2];
        int64_t qa_key = -1;  // q_key of the rows whose query fragments qa holds
        uint32_t T = 0;        // tiles consumed (ring position)
        uint32_t X = 0;        // end-of-unit exchanges done
        bool stop = false;
        constexpr float kLn2 = 0.69314718055994530942f;
        for (int64_t u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
            const Unit x = unit_at(p, u);
            const int64_t part = (int64_t)x.s * p.part_stride + p.part_base + x.split_idx;
            if (x.n_tiles == 0) {
                if (warp == 0 && x.write_empty) {
                    if constexpr (MQ8) {
                        const int64_t HR = (int64_t)p.n_q * H;
                        for (int idx = lane; idx < 8 * D; idx += 32) {
                            const int r = 8 * x.rg + idx / D;
                            const int d = idx % D;
                            if (r < p.group * p.n_q) {
                                const int64_t row = (int64_t)(r / p.group) * H + x.g * p.group + r % p.group;
                                p.part_o[(part * HR + row) * D + d] = 0.f;
                                if (d == 0) p.part_lse[part * HR + row] = -INFINITY;
                            }
                        }
                    } else {
                        for (int idx = lane; idx < p.group * D; idx += 32) {
                            const int r = idx / D;
                            const int d = idx - r * D;
                            const int h = x.g * p.group + r;
                            p.part_o[(part * H + h) * D + d] = 0.f;
                            if (d == 0) p.part_lse[part * H + h] = -INFINITY;
                        }
                    }
                }
                continue;
            }
            if (qa_key != q_key(p, x)) {
                load_q_frags<KVT, D>(p, x.s, x.g, gq, tq, qa, MQ8 ? x.rg : -1);
                qa_key = q_key(p, x);
            }
            // MQ8: causal limit (logical position, exclusive) of the lane's row 8 rg + gq
            const int64_t lim_row = MQ8 ? x.len - p.n_q + 1 + (8 * x.rg + gq) / p.group : 0;
            float oacc[D / 16][4];
            float m_run = -INFINITY, l_run = 0.f;
#pragma unroll
            for (int i = 0; i < D / 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

            for (int t = 0; t < x.n_tiles; ++t, ++T) {
                const int st = (int)(T % (uint32_t)n_stages);
                const uint32_t use = T / (uint32_t)n_stages;
                const bool ok =
                    mbar_wait_bounded(smem_addr(&full_bar[st]), use & 1u, abort_flag, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    stop = true;
                    break;
                }
                const uint32_t mask = (tile_mask[st] >> (warp * kWarpCells)) & 0xffffu;
                const bool swz = tile_swz[st] != 0u;
                unsigned char* stage = stages + st * G::kBytes;
                const uint32_t ebar = smem_addr(&empty_bar[st]);
                bool released = false;
                uint32_t lmask = mask;  // this lane's cells
                if constexpr (MQ8) {
                    const int64_t rel = lim_row - (x.i0 + (int64_t)t * kTileCells + warp * kWarpCells);
                    const int lim = rel < 0 ? 0 : (rel > kWarpCells ? kWarpCells : (int)rel);
                    lmask &= (lim >= 32 ? 0xffffffffu : (1u << lim)) - 1u;
                }
                if (mask != 0u) {
                    if (swz) {
                        const uint32_t kb = smem_addr(stage);
                        const uint32_t vb = kb + G::kSwzSection;
                        if (mask != 0xffffu) {
                            // masked rows came in with the box: zero their V rows (every plane)
                            const int r = warp * kWarpCells + (lane & 15);
                            if (lane < 16 && !((mask >> lane) & 1u)) {
#pragma unroll
                                for (int pl = 0; pl < G::kPlanes; ++pl) {
                                    uint4* z = reinterpret_cast<uint4*>(stage + G::kSwzSection + pl * kPlaneBytes +
                                                                        r * 128);
#pragma unroll
                                    for (int k = 0; k < 8; ++k) z[k] = make_uint4(0, 0, 0, 0);
                                }
                                fence_proxy_async();
                            }
                            __syncwarp();
                        }
                        if constexpr (D == 128) {
                            consume_tile_staged<true>(kb, vb, lmask, warp, lane, ebar, qa, oacc, m_run, l_run,
                                                      p.scale_log2);
                            released = true;
                        } else {
                            consume_tile<KVT, D, true>(kb, vb, nullptr, nullptr, lmask, warp, lane, qa, oacc, m_run,
                                                       l_run, p.scale_log2);
                        }
                    } else {
                        const uint32_t kb = smem_addr(stage);
                        const uint32_t vb = kb + G::kPadSection;
                        if constexpr (D == 128) {
                            consume_tile_staged<false>(kb, vb, lmask, warp, lane, ebar, qa, oacc, m_run, l_run,
                                                       p.scale_log2);
                            released = true;
                        } else {
                            consume_tile<KVT, D, false>(kb, vb, nullptr, nullptr, lmask, warp, lane, qa, oacc, m_run,
                                                        l_run, p.scale_log2);
                        }
                    }
                }
                if (!released) {
                    __syncwarp();
                    mbar_arrive(ebar);
                }
            }
            if (stop) break;
            l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
            l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
            // the next unit's query fragments load while this unit is combined and written
            const int64_t un = u + gridDim.x;
            if (un < n_units) {
                const Unit y = unit_at(p, un);
                if (y.n_tiles > 0 && q_key(p, y) != qa_key) {
                    load_q_frags<KVT, D>(p, y.s, y.g, gq, tq, qa, MQ8 ? y.rg : -1);
                    qa_key = q_key(p, y);
                }
            }

            // ---------------- combine the two consumer warps, write the partial ----------------
            if (warp == 1) {
                if (X > 0) {
                    const bool ok = mbar_wait_bounded(smem_addr(&xchg_bar[1]), (X - 1) & 1u, abort_flag,
                                                      p.wait_limit_ns);
                    if (!__all_sync(0xffffffffu, ok)) break;
                }
                if (tq == 0) {
                    xm[gq] = m_run;
                    xl[gq] = l_run;
                }
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt)
                    xo[mt * 32 + lane] = make_float4(oacc[mt][0], oacc[mt][1], oacc[mt][2], oacc[mt][3]);
                __syncwarp();
                mbar_arrive(smem_addr(&xchg_bar[0]));
            } else {
                const bool ok =
                    mbar_wait_bounded(smem_addr(&xchg_bar[0]), X & 1u, abort_flag, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, ok)) break;
                // this lane's O rows are 2tq and 2tq+1; their max / sum sit in lanes 8tq, 8tq+4
                float f0[2], f1[2], inv[2], lse[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float m0 = __shfl_sync(0xffffffffu, m_run, 8 * tq + 4 * e);
                    const float l0 = __shfl_sync(0xffffffffu, l_run, 8 * tq + 4 * e);
                    const float m1 = xm[2 * tq + e];
                    const float l1 = xl[2 * tq + e];
                    const float M = fmaxf(m0, m1);
                    f0[e] = (m0 == -INFINITY) ? 0.f : fast_exp2(m0 - M);
                    f1[e] = (m1 == -INFINITY) ? 0.f : fast_exp2(m1 - M);
                    const float den = l0 * f0[e] + l1 * f1[e];
                    const bool have = M != -INFINITY && den > 0.f;
                    inv[e] = have ? 1.f / den : 0.f;
                    lse[e] = have ? (M + fast_log2(den)) * kLn2 : -INFINITY;
                }
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    const float4 o1 = xo[mt * 32 + lane];
                    oacc[mt][0] = (oacc[mt][0] * f0[0] + o1.x * f1[0]) * inv[0];
                    oacc[mt][1] = (oacc[mt][1] * f0[1] + o1.y * f1[1]) * inv[1];
                    oacc[mt][2] = (oacc[mt][2] * f0[0] + o1.z * f1[0]) * inv[0];
                    oacc[mt][3] = (oacc[mt][3] * f0[1] + o1.w * f1[1]) * inv[1];
                }
                __syncwarp();
                mbar_arrive(smem_addr(&xchg_bar[1]));
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    bool ok;
                    int64_t prow;  // partial row index (part, row)
                    if constexpr (MQ8) {
                        const int r = 8 * x.rg + 2 * tq + e;
                        ok = r < p.group * p.n_q;
                        prow = part * ((int64_t)p.n_q * H) + (int64_t)(r / p.group) * H + x.g * p.group +
                               r % p.group;
                    } else {
                        const int r = 2 * tq + e;
                        ok = r < p.group;
                        prow = part * H + x.g * p.group + r;
                    }
                    if (ok) {
                        float* orow = p.part_o + prow * D;
#pragma unroll
                        for (int mt = 0; mt < D / 16; ++mt) {
                            orow[out_dim<KVT>(mt, 0, gq)] = oacc[mt][e];
                            orow[out_dim<KVT>(mt, 1, gq)] = oacc[mt][2 + e];
                        }
                        if (gq == 0) p.part_lse[prow] = lse[e];
                    }
                }
            }
            ++X;
        }
        }  // single-query consumers
    }

    // Every wait above is bounded, so all warps get here; a timed-out wait left abort set.
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag != 0) atomicOr(p.status, KVATTN_DEVICE_WAIT_TIMEOUT);
    if (!one_wave) pdl_launch_dependents();
}

constexpr int kChunkCells = 16;  // cells per chunk of the Q8_0 self-loading warps

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

// One warp's 16-cell Q8_0 chunk in the 128-byte-swizzled layout of 16-row planes: scores,
// online softmax, P V.  In a 1024-byte-aligned plane the byte (row r, column b) sits at
// r*128 + 16*((b >> 4) ^ (r & 7)) + (b & 15); every address below is a per-lane base whose
// bits 4-6 already hold the row's swizzle key, XOR-ed with 16*(b >> 4) and offset by
// immediates, so the swizzle costs one logic op per 16-byte column instead of an index
// computation per load.  The scales of a cell (D/32 halves) are read once per chunk.
template <int D>
__device__ __forceinline__ void q8_chunk_swz(uint32_t kb, uint32_t vb, const unsigned char* ks,
                                             const unsigned char* vs, uint32_t mask, int lane,
                                             const uint32_t (&qa)[D / 16][2], float (&oacc)[D / 16][4],
                                             float& m_run, float& l_run, float scale_log2) {
    constexpr int kPlane = kChunkCells * 128;
    constexpr int kScl = 16;  // bytes between two cells' scale rows in the stage
    const int gq = lane >> 2;
    const int tq = lane & 3;
    // K rows gq (n-tile 0) and 8 + gq (+1024); this lane's bytes 4tq.. of each 16-byte column
    const uint32_t ka = (kb + 128u * gq + 4u * tq) | (16u * gq);
    // V rows 2tq and 2tq + 1 (and +8, +9 at +1024); bytes 4(gq & 3).. of column 2blk + (gq >> 2)
    const uint32_t va0 = (vb + 256u * tq + 4u * (gq & 3)) | (16u * ((gq >> 2) ^ (2 * tq)));
    const uint32_t va1 = (vb + 256u * tq + 128u + 4u * (gq & 3)) | (16u * ((gq >> 2) ^ (2 * tq + 1)));
    const uint32_t kss = smem_addr(ks) + 2u * kScl * tq;  // cell 2tq's scales; cell c at + (c - 2tq) * kScl
    const uint32_t vss = smem_addr(vs) + 2u * kScl * tq;

    float sacc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
    // K scales of cells 8j + 2tq + e: D/32 halves each
    uint32_t ksw[2][2][D / 64];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int h = 0; h < D / 128; ++h) {
                const uint2 w = lds64(kss + (8 * j + e) * kScl + 8 * h);
                ksw[j][e][2 * h] = w.x;
                ksw[j][e][2 * h + 1] = w.y;
            }
#pragma unroll
    for (int b = 0; b < D / 32; ++b) {
        const uint32_t pl = kPlane * (b >> 2);
        const uint32_t a0 = (ka ^ (32u * (b & 3))) + pl;      // column 2(b & 3): half 0 of block b
        const uint32_t a1 = (ka ^ (32u * (b & 3) + 16u)) + pl;  // column 2(b & 3) + 1: half 1
        uint32_t kw[2][2];
        float ksc[2][2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            kw[j][0] = lds32(a0 + 1024u * j);
            kw[j][1] = lds32(a1 + 1024u * j);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const uint32_t w = ksw[j][e][b >> 1];
                ksc[j][e] = __half2float(__ushort_as_half((unsigned short)((b & 1) ? (w >> 16) : (w & 0xffffu))));
            }
        }
        q8_qk_block(sacc, qa[2 * b], qa[2 * b + 1], kw, ksc);
    }

    float alpha, pf[2][2];
    if (softmax_step(sacc, mask, tq, scale_log2, m_run, alpha, pf)) {
        rescale_o<D>(oacc, alpha, tq);
        l_run *= alpha;
    }
    l_run += (pf[0][0] + pf[0][1]) + (pf[1][0] + pf[1][1]);
    const uint32_t ph0 = pack_half2(pf[0][0], pf[0][1]);
    const uint32_t ph1 = pack_half2(pf[1][0], pf[1][1]);
    // V scales of cells 2tq, 2tq + 1, 2tq + 8, 2tq + 9
    uint32_t vsw[4][D / 64];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int h = 0; h < D / 128; ++h) {
            const uint2 w = lds64(vss + ((c & 1) + 8 * (c >> 1)) * kScl + 8 * h);
            vsw[c][2 * h] = w.x;
            vsw[c][2 * h + 1] = w.y;
        }
#pragma unroll
    for (int b = 0; b < D / 32; ++b) {
        const uint32_t pl = kPlane * (b >> 2);
        const uint32_t c0 = (va0 ^ (32u * (b & 3))) + pl;
        const uint32_t c1 = (va1 ^ (32u * (b & 3))) + pl;
        const uint32_t vw[4] = {lds32(c0), lds32(c1), lds32(c0 + 1024u), lds32(c1 + 1024u)};
        const uint32_t sel = (b & 1) ? 0x7632u : 0x5410u;
        const uint32_t s01 = prmt_b32(vsw[0][b >> 1], vsw[1][b >> 1], sel);
        const uint32_t s89 = prmt_b32(vsw[2][b >> 1], vsw[3][b >> 1], sel);
        q8_pv_block(oacc[2 * b], oacc[2 * b + 1], vw, hmul2_u32(ph0, s01), hmul2_u32(ph1, s89));
    }
}

__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// Q4_0 values -> exact f16 pairs.  w holds, for two cells, one byte each in bits 0-7 and
// 16-23 (a byte: element e in its low nibble, element e + 16 in its high nibble).  With the
// f16 bit pattern 0x6400 (1024) OR-ed in, a low nibble n reads as 1024 + n and a high
// nibble as 1024 + 16 n; subtracting 1032, or scaling by 1/16 and subtracting 72, leaves
// n - 8 exactly (the same magic-number idea as the int8 conversion).
__device__ __forceinline__ uint32_t q4x2_lo(uint32_t w) {
    uint32_t t, r;
    asm("lop3.b32 %0, %1, 0x000f000f, 0x64006400, 0xea;" : "=r"(t) : "r"(w));  // (w & m) | c
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(0x64086408u));
    return r;
}
__device__ __forceinline__ uint32_t q4x2_hi(uint32_t w) {
    uint32_t t, r;
    asm("lop3.b32 %0, %1, 0x00f000f0, 0x64006400, 0xea;" : "=r"(t) : "r"(w));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(t), "r"(0x2c002c00u), "r"(0xd480d480u));  // x/16 - 72
    return r;
}

// Q4_0 q.K of one 32-element block b for the two 8-cell n-tiles.  kw[j] is the 32-bit word at
// bytes 4tq .. 4tq+3 of the block for cell 8j + gq: low nibbles = elements 4tq .. 4tq+3, high
// nibbles = elements 16 + 4tq .. 16 + 4tq+3.  The mask-and-convert step pairs bytes 0 and 2
// (and 1 and 3, after a shift), so the MMA k pairs (2tq, 2tq+1) and (2tq+8, 2tq+9) are the
// element pairs (4tq, 4tq+2) and (4tq+1, 4tq+3) -- the query fragments are loaded in that
// order (load_q_frags_q4k).
__device__ __forceinline__ void q4_qk_block(float (&sacc)[2][4], const uint32_t (&qa0)[2], const uint32_t (&qa1)[2],
                                            const uint32_t (&kw)[2], const float (&ksc)[2][2]) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        float cb[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t w = kw[j], x = kw[j] >> 8;
        mma_16816(cb, qa0[0], 0u, qa0[1], 0u, q4x2_lo(w), q4x2_lo(x));
        mma_16816(cb, qa1[0], 0u, qa1[1], 0u, q4x2_hi(w), q4x2_hi(x));
        sacc[j][0] = fmaf(cb[0], ksc[j][0], sacc[j][0]);
        sacc[j][1] = fmaf(cb[1], ksc[j][1], sacc[j][1]);
    }
}

// One warp's 16-cell chunk of Q8_0 or Q4_0 keys (KQ4) and Q4_0 values: scores, online
// softmax, P V.  SWZ: the chunk came by TMA boxes (8-bit K in 128-byte-wide planes under the
// 128-byte swizzle as for Q8_0; 4-bit K and V each in one box of D/2-byte rows under the
// swizzle of that width); otherwise by one copy per row into plain rows.
// V operand (O^T += V^T P'^T, head_dim in M): a lane reads the 16-bit word at bytes
// 2gq, 2gq+1 of block b for cells 2tq, 2tq+1, 2tq+8, 2tq+9 -- elements 2gq, 2gq+1 in the low
// nibbles and 2gq+16, 2gq+17 in the high ones -- so m-tile 2b holds dims 32b + 2gq (row gq)
// and 32b + 2gq + 1 (row gq + 8), and m-tile 2b+1 the same plus 16.  Every dim of an m-tile
// lies in block b, whose V scale multiplies P as in the Q8_0 path.
template <int D, bool SWZ, bool KQ4>
__device__ __forceinline__ void q4v_chunk(uint32_t kb, uint32_t vb, const unsigned char* ks,
                                           const unsigned char* vs, uint32_t mask, int lane,
                                           const uint32_t (&qa)[D / 16][2], float (&oacc)[D / 16][4],
                                           float& m_run, float& l_run, float scale_log2) {
    constexpr int kPlane = kChunkCells * 128;
    constexpr int kScl = 16;      // bytes between two cells' scale rows in the stage
    constexpr int kVRow = D / 2;  // bytes of a 4-bit V row
    const int gq = lane >> 2;
    const int tq = lane & 3;
    // K rows gq and 8 + gq.  8-bit: swizzled planes (see q8_chunk_swz) or plain D-byte rows.
    // 4-bit: the word at bytes 16b + 4tq of the row; under the swizzle its 16-byte column is
    // b ^ (gq >> 1 & 3) (64-byte rows) or b ^ gq (128-byte rows), the same for row gq + 8.
    uint32_t ka;
    if (KQ4) {
        if (SWZ)
            ka = D == 128 ? ((kb + 64u * gq + 4u * tq) | (16u * ((gq >> 1) & 3))) : ((kb + 128u * gq + 4u * tq) | (16u * gq));
        else
            ka = kb + (uint32_t)kVRow * gq + 4u * tq;
    } else {
        ka = SWZ ? ((kb + 128u * gq + 4u * tq) | (16u * gq)) : (kb + (uint32_t)D * gq + 4u * tq);
    }
    // V: base addresses whose XOR with 16b (plus immediates) give cells 2tq, 2tq+1, 2tq+8, 2tq+9
    // of block b.  head_dim 256 (128-byte rows, 128-byte swizzle): the 16-byte column of
    // (row c, byte x) is (x >> 4) ^ (c & 7).  head_dim 128 (64-byte rows, 64-byte swizzle):
    // the column of byte offset a = 64c + x is (a >> 4 & 3) ^ (a >> 7 & 3) = (x >> 4) ^ (c >> 1 & 3).
    uint32_t va0, va1;
    if (SWZ) {
        if (D == 128) {  // cells 2tq, 2tq+1 (and 2tq+8, 2tq+9) share the key tq
            va0 = (vb + 128u * tq + 2u * gq) | (16u * tq);
            va1 = va0 + 64u;
        } else {  // 128-byte rows: line c, key c & 7
            va0 = (vb + 256u * tq + 2u * gq) | (32u * tq);
            va1 = (vb + 256u * tq + 128u + 2u * gq) | (16u * (2 * tq + 1));
        }
    } else {
        va0 = vb + (uint32_t)kVRow * (2 * tq) + 2u * gq;
        va1 = va0 + kVRow;
    }
    const uint32_t kss = smem_addr(ks) + 2u * kScl * tq;
    const uint32_t vss = smem_addr(vs) + 2u * kScl * tq;

    float sacc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
    uint32_t ksw[2][2][D / 64];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int h = 0; h < D / 128; ++h) {
                const uint2 w = lds64(kss + (8 * j + e) * kScl + 8 * h);
                ksw[j][e][2 * h] = w.x;
                ksw[j][e][2 * h + 1] = w.y;
            }
#pragma unroll
    for (int b = 0; b < D / 32; ++b) {
        float ksc[2][2];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const uint32_t w = ksw[j][e][b >> 1];
                ksc[j][e] = __half2float(__ushort_as_half((unsigned short)((b & 1) ? (w >> 16) : (w & 0xffffu))));
            }
        if constexpr (KQ4) {
            const uint32_t a = SWZ ? (ka ^ (16u * b)) : (ka + 16u * b);
            const uint32_t rs = SWZ ? (D == 128 ? 512u : 1024u) : 8u * kVRow;  // rows 8..15
            const uint32_t kw[2] = {lds32(a), lds32(a + rs)};
            q4_qk_block(sacc, qa[2 * b], qa[2 * b + 1], kw, ksc);
        } else {
            uint32_t a0, a1, rs;
            if (SWZ) {
                const uint32_t pl = kPlane * (b >> 2);
                a0 = (ka ^ (32u * (b & 3))) + pl;
                a1 = (ka ^ (32u * (b & 3) + 16u)) + pl;
                rs = 1024u;  // rows 8..15 of the plane
            } else {
                a0 = ka + 32u * b;
                a1 = a0 + 16u;
                rs = 8u * D;
            }
            uint32_t kw[2][2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                kw[j][0] = lds32(a0 + rs * j);
                kw[j][1] = lds32(a1 + rs * j);
            }
            q8_qk_block(sacc, qa[2 * b], qa[2 * b + 1], kw, ksc);
        }
    }

    float alpha, pf[2][2];
    if (softmax_step(sacc, mask, tq, scale_log2, m_run, alpha, pf)) {
        rescale_o<D>(oacc, alpha, tq);
        l_run *= alpha;
    }
    l_run += (pf[0][0] + pf[0][1]) + (pf[1][0] + pf[1][1]);
    const uint32_t ph0 = pack_half2(pf[0][0], pf[0][1]);
    const uint32_t ph1 = pack_half2(pf[1][0], pf[1][1]);
    uint32_t vsw[4][D / 64];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int h = 0; h < D / 128; ++h) {
            const uint2 w = lds64(vss + ((c & 1) + 8 * (c >> 1)) * kScl + 8 * h);
            vsw[c][2 * h] = w.x;
            vsw[c][2 * h + 1] = w.y;
        }
#pragma unroll
    for (int b = 0; b < D / 32; ++b) {
        uint32_t c0, c1, c8, c9;  // 16-bit words of cells 2tq, 2tq+1, 2tq+8, 2tq+9
        if (SWZ) {
            if (D == 128) {
                const uint32_t x = va0 ^ (16u * b);
                c0 = lds16(x);
                c1 = lds16(x + 64u);
                c8 = lds16(x + 512u);
                c9 = lds16(x + 576u);
            } else {
                const uint32_t x0 = va0 ^ (16u * b), x1 = va1 ^ (16u * b);
                c0 = lds16(x0);
                c1 = lds16(x1);
                c8 = lds16(x0 + 1024u);
                c9 = lds16(x1 + 1024u);
            }
        } else {
            const uint32_t x = va0 + 16u * b;
            c0 = lds16(x);
            c1 = lds16(x + kVRow);
            c8 = lds16(x + 8u * kVRow);
            c9 = lds16(x + 9u * kVRow);
        }
        // byte 0 of both cells of a pair in bits 0-7 / 16-23 (w), byte 1 likewise (x)
        const uint32_t w01 = prmt_b32(c0, c1, 0x5410u), x01 = prmt_b32(c0, c1, 0x5511u);
        const uint32_t w89 = prmt_b32(c8, c9, 0x5410u), x89 = prmt_b32(c8, c9, 0x5511u);
        const uint32_t sel = (b & 1) ? 0x7632u : 0x5410u;
        const uint32_t pb0 = hmul2_u32(ph0, prmt_b32(vsw[0][b >> 1], vsw[1][b >> 1], sel));
        const uint32_t pb1 = hmul2_u32(ph1, prmt_b32(vsw[2][b >> 1], vsw[3][b >> 1], sel));
        mma_16816(oacc[2 * b], q4x2_lo(w01), q4x2_lo(x01), q4x2_lo(w89), q4x2_lo(x89), pb0, pb1);
        mma_16816(oacc[2 * b + 1], q4x2_hi(w01), q4x2_hi(x01), q4x2_hi(w89), q4x2_hi(x89), pb0, pb1);
    }
}

// Query fragments of the multi-query quantised kernels: rows gq (qa[kk][0..1]) and gq + 8
// (qa[kk][2..3]) of the KV head's G x n_q rows, in the element order of load_q_frags (8-bit
// keys) or load_q_frags_q4k (4-bit keys).
template <int D, bool KQ4>
__device__ __forceinline__ void load_q_frags_mq_q8(const SplitDecodeParams& p, int s, int g, int gq, int tq,
                                                   int row0, uint32_t (&qa)[D / 16][4]) {
    const int rows = p.group * p.n_q;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = row0 + gq + 8 * half;
        const bool ok = r < rows;
        const int t = ok ? r / p.group : 0;
        const int h = g * p.group + (ok ? r % p.group : 0);
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + (((int64_t)s * p.n_q + t) * p.n_head + h) * D);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int d0 = 32 * (kk >> 1) + 16 * (kk & 1) + 4 * tq;
            const uint32_t w0 = ok ? __ldg(qrow + d0 / 2) : 0u;      // elements d0, d0+1
            const uint32_t w1 = ok ? __ldg(qrow + d0 / 2 + 1) : 0u;  // elements d0+2, d0+3
            qa[kk][2 * half] = KQ4 ? prmt_b32(w0, w1, 0x5410u) : w0;
            qa[kk][2 * half + 1] = KQ4 ? prmt_b32(w0, w1, 0x7632u) : w1;
        }
    }
}

// One warp's 16-cell quantised chunk for up to 16 query rows (multi-query decode): q.K with
// the whole M = 16 of the MMA, an online softmax per row (row gq + 8 hh, causal limit lim[hh]
// cells of the chunk), and P V into two N = 8 tiles that share every converted V fragment.
// Keys 8-bit or 4-bit (KQ4), values 8-bit or 4-bit (VQ4), in the layouts of q8_chunk_swz and
// q4v_chunk: SWZ the TMA boxes' swizzled layout, else plain rows.
template <int D, bool SWZ, bool VQ4 = false, bool KQ4 = false>
__device__ __forceinline__ void q8_mq_chunk(uint32_t kb, uint32_t vb, const unsigned char* ks,
                                            const unsigned char* vs, uint32_t mask, int lane, const int (&lim)[2],
                                            const uint32_t (&qa)[D / 16][4], float (&oacc)[2][D / 16][4],
                                            float (&m_run)[2], float (&l_run)[2], float scale_log2) {
    constexpr int kPlane = kChunkCells * 128;
    constexpr int kScl = 16;         // bytes between two cells' scale rows in the stage
    constexpr int kHalfRow = D / 2;  // bytes of a 4-bit row
    const int gq = lane >> 2;
    const int tq = lane & 3;
    uint32_t ka;
    if (KQ4)
        ka = SWZ ? ((kb + 64u * gq + 4u * tq) | (16u * ((gq >> 1) & 3))) : (kb + (uint32_t)kHalfRow * gq + 4u * tq);
    else
        ka = SWZ ? ((kb + 128u * gq + 4u * tq) | (16u * gq)) : (kb + (uint32_t)D * gq + 4u * tq);
    uint32_t va0, va1;
    if (VQ4) {
        va0 = SWZ ? ((vb + 128u * tq + 2u * gq) | (16u * tq)) : (vb + (uint32_t)kHalfRow * (2 * tq) + 2u * gq);
        va1 = 0u;
    } else if (SWZ) {
        va0 = (vb + 256u * tq + 4u * (gq & 3)) | (16u * ((gq >> 2) ^ (2 * tq)));
        va1 = (vb + 256u * tq + 128u + 4u * (gq & 3)) | (16u * ((gq >> 2) ^ (2 * tq + 1)));
    } else {
        va0 = vb + (uint32_t)D * (2 * tq) + 4u * gq;
        va1 = va0 + D;
    }
    const uint32_t kss = smem_addr(ks) + 2u * kScl * tq;
    const uint32_t vss = smem_addr(vs) + 2u * kScl * tq;

    float sacc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
    uint32_t ksw[2][2][D / 64];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int h = 0; h < D / 128; ++h) {
                const uint2 w = lds64(kss + (8 * j + e) * kScl + 8 * h);
                ksw[j][e][2 * h] = w.x;
                ksw[j][e][2 * h + 1] = w.y;
            }
#pragma unroll
    for (int b = 0; b < D / 32; ++b) {
        uint32_t a0, a1, rs;
        if (KQ4) {
            a0 = SWZ ? (ka ^ (16u * b)) : (ka + 16u * b);
            a1 = 0u;
            rs = SWZ ? 512u : 8u * kHalfRow;
        } else if (SWZ) {
            const uint32_t pl = kPlane * (b >> 2);
            a0 = (ka ^ (32u * (b & 3))) + pl;
            a1 = (ka ^ (32u * (b & 3) + 16u)) + pl;
            rs = 1024u;
        } else {
            a0 = ka + 32u * b;
            a1 = a0 + 16u;
            rs = 8u * D;
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            uint32_t b00, b01, b10, b11;  // B operands of the block's two MMAs
            if (KQ4) {
                const uint32_t w = lds32(a0 + rs * j), x = w >> 8;
                b00 = q4x2_lo(w);
                b01 = q4x2_lo(x);
                b10 = q4x2_hi(w);
                b11 = q4x2_hi(x);
            } else {
                const uint32_t w0 = lds32(a0 + rs * j) ^ 0x80808080u, w1 = lds32(a1 + rs * j) ^ 0x80808080u;
                b00 = i8x2_lo(w0);
                b01 = i8x2_hi(w0);
                b10 = i8x2_lo(w1);
                b11 = i8x2_hi(w1);
            }
            float cb[4] = {0.f, 0.f, 0.f, 0.f};
            mma_16816(cb, qa[2 * b][0], qa[2 * b][2], qa[2 * b][1], qa[2 * b][3], b00, b01);
            mma_16816(cb, qa[2 * b + 1][0], qa[2 * b + 1][2], qa[2 * b + 1][1], qa[2 * b + 1][3], b10, b11);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const uint32_t w = ksw[j][e][b >> 1];
                const float sc = __half2float(__ushort_as_half((unsigned short)((b & 1) ? (w >> 16) : (w & 0xffffu))));
                sacc[j][e] = fmaf(cb[e], sc, sacc[j][e]);          // row gq
                sacc[j][2 + e] = fmaf(cb[2 + e], sc, sacc[j][2 + e]);  // row gq + 8
            }
        }
    }

    // online softmax, one (max, sum) per row: hh = 0 -> row gq, hh = 1 -> row gq + 8
    float x[2][2][2];
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int c = 8 * j + 2 * tq + e;
                const bool ok = ((mask >> c) & 1u) && c < lim[hh];
                x[hh][j][e] = ok ? sacc[j][2 * hh + e] * scale_log2 : -INFINITY;
                tmax[hh] = fmaxf(tmax[hh], x[hh][j][e]);
            }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        tmax[hh] = fmaxf(tmax[hh], __shfl_xor_sync(0xffffffffu, tmax[hh], 1));
        tmax[hh] = fmaxf(tmax[hh], __shfl_xor_sync(0xffffffffu, tmax[hh], 2));
    }
    if (__any_sync(0xffffffffu, tmax[0] > m_run[0] + kRescaleSlack || tmax[1] > m_run[1] + kRescaleSlack)) {
        float alpha[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const float m_new = fmaxf(m_run[hh], tmax[hh]);
            alpha[hh] = fast_exp2(m_run[hh] - ((m_new == -INFINITY) ? 0.f : m_new));
            m_run[hh] = m_new;
            l_run[hh] *= alpha[hh];
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const float a0 = __shfl_sync(0xffffffffu, alpha[nt], 8 * tq);
            const float a1 = __shfl_sync(0xffffffffu, alpha[nt], 8 * tq + 4);
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                oacc[nt][mt][0] *= a0;
                oacc[nt][mt][1] *= a1;
                oacc[nt][mt][2] *= a0;
                oacc[nt][mt][3] *= a1;
            }
        }
    }
    uint32_t ph[2][2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const float m_use = (m_run[hh] == -INFINITY) ? 0.f : m_run[hh];
        float psum = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float p0 = fast_exp2(x[hh][j][0] - m_use), p1 = fast_exp2(x[hh][j][1] - m_use);
            ph[hh][j] = pack_half2(p0, p1);
            psum += p0 + p1;
        }
        l_run[hh] += psum;
    }
    // V scales of cells 2tq, 2tq + 1, 2tq + 8, 2tq + 9
    uint32_t vsw[4][D / 64];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int h = 0; h < D / 128; ++h) {
            const uint2 w = lds64(vss + ((c & 1) + 8 * (c >> 1)) * kScl + 8 * h);
            vsw[c][2 * h] = w.x;
            vsw[c][2 * h + 1] = w.y;
        }
#pragma unroll
    for (int b = 0; b < D / 32; ++b) {
        uint32_t A0[4], A1[4];  // V^T operands of m-tiles 2b and 2b + 1
        if (VQ4) {
            // 16-bit words of cells 2tq, 2tq+1, 2tq+8, 2tq+9 (layout as in q4v_chunk)
            uint32_t c0, c1, c8, c9;
            if (SWZ) {
                const uint32_t x = va0 ^ (16u * b);
                c0 = lds16(x);
                c1 = lds16(x + 64u);
                c8 = lds16(x + 512u);
                c9 = lds16(x + 576u);
            } else {
                const uint32_t x = va0 + 16u * b;
                c0 = lds16(x);
                c1 = lds16(x + kHalfRow);
                c8 = lds16(x + 8u * kHalfRow);
                c9 = lds16(x + 9u * kHalfRow);
            }
            const uint32_t w01 = prmt_b32(c0, c1, 0x5410u), x01 = prmt_b32(c0, c1, 0x5511u);
            const uint32_t w89 = prmt_b32(c8, c9, 0x5410u), x89 = prmt_b32(c8, c9, 0x5511u);
            A0[0] = q4x2_lo(w01);
            A0[1] = q4x2_lo(x01);
            A0[2] = q4x2_lo(w89);
            A0[3] = q4x2_lo(x89);
            A1[0] = q4x2_hi(w01);
            A1[1] = q4x2_hi(x01);
            A1[2] = q4x2_hi(w89);
            A1[3] = q4x2_hi(x89);
        } else {
            uint32_t vw[4];
            if (SWZ) {
                const uint32_t pl = kPlane * (b >> 2);
                const uint32_t c0 = (va0 ^ (32u * (b & 3))) + pl;
                const uint32_t c1 = (va1 ^ (32u * (b & 3))) + pl;
                vw[0] = lds32(c0);
                vw[1] = lds32(c1);
                vw[2] = lds32(c0 + 1024u);
                vw[3] = lds32(c1 + 1024u);
            } else {
                const uint32_t c0 = va0 + 32u * b;
                vw[0] = lds32(c0);
                vw[1] = lds32(c0 + D);
                vw[2] = lds32(c0 + 8u * D);
                vw[3] = lds32(c0 + 9u * D);
            }
            const uint32_t f0 = vw[0] ^ 0x80808080u, f1 = vw[1] ^ 0x80808080u;
            const uint32_t f2 = vw[2] ^ 0x80808080u, f3 = vw[3] ^ 0x80808080u;
            const uint32_t u00 = prmt_b32(f0, f1, 0x5140u), u01 = prmt_b32(f0, f1, 0x7362u);
            const uint32_t u10 = prmt_b32(f2, f3, 0x5140u), u11 = prmt_b32(f2, f3, 0x7362u);
            A0[0] = i8x2_lo(u00);
            A0[1] = i8x2_hi(u00);
            A0[2] = i8x2_lo(u10);
            A0[3] = i8x2_hi(u10);
            A1[0] = i8x2_lo(u01);
            A1[1] = i8x2_hi(u01);
            A1[2] = i8x2_lo(u11);
            A1[3] = i8x2_hi(u11);
        }
        const uint32_t sel = (b & 1) ? 0x7632u : 0x5410u;
        const uint32_t s01 = prmt_b32(vsw[0][b >> 1], vsw[1][b >> 1], sel);
        const uint32_t s89 = prmt_b32(vsw[2][b >> 1], vsw[3][b >> 1], sel);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t pb0 = hmul2_u32(ph[nt][0], s01), pb1 = hmul2_u32(ph[nt][1], s89);
            mma_16816(oacc[nt][2 * b], A0[0], A0[1], A0[2], A0[3], pb0, pb1);
            mma_16816(oacc[nt][2 * b + 1], A1[0], A1[1], A1[2], A1[3], pb0, pb1);
        }
    }
}

// ---------------------------------------------------------------------------------------
// Q8_0: self-loading warps.  The Q8_0 kernels are bound by their consumer warps (every K
// and V byte costs an int8 -> f16 conversion), so they drop the producer warp: each of the
// CTA's W warps streams its own 16-cell chunks through a private ring of S stages (TMA
// boxes of 16 rows for one-run chunks, one bulk copy per row otherwise, cp.async for the
// scales) and attends to them.  The warps of a CTA take interleaved chunks of the same unit
// (chunk j goes to warp j mod W) and meet in the same end-of-unit exchange as above.  With
// no producer warp, all the registers of an SM go to warps that compute.
// ---------------------------------------------------------------------------------------
// Byte offset of KV head g's scales within its cell's 16-byte stage row, and the first
// element (in halves) of the 16-byte scale box that holds them.
template <int D>
__device__ __forceinline__ int scl_off(int g) {
    return 2 * ((g * (D / 32)) & 7);
}
template <int D>
__device__ __forceinline__ int scl_box_x(int g) {
    return (g * (D / 32)) & ~7;
}

template <int D, bool VQ4 = false, bool KQ4 = false, bool MQ = false>
struct Q8Self {
    static constexpr int kRowBytes = KQ4 ? D / 2 : D;              // K row per (cell, KV head): int8 or 4-bit
    static constexpr int kVRowBytes = VQ4 ? D / 2 : D;             // V row: int8, or two 4-bit values a byte
    static constexpr int kPlanes = D / 128;
    static constexpr int kPlane = kChunkCells * 128;               // one 128-byte-wide plane
    static constexpr int kSection = KQ4 ? kChunkCells * kRowBytes : kPlanes * kPlane;  // K rows (V rows follow)
    static constexpr int kVSection = kChunkCells * kVRowBytes;     // V rows of a chunk
    static constexpr int kChunkBytes = kSection + kVSection;       // a multiple of 1024
    static constexpr int kSclBytes = D / 16;                       // D/32 half scales per row
    // scales in a stage: one 16-byte row per cell (the tensor-map box row), K rows then V
    // rows; a head's D/32 halves sit at byte scl_off(g) of its cell's row (head_dim 128: the
    // rows hold the scales of the KV-head pair g & ~1, g | 1)
    static constexpr int kSclRow = 16;
    static constexpr int kSclChunk = 2 * kChunkCells * kSclRow;  // K then V scales
    // exchange slot of a warp: its O fragments ([N tiles][D/16][32 lanes] float4), max, sum
    static constexpr int kXchgSlot = ((MQ ? 2 : 1) * (D / 16) * 32 * 16 + (MQ ? 128 : 64) + 1023) / 1024 * 1024;
    static_assert(kChunkBytes % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
};

template <int D, int W, int S, bool VQ4 = false, bool KQ4 = false, bool MQ = false>
constexpr int q8_self_smem() {
    using Q = Q8Self<D, VQ4, KQ4, MQ>;
    return kHeaderBytes + 1024 + (W - 1) * Q::kXchgSlot + W * S * (Q::kChunkBytes + Q::kSclChunk);
}

// Position of a warp's load stream: unit u (its fields) and chunk j of it.  Units are
// numbered in 32 bits (checked on the host); a unit holds at most `split` cells.
struct ChunkCursor {
    int64_t i0;          // first plan entry / cell of the unit
    uint32_t u;
    int len;             // entries of the unit (i1 - i0)
    int s, g, j, n_chunks;
};

__device__ __forceinline__ int unit_chunks(const Unit& x) {
    return x.n_tiles == 0 ? 0 : (int)((x.i1 - x.i0 + kChunkCells - 1) / kChunkCells);
}

// Moves c forward (from chunk c.j of unit c.u) to the first chunk this warp owns; c.u >=
// n_units afterwards when the warp has no more chunks.
__device__ __forceinline__ void cursor_fill(const SplitDecodeParams& p, ChunkCursor& c) {
    const Unit x = unit_at(p, c.u);
    c.i0 = x.i0;
    c.len = (int)(x.i1 - x.i0);
    c.s = x.s;
    c.g = x.g;
    c.n_chunks = unit_chunks(x);
}
__device__ __forceinline__ void cursor_seek(const SplitDecodeParams& p, ChunkCursor& c, uint32_t n_units, int warp) {
    while (c.u < n_units && c.j >= c.n_chunks) {
        c.u += gridDim.x;
        c.j = warp;
        if (c.u < n_units) {
            const Unit x = unit_at(p, c.u);
            c.i0 = x.i0;
            c.len = (int)(x.i1 - x.i0);
            c.s = x.s;
            c.g = x.g;
            c.n_chunks = unit_chunks(x);
        }
    }
}

// MQ: multi-query units of up to 16 query rows (head_dim 128).  MQ8: multi-query units of up
// to 8 rows on the single-query geometry (head_dim 256), rows 8 rg .. 8 rg + 7 of the unit's
// row group rg, each lane's cell mask cut at its row's causal limit.
template <int D, int W, int S, bool VQ4 = false, bool KQ4 = false, bool MQ = false, bool MQ8 = false>
__device__ __forceinline__ void q8_self_body(const SplitDecodeParams& p) {
    static_assert(VQ4 || !KQ4, "4-bit keys come with 4-bit values");
    static_assert(!MQ || D == 128, "multi-query: head_dim 128");
    static_assert(!(MQ && MQ8), "one multi-query layout");
    constexpr int KVT = KVATTN_KV_Q8_0;  // 8-bit keys' query fragment order (load_q_frags)
    using Q = Q8Self<D, VQ4, KQ4, MQ>;
    using G = Geom<KVT, D>;
    static_assert(G::kSclBytes == Q::kSclBytes, "scale rows");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem);  // [W][S]
    uint64_t* xchg_bar = full_bar + W * S;                    // [0] W-1 warps posted, [1] area free
    uint32_t* st_mask = reinterpret_cast<uint32_t*>(xchg_bar + 2);  // [W][S]
    uint32_t* st_swz = st_mask + W * S;                              // [W][S]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(st_swz + W * S);
    unsigned char* xchg = smem + kHeaderBytes;  // W-1 slots: [D/16][32 lanes] float4, max[8], sum[8]
    unsigned char* rings = xchg + (W - 1) * Q::kXchgSlot;
    unsigned char* scales = rings + W * S * Q::kChunkBytes;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2;
    const int tq = lane & 3;
    const int H = p.n_head;
    // work units are numbered in 32 bits (checked on the host)
    const uint32_t n_units = (uint32_t)((int64_t)p.n_seq * p.unit_splits * p.n_head_kv * (p.n_rg > 1 ? p.n_rg : 1));

    if (threadIdx.x == 0) {
        for (int i = 0; i < W * S; ++i) mbar_init(smem_addr(&full_bar[i]), 64);
        mbar_init(smem_addr(&xchg_bar[0]), 32 * (W - 1 > 0 ? W - 1 : 1));
        mbar_init(smem_addr(&xchg_bar[1]), 32);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    __syncthreads();
    const bool one_wave = (int64_t)gridDim.x >= n_units;
    if (one_wave) pdl_launch_dependents();  // see split_decode_body
    // While the previous kernel drains (this CTA may be resident already, waiting for it),
    // each warp pulls the first chunks it will load into L2.  The lengths read here may still
    // change before the dependency wait; they only steer these hints, never the loads (boxes
    // outside the cache are not fetched).
    if (lane == 0 && p.use_tma != 0 && p.scl_tma != 0 && p.plan == nullptr && blockIdx.x < n_units) {
        const Unit x = unit_at(p, blockIdx.x);
        const int nch = unit_chunks(x);
        for (int j = warp, k = 0; j < nch && k <= S; j += W, ++k) {
            const int64_t base = (int64_t)x.s * p.n_cells + x.i0 + (int64_t)j * kChunkCells;
            if (base >= INT_MAX / 2) break;
            if constexpr (!KQ4 && Q::kPlanes > 1)
                tma_prefetch_4d(&p.tmap_k, 0, (int)base, 0, x.g);
            else
                tma_prefetch_3d(&p.tmap_k, 0, x.g, (int)base);
            if constexpr (!VQ4 && Q::kPlanes > 1)
                tma_prefetch_4d(&p.tmap_v, 0, (int)base, 0, x.g);
            else
                tma_prefetch_3d(&p.tmap_v, 0, x.g, (int)base);
            tma_prefetch_2d(&p.tmap_ks, scl_box_x<D>(x.g), (int)base);
            tma_prefetch_2d(&p.tmap_vs, scl_box_x<D>(x.g), (int)base);
        }
    }
    pdl_wait();

    unsigned char* ring = rings + warp * S * Q::kChunkBytes;
    unsigned char* sring = scales + warp * S * Q::kSclChunk;
    uint64_t* fb = full_bar + warp * S;
    bool bad = false;

    // The chunk's K and V rows by TMA into the stage at kdst: 8-bit rows of 256 bytes in one
    // 4-D box each (both 128-byte swizzled planes), 128-byte 8-bit rows and 4-bit rows (64
    // or 128 bytes) in one 3-D box.
    auto load_rows = [&](uint32_t kdst, int g, int base, uint32_t bar, uint64_t pol) {
        if constexpr (!KQ4 && Q::kPlanes > 1)
            tma_load_4d_hint(kdst, &p.tmap_k, 0, base, 0, g, bar, pol);
        else
            tma_load_3d_hint(kdst, &p.tmap_k, 0, g, base, bar, pol);
        if constexpr (!VQ4 && Q::kPlanes > 1)
            tma_load_4d_hint(kdst + Q::kSection, &p.tmap_v, 0, base, 0, g, bar, pol);
        else
            tma_load_3d_hint(kdst + Q::kSection, &p.tmap_v, 0, g, base, bar, pol);
    };

    // Issues the loads of chunk c.j of unit c.u into stage st.
    // Cache without a plan: the chunk's cells are consecutive rows, so the mask, the box
    // coordinate and the scale rows follow from 32-bit offsets into the unit.
    auto issue_contiguous = [&](const ChunkCursor& c, int st, uint32_t extra_tx) {
        const int off = c.j * kChunkCells;
        const int rem = c.len - off;  // cells of the unit from this chunk on (>= 1)
        const uint32_t mask = rem >= kChunkCells ? 0xffffu : (1u << rem) - 1u;
        const int64_t base = (int64_t)c.s * p.n_cells + c.i0 + off;
        const bool use_tma = p.use_tma != 0 && base < INT_MAX / 2;
        unsigned char* stage = ring + st * Q::kChunkBytes;
        const uint32_t bar = smem_addr(&fb[st]);
        if (use_tma && p.scl_tma != 0) {
            // every byte of the chunk comes by TMA: one lane issues, the others only arrive
            if (lane == 0) {
                st_mask[warp * S + st] = mask;
                st_swz[warp * S + st] = 1u;
                mbar_expect_tx(bar, (uint32_t)(Q::kChunkBytes + Q::kSclChunk) + extra_tx);
                const uint64_t pol = l2_evict_first_policy();
                const uint32_t kdst = smem_addr(stage);
                load_rows(kdst, c.g, (int)base, bar, pol);
                const uint32_t sdst = smem_addr(sring + st * Q::kSclChunk);
                tma_load_2d_hint(sdst, &p.tmap_ks, scl_box_x<D>(c.g), (int)base, bar, pol);
                tma_load_2d_hint(sdst + kChunkCells * Q::kSclRow, &p.tmap_vs, scl_box_x<D>(c.g), (int)base, bar, pol);
            }
            __syncwarp();
            cp_async_arrive_noinc(bar);  // (no copies pending: the barrier's 64 arrivals)
            mbar_arrive(bar);
            return;
        }
        const bool valid = lane < (rem < kChunkCells ? rem : kChunkCells);
        const bool scl_tma = use_tma && p.scl_tma != 0;
        if (lane == 0) {
            st_mask[warp * S + st] = mask;
            st_swz[warp * S + st] = use_tma ? 1u : 0u;
            const uint32_t bytes =
                use_tma ? (uint32_t)(Q::kChunkBytes + (scl_tma ? Q::kSclChunk : 0))
                        : (uint32_t)__popc(mask) * (uint32_t)(Q::kRowBytes + Q::kVRowBytes);
            mbar_expect_tx(bar, bytes + extra_tx);
        }
        __syncwarp();
        const int64_t row = (base + lane) * p.n_head_kv + c.g;  // this lane's (cell, KV head) row
        if (use_tma) {
            if (lane == 0) {
                const uint32_t kdst = smem_addr(stage);
                load_rows(kdst, c.g, (int)base, bar, l2_evict_first_policy());
                if (scl_tma) {
                    const uint32_t sdst = smem_addr(sring + st * Q::kSclChunk);
                    tma_load_2d_hint(sdst, &p.tmap_ks, scl_box_x<D>(c.g), (int)base, bar, l2_evict_first_policy());
                    tma_load_2d_hint(sdst + kChunkCells * Q::kSclRow, &p.tmap_vs, scl_box_x<D>(c.g), (int)base, bar,
                                     l2_evict_first_policy());
                }
            }
        } else if (valid) {
            bulk_g2s(smem_addr(stage + lane * Q::kRowBytes), static_cast<const char*>(p.k) + row * Q::kRowBytes,
                     Q::kRowBytes, bar);
            bulk_g2s(smem_addr(stage + Q::kSection + lane * Q::kVRowBytes),
                     static_cast<const char*>(p.v) + row * Q::kVRowBytes, Q::kVRowBytes, bar);
        }
        if (lane < kChunkCells && !scl_tma) {
            unsigned char* ksd = sring + st * Q::kSclChunk + lane * Q::kSclRow + scl_off<D>(c.g);
            unsigned char* vsd = ksd + kChunkCells * Q::kSclRow;
            if (valid) {
                if (D == 128) {
                    cp_async_8(smem_addr(ksd), p.k_scale + row * (D / 32));
                    cp_async_8(smem_addr(vsd), p.v_scale + row * (D / 32));
                } else {
                    cp_async_16(smem_addr(ksd), p.k_scale + row * (D / 32));
                    cp_async_16(smem_addr(vsd), p.v_scale + row * (D / 32));
                }
            } else {
#pragma unroll
                for (int k = 0; k < Q::kSclBytes / 4; ++k) {
                    reinterpret_cast<uint32_t*>(ksd)[k] = 0u;
                    reinterpret_cast<uint32_t*>(vsd)[k] = 0u;
                }
            }
        }
        cp_async_arrive_noinc(bar);
        mbar_arrive(bar);
    };

    // Any cache: plan entries, the one-run test, TMA or per-row copies.
    auto issue_general = [&](const ChunkCursor& c, int st, uint32_t extra_tx) {
        const int64_t c0 = c.i0 + (int64_t)c.j * kChunkCells;
        const int64_t i = c0 + lane;
        bool valid = lane < kChunkCells && c.j * kChunkCells + lane < c.len;
        int64_t cell = 0;
        if (valid) {
            if (p.plan != nullptr) {
                const int32_t e = __ldg(p.plan + (int64_t)c.s * p.plan_stride + i);
                if (e < -1 || (int64_t)e >= p.n_cells) {
                    bad = true;
                    valid = false;
                } else {
                    valid = e >= 0;
                    cell = e;
                }
            } else {
                cell = (int64_t)c.s * p.n_cells + i;
            }
        }
        const uint32_t mask = __ballot_sync(0xffffffffu, valid);
        int64_t base = (int64_t)c.s * p.n_cells + c0;
        bool run = true;
        if (p.plan != nullptr) {
            long long off_lo = valid ? (long long)(cell - i) : LLONG_MAX;
            long long off_hi = valid ? (long long)(cell - i) : LLONG_MIN;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                off_lo = min(off_lo, __shfl_xor_sync(0xffffffffu, off_lo, o));
                off_hi = max(off_hi, __shfl_xor_sync(0xffffffffu, off_hi, o));
            }
            run = mask != 0u && off_lo == off_hi;
            base = off_lo + c0;
        }
        const bool use_tma = run && p.use_tma != 0 && mask != 0u && base > INT_MIN / 2 && base < INT_MAX / 2;
        const bool scl_tma = use_tma && p.scl_tma != 0;
        unsigned char* stage = ring + st * Q::kChunkBytes;
        const uint32_t bar = smem_addr(&fb[st]);
        if (lane == 0) {
            st_mask[warp * S + st] = mask;
            st_swz[warp * S + st] = use_tma ? 1u : 0u;
            const uint32_t bytes =
                use_tma ? (uint32_t)(Q::kChunkBytes + (scl_tma ? Q::kSclChunk : 0))
                        : (uint32_t)__popc(mask) * (uint32_t)(Q::kRowBytes + Q::kVRowBytes);
            mbar_expect_tx(bar, bytes + extra_tx);
        }
        __syncwarp();
        const int64_t Hk = p.n_head_kv;
        if (use_tma) {
            if (lane == 0) {
                const uint32_t kdst = smem_addr(stage);
                load_rows(kdst, c.g, (int)base, bar, l2_evict_first_policy());
                if (scl_tma) {
                    const uint32_t sdst = smem_addr(sring + st * Q::kSclChunk);
                    tma_load_2d_hint(sdst, &p.tmap_ks, scl_box_x<D>(c.g), (int)base, bar, l2_evict_first_policy());
                    tma_load_2d_hint(sdst + kChunkCells * Q::kSclRow, &p.tmap_vs, scl_box_x<D>(c.g), (int)base, bar,
                                     l2_evict_first_policy());
                }
            }
        } else if (valid) {
            const int64_t row = cell * Hk + c.g;
            bulk_g2s(smem_addr(stage + lane * Q::kRowBytes), static_cast<const char*>(p.k) + row * Q::kRowBytes,
                     Q::kRowBytes, bar);
            bulk_g2s(smem_addr(stage + Q::kSection + lane * Q::kVRowBytes),
                     static_cast<const char*>(p.v) + row * Q::kVRowBytes, Q::kVRowBytes, bar);
        }
        // scales: a masked cell's are zero, so its (finite) int8 row contributes nothing
        if (lane < kChunkCells && !scl_tma) {
            unsigned char* ksd = sring + st * Q::kSclChunk + lane * Q::kSclRow + scl_off<D>(c.g);
            unsigned char* vsd = ksd + kChunkCells * Q::kSclRow;
            if (valid) {
                const int64_t row = cell * Hk + c.g;
                if (D == 128) {
                    cp_async_8(smem_addr(ksd), p.k_scale + row * (D / 32));
                    cp_async_8(smem_addr(vsd), p.v_scale + row * (D / 32));
                } else {
                    cp_async_16(smem_addr(ksd), p.k_scale + row * (D / 32));
                    cp_async_16(smem_addr(vsd), p.v_scale + row * (D / 32));
                }
            } else {
#pragma unroll
                for (int k = 0; k < Q::kSclBytes / 4; ++k) {
                    reinterpret_cast<uint32_t*>(ksd)[k] = 0u;
                    reinterpret_cast<uint32_t*>(vsd)[k] = 0u;
                }
            }
        }
        cp_async_arrive_noinc(bar);
        mbar_arrive(bar);
    };
    auto issue = [&](const ChunkCursor& c, int st, uint32_t extra_tx) {
        if (p.plan == nullptr)
            issue_contiguous(c, st, extra_tx);
        else
            issue_general(c, st, extra_tx);
    };

    // Prime the ring with this warp's first S chunks.
    ChunkCursor ld;
    ld.u = blockIdx.x;
    ld.j = warp;
    ld.n_chunks = 0;
    if (ld.u < n_units) cursor_fill(p, ld);
    cursor_seek(p, ld, n_units, warp);
    uint32_t L = 0;  // chunks issued
    for (; L < (uint32_t)S && ld.u < n_units; ++L) {
        issue(ld, (int)L, L == 0 ? p.stall_tx : 0u);
        ++ld.j;
        ld.j += W - 1;
        cursor_seek(p, ld, n_units, warp);
    }

    if constexpr (MQ) {
        // ---- causal multi-query consumers: 16 query rows (token r / G, head g G + r % G), or
        // row groups of 16 that are units of their own beyond that ----
        const int GQ = p.group, NQ = p.n_q;
        const int rows = GQ * NQ;
        const int64_t HR = (int64_t)NQ * H;  // partial rows per (sequence, split)
        uint32_t qa[D / 16][4];
        int64_t qa_key = -1;  // q_key of the rows whose query fragments qa holds
        uint32_t C = 0, X = 0;
        bool stop = false;
        constexpr float kLn2 = 0.69314718055994530942f;
        for (uint32_t u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
            const Unit x = unit_at(p, u);
            const int64_t part = (int64_t)x.s * p.part_stride + p.part_base + x.split_idx;
            const int row0 = p.rg_rows * x.rg;  // the unit's first query row
            if (x.n_tiles == 0) {
                if (warp == 0 && x.write_empty) {
                    const int n_rows = p.n_rg > 1 ? (rows - row0 < p.rg_rows ? rows - row0 : p.rg_rows) : rows;
                    for (int idx = lane; idx < n_rows * D; idx += 32) {
                        const int r = row0 + idx / D;
                        const int d = idx % D;
                        const int64_t row = (int64_t)(r / GQ) * H + x.g * GQ + r % GQ;
                        p.part_o[(part * HR + row) * D + d] = 0.f;
                        if (d == 0) p.part_lse[part * HR + row] = -INFINITY;
                    }
                }
                continue;
            }
            if (qa_key != q_key(p, x)) {
                load_q_frags_mq_q8<D, KQ4>(p, x.s, x.g, gq, tq, row0, qa);
                qa_key = q_key(p, x);
            }
            float oacc[2][D / 16][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < D / 16; ++i) oacc[nt][i][0] = oacc[nt][i][1] = oacc[nt][i][2] = oacc[nt][i][3] = 0.f;
            float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
            // causal limit (logical position, exclusive) of the lane's rows row0 + gq and row0 + gq + 8
            const int64_t lim_row[2] = {x.len - NQ + 1 + (row0 + gq) / GQ, x.len - NQ + 1 + (row0 + gq + 8) / GQ};
            const int nch = unit_chunks(x);
            for (int j = warp; j < nch; j += W, ++C) {
                const int st = (int)(C % (uint32_t)S);
                const bool ok = mbar_wait_bounded(smem_addr(&fb[st]), (C / (uint32_t)S) & 1u, abort_flag, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    stop = true;
                    break;
                }
                const uint32_t mask = st_mask[warp * S + st] & 0xffffu;
                const bool swz = st_swz[warp * S + st] != 0u;
                const uint32_t kb = smem_addr(ring + st * Q::kChunkBytes);
                const uint32_t vb = kb + Q::kSection;
                const unsigned char* ks = sring + st * Q::kSclChunk + scl_off<D>(x.g);
                const unsigned char* vs = ks + kChunkCells * Q::kSclRow;
                if (swz && p.scl_tma != 0 && mask != 0xffffu) {
                    // the scale box brought masked cells' rows too (plan holes, cells past the
                    // unit): zero them, so that P = 0 never meets a non-finite V scale
                    if (lane < kChunkCells && !((mask >> lane) & 1u)) {
                        uint4* z = reinterpret_cast<uint4*>(sring + st * Q::kSclChunk + lane * Q::kSclRow);
                        z[0] = make_uint4(0u, 0u, 0u, 0u);
                        z[kChunkCells] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    __syncwarp();
                }
                if (mask != 0u) {
                    const int64_t p0 = x.i0 + (int64_t)j * kChunkCells;
                    int lim[2];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int64_t rel = lim_row[hh] - p0;
                        lim[hh] = rel < 0 ? 0 : (rel > kChunkCells ? kChunkCells : (int)rel);
                    }
                    if (swz)
                        q8_mq_chunk<D, true, VQ4, KQ4>(kb, vb, ks, vs, mask, lane, lim, qa, oacc, m_run, l_run,
                                                       p.scale_log2);
                    else
                        q8_mq_chunk<D, false, VQ4, KQ4>(kb, vb, ks, vs, mask, lane, lim, qa, oacc, m_run, l_run,
                                                        p.scale_log2);
                }
                // refill the stage just read with the chunk S ahead (every lane's reads are done)
                __syncwarp();
                if (ld.u < n_units) {
                    fence_proxy_async();
                    issue(ld, st, 0u);
                    ++L;
                    ld.j += W;
                    cursor_seek(p, ld, n_units, warp);
                }
            }
            if (stop) break;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 1);
                l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 2);
            }
            const int64_t un = u + gridDim.x;
            if (un < n_units) {
                const Unit y = unit_at(p, un);
                if (y.n_tiles > 0 && q_key(p, y) != qa_key) {
                    load_q_frags_mq_q8<D, KQ4>(p, y.s, y.g, gq, tq, p.rg_rows * y.rg, qa);
                    qa_key = q_key(p, y);
                }
            }
            if constexpr (W > 1) {
                if (warp > 0) {
                    if (X > 0) {
                        const bool ok = mbar_wait_bounded(smem_addr(&xchg_bar[1]), (X - 1) & 1u, abort_flag, p.wait_limit_ns);
                        if (!__all_sync(0xffffffffu, ok)) break;
                    }
                    unsigned char* slot = xchg + (warp - 1) * Q::kXchgSlot;
                    float4* xo = reinterpret_cast<float4*>(slot);
                    float* xm = reinterpret_cast<float*>(xo + 2 * (D / 16) * 32);
                    if (tq == 0) {
                        xm[gq] = m_run[0];
                        xm[8 + gq] = m_run[1];
                        xm[16 + gq] = l_run[0];
                        xm[24 + gq] = l_run[1];
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int mt = 0; mt < D / 16; ++mt)
                            xo[(nt * (D / 16) + mt) * 32 + lane] =
                                make_float4(oacc[nt][mt][0], oacc[nt][mt][1], oacc[nt][mt][2], oacc[nt][mt][3]);
                    __syncwarp();
                    mbar_arrive(smem_addr(&xchg_bar[0]));
                    ++X;
                    continue;
                }
                const bool ok = mbar_wait_bounded(smem_addr(&xchg_bar[0]), X & 1u, abort_flag, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, ok)) break;
            }
            // warp 0: combine the W warps' (max, sum, O) of query rows 8nt + 2tq + e, write them
            float fw[W][2][2], inv[2][2], lse[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = 8 * nt + 2 * tq + e;
                    float mw[W], lw[W];
                    mw[0] = __shfl_sync(0xffffffffu, m_run[nt], 8 * tq + 4 * e);
                    lw[0] = __shfl_sync(0xffffffffu, l_run[nt], 8 * tq + 4 * e);
#pragma unroll
                    for (int w = 1; w < W; ++w) {
                        const float* xm = reinterpret_cast<const float*>(xchg + (w - 1) * Q::kXchgSlot +
                                                                         2 * (D / 16) * 32 * 16);
                        mw[w] = xm[r];
                        lw[w] = xm[16 + r];
                    }
                    float M = mw[0];
#pragma unroll
                    for (int w = 1; w < W; ++w) M = fmaxf(M, mw[w]);
                    float den = 0.f;
#pragma unroll
                    for (int w = 0; w < W; ++w) {
                        fw[w][nt][e] = (mw[w] == -INFINITY) ? 0.f : fast_exp2(mw[w] - M);
                        den = fmaf(lw[w], fw[w][nt][e], den);
                    }
                    const bool have = M != -INFINITY && den > 0.f;
                    inv[nt][e] = have ? 1.f / den : 0.f;
                    lse[nt][e] = have ? (M + fast_log2(den)) * kLn2 : -INFINITY;
                }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    float o0 = oacc[nt][mt][0] * fw[0][nt][0], o1 = oacc[nt][mt][1] * fw[0][nt][1];
                    float o2 = oacc[nt][mt][2] * fw[0][nt][0], o3 = oacc[nt][mt][3] * fw[0][nt][1];
#pragma unroll
                    for (int w = 1; w < W; ++w) {
                        const float4 t = reinterpret_cast<const float4*>(xchg + (w - 1) * Q::kXchgSlot)
                            [(nt * (D / 16) + mt) * 32 + lane];
                        o0 = fmaf(t.x, fw[w][nt][0], o0);
                        o1 = fmaf(t.y, fw[w][nt][1], o1);
                        o2 = fmaf(t.z, fw[w][nt][0], o2);
                        o3 = fmaf(t.w, fw[w][nt][1], o3);
                    }
                    oacc[nt][mt][0] = o0 * inv[nt][0];
                    oacc[nt][mt][1] = o1 * inv[nt][1];
                    oacc[nt][mt][2] = o2 * inv[nt][0];
                    oacc[nt][mt][3] = o3 * inv[nt][1];
                }
            if constexpr (W > 1) {
                __syncwarp();
                mbar_arrive(smem_addr(&xchg_bar[1]));
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = row0 + 8 * nt + 2 * tq + e;
                    if (r < rows) {
                        const int64_t row = (int64_t)(r / GQ) * H + x.g * GQ + r % GQ;
                        float* orow = p.part_o + (part * HR + row) * D;
#pragma unroll
                        for (int b = 0; b < D / 32; ++b) {
                            if constexpr (VQ4) {
                                *reinterpret_cast<float2*>(orow + 32 * b + 2 * gq) =
                                    make_float2(oacc[nt][2 * b][e], oacc[nt][2 * b][2 + e]);
                                *reinterpret_cast<float2*>(orow + 32 * b + 16 + 2 * gq) =
                                    make_float2(oacc[nt][2 * b + 1][e], oacc[nt][2 * b + 1][2 + e]);
                            } else {
                                *reinterpret_cast<float4*>(orow + 32 * b + 4 * gq) =
                                    make_float4(oacc[nt][2 * b][e], oacc[nt][2 * b][2 + e], oacc[nt][2 * b + 1][e],
                                                oacc[nt][2 * b + 1][2 + e]);
                            }
                        }
                        if (gq == 0) p.part_lse[part * HR + row] = lse[nt][e];
                    }
                }
            ++X;
        }
    } else {
        uint32_t qa[D / 16][2];
        int64_t qa_key = -1;  // q_key of the rows whose query fragments qa holds
        uint32_t C = 0;  // chunks consumed
        uint32_t X = 0;  // exchanges
        bool stop = false;
        constexpr float kLn2 = 0.69314718055994530942f;
        // multi-query units (MQ8): row r = 8 rg + r_local of the unit's KV head is partial row
        // (r / G) H + g G + r % G of n_q H per (sequence, split)
        auto mq_row = [&](const Unit& y, int r_local, bool& ok) -> int64_t {
            const int r = 8 * y.rg + r_local;
            ok = r < p.group * p.n_q;
            return (int64_t)(r / p.group) * H + y.g * p.group + r % p.group;
        };
        // head-pair units (head_dim 256 only): the partials keep head_dim 128
        const bool pair = D == 256 && !MQ8 && p.pair != 0;
        const int DO = pair ? D / 2 : D;
        auto load_q = [&](const Unit& y) {
            if constexpr (D == 256 && !MQ8) {
                if (pair) {
                    load_q_frags_pair<KQ4>(p, y.s, y.g, gq, tq, qa);
                    return;
                }
            }
            if (KQ4)
                load_q_frags_q4k<D>(p, y.s, y.g, gq, tq, qa, MQ8 ? y.rg : -1);
            else
                load_q_frags<KVT, D>(p, y.s, y.g, gq, tq, qa, MQ8 ? y.rg : -1);
        };
        for (uint32_t u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
            const Unit x = unit_at(p, u);
            const int64_t part = (int64_t)x.s * p.part_stride + p.part_base + x.split_idx;
            if (x.n_tiles == 0) {
                if (warp == 0 && x.write_empty) {
                    if constexpr (MQ8) {
                        const int64_t HR = (int64_t)p.n_q * H;
                        for (int idx = lane; idx < 8 * D; idx += 32) {
                            bool ok;
                            const int64_t row = mq_row(x, idx / D, ok);
                            const int d = idx % D;
                            if (ok) {
                                p.part_o[(part * HR + row) * D + d] = 0.f;
                                if (d == 0) p.part_lse[part * HR + row] = -INFINITY;
                            }
                        }
                    } else {
                        for (int idx = lane; idx < p.group * DO; idx += 32) {
                            const int r = idx / DO;
                            const int d = idx - r * DO;
                            const int h = x.g * p.group + r;
                            p.part_o[(part * H + h) * DO + d] = 0.f;
                            if (d == 0) p.part_lse[part * H + h] = -INFINITY;
                        }
                    }
                }
                continue;
            }
            if (qa_key != q_key(p, x)) {
                load_q(x);
                qa_key = q_key(p, x);
            }
            // MQ8: causal limit (logical position, exclusive) of the lane's row 8 rg + gq
            const int64_t lim_row = MQ8 ? x.len - p.n_q + 1 + (8 * x.rg + gq) / p.group : 0;
            float oacc[D / 16][4];
            float m_run = -INFINITY, l_run = 0.f;
#pragma unroll
            for (int i = 0; i < D / 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
            const int nch = unit_chunks(x);
            for (int j = warp; j < nch; j += W, ++C) {
                const int st = (int)(C % (uint32_t)S);
                const bool ok = mbar_wait_bounded(smem_addr(&fb[st]), (C / (uint32_t)S) & 1u, abort_flag, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    stop = true;
                    break;
                }
                const uint32_t mask = st_mask[warp * S + st] & 0xffffu;
                const bool swz = st_swz[warp * S + st] != 0u;
                const uint32_t kb = smem_addr(ring + st * Q::kChunkBytes);
                const uint32_t vb = kb + Q::kSection;
                const unsigned char* ks = sring + st * Q::kSclChunk + scl_off<D>(x.g);
                const unsigned char* vs = ks + kChunkCells * Q::kSclRow;
                if (swz && p.scl_tma != 0 && mask != 0xffffu) {
                    // the scale box brought masked cells' rows too (plan holes, cells past the
                    // unit): zero them, so that P = 0 never meets a non-finite V scale
                    if (lane < kChunkCells && !((mask >> lane) & 1u)) {
                        uint4* z = reinterpret_cast<uint4*>(sring + st * Q::kSclChunk + lane * Q::kSclRow);
                        z[0] = make_uint4(0u, 0u, 0u, 0u);
                        z[kChunkCells] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    __syncwarp();
                }
                // (fragments are read straight from the stage: staging them in registers first
                // measured slower here, the extra registers spill at this CTA count)
                if (mask != 0u) {
                    uint32_t lmask = mask;  // this lane's cells
                    if constexpr (MQ8) {    // the lane's row sees the chunk's cells below its limit
                        const int64_t rel = lim_row - (x.i0 + (int64_t)j * kChunkCells);
                        const int lim = rel < 0 ? 0 : (rel > kChunkCells ? kChunkCells : (int)rel);
                        lmask &= (1u << lim) - 1u;
                    }
                    if constexpr (VQ4) {
                        if (swz)
                            q4v_chunk<D, true, KQ4>(kb, vb, ks, vs, lmask, lane, qa, oacc, m_run, l_run, p.scale_log2);
                        else
                            q4v_chunk<D, false, KQ4>(kb, vb, ks, vs, lmask, lane, qa, oacc, m_run, l_run, p.scale_log2);
                    } else {
                        if (swz)
                            q8_chunk_swz<D>(kb, vb, ks, vs, lmask, lane, qa, oacc, m_run, l_run, p.scale_log2);
                        else
                            consume_tile<KVT, D, false, Q::kPlane, Q::kSclRow>(kb, vb, ks, vs, lmask, 0, lane, qa, oacc, m_run,
                                                                   l_run, p.scale_log2);
                    }
                }
                // refill the stage just read with the chunk S ahead (every lane's reads are done)
                __syncwarp();
                if (ld.u < n_units) {
                    fence_proxy_async();
                    issue(ld, st, 0u);
                    ++L;
                    ld.j += W;
                    cursor_seek(p, ld, n_units, warp);
                }
            }
            if (stop) break;
            l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
            l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
            const int64_t un = u + gridDim.x;
            if (un < n_units) {
                const Unit y = unit_at(p, un);
                if (y.n_tiles > 0 && q_key(p, y) != qa_key) {
                    load_q(y);
                    qa_key = q_key(p, y);
                }
            }
            if constexpr (W > 1) {
                // the warp that combines and writes the unit rotates with the exchange count,
                // so that every warp takes its share of that work; the others post their
                // (max, sum, O) to slots 0 .. W-2 in turn after it
                const int comb = (int)(X % (uint32_t)W);
                if (warp != comb) {
                    if (X > 0) {
                        const bool ok = mbar_wait_bounded(smem_addr(&xchg_bar[1]), (X - 1) & 1u, abort_flag, p.wait_limit_ns);
                        if (!__all_sync(0xffffffffu, ok)) break;
                    }
                    unsigned char* slot = xchg + ((warp - comb - 1 + W) % W) * Q::kXchgSlot;
                    float4* xo = reinterpret_cast<float4*>(slot);
                    float* xm = reinterpret_cast<float*>(xo + (D / 16) * 32);
                    if (tq == 0) {
                        xm[gq] = m_run;
                        xm[8 + gq] = l_run;
                    }
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt)
                        xo[mt * 32 + lane] = make_float4(oacc[mt][0], oacc[mt][1], oacc[mt][2], oacc[mt][3]);
                    __syncwarp();
                    mbar_arrive(smem_addr(&xchg_bar[0]));
                    ++X;
                    continue;
                }
                const bool ok = mbar_wait_bounded(smem_addr(&xchg_bar[0]), X & 1u, abort_flag, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, ok)) break;
            }
            // the combining warp: merge the W warps' (max, sum, O) for rows 2tq, 2tq+1 and write
            // the partial
            float mw[W][2], lw[W][2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                mw[0][e] = __shfl_sync(0xffffffffu, m_run, 8 * tq + 4 * e);
                lw[0][e] = __shfl_sync(0xffffffffu, l_run, 8 * tq + 4 * e);
#pragma unroll
                for (int w = 1; w < W; ++w) {
                    const float* xm = reinterpret_cast<const float*>(xchg + (w - 1) * Q::kXchgSlot + (D / 16) * 32 * 16);
                    mw[w][e] = xm[2 * tq + e];
                    lw[w][e] = xm[8 + 2 * tq + e];
                }
            }
            float fw[W][2], inv[2], lse[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float M = mw[0][e];
#pragma unroll
                for (int w = 1; w < W; ++w) M = fmaxf(M, mw[w][e]);
                float den = 0.f;
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    fw[w][e] = (mw[w][e] == -INFINITY) ? 0.f : fast_exp2(mw[w][e] - M);
                    den = fmaf(lw[w][e], fw[w][e], den);
                }
                const bool have = M != -INFINITY && den > 0.f;
                inv[e] = have ? 1.f / den : 0.f;
                lse[e] = have ? (M + fast_log2(den)) * kLn2 : -INFINITY;
            }
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                float o0 = oacc[mt][0] * fw[0][0], o1 = oacc[mt][1] * fw[0][1];
                float o2 = oacc[mt][2] * fw[0][0], o3 = oacc[mt][3] * fw[0][1];
#pragma unroll
                for (int w = 1; w < W; ++w) {
                    const float4 t = reinterpret_cast<const float4*>(xchg + (w - 1) * Q::kXchgSlot)[mt * 32 + lane];
                    o0 = fmaf(t.x, fw[w][0], o0);
                    o1 = fmaf(t.y, fw[w][1], o1);
                    o2 = fmaf(t.z, fw[w][0], o2);
                    o3 = fmaf(t.w, fw[w][1], o3);
                }
                oacc[mt][0] = o0 * inv[0];
                oacc[mt][1] = o1 * inv[1];
                oacc[mt][2] = o2 * inv[0];
                oacc[mt][3] = o3 * inv[1];
            }
            if constexpr (W > 1) {
                __syncwarp();
                mbar_arrive(smem_addr(&xchg_bar[1]));
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                bool ok;
                int64_t prow;  // partial row index (part, row)
                if constexpr (MQ8) {
                    const int64_t row = mq_row(x, 2 * tq + e, ok);
                    prow = part * ((int64_t)p.n_q * H) + row;
                } else {
                    const int r = 2 * tq + e;
                    ok = r < p.group;
                    prow = part * H + x.g * p.group + r;
                }
                if (ok) {
                    float* orow = p.part_o + prow * DO;
                    // head pairs: row 2tq + e keeps only its own head's half of the 256 dims
                    const int own = pair ? ((2 * tq + e) >= (p.group >> 1) ? 1 : 0) : -1;
#pragma unroll
                    for (int b = 0; b < D / 32; ++b) {
                        if (own >= 0 && (b >= D / 64 ? 1 : 0) != own) continue;
                        float* ob = orow + 32 * (own >= 0 ? b - own * (D / 64) : b);
                        if constexpr (VQ4) {
                            // 4-bit V: m-tile 2b holds dims 32b + 2gq (+1), m-tile 2b+1 dims 32b + 16 + 2gq (+1)
                            *reinterpret_cast<float2*>(ob + 2 * gq) = make_float2(oacc[2 * b][e], oacc[2 * b][2 + e]);
                            *reinterpret_cast<float2*>(ob + 16 + 2 * gq) =
                                make_float2(oacc[2 * b + 1][e], oacc[2 * b + 1][2 + e]);
                        } else {
                            *reinterpret_cast<float4*>(ob + 4 * gq) =
                                make_float4(oacc[2 * b][e], oacc[2 * b][2 + e], oacc[2 * b + 1][e], oacc[2 * b + 1][2 + e]);
                        }
                    }
                    if (gq == 0) p.part_lse[prow] = lse[e];
                }
            }
            ++X;
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, KVATTN_DEVICE_BAD_PLAN_ENTRY);
    // Every wait above is bounded, so all warps get here; a timed-out wait left abort set.
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag != 0) atomicOr(p.status, KVATTN_DEVICE_WAIT_TIMEOUT);
    if (!one_wave) pdl_launch_dependents();
}

#ifndef KVATTN_F16_D256_MIN_CTAS
#define KVATTN_F16_D256_MIN_CTAS 1
#endif

// Q8_0 geometry: warps per CTA, ring stages per warp, CTAs per SM.  head_dim 128: four
// warps of 128 registers, four CTAs on an SM (sixteen computing warps; measured faster
// than twelve warps of 168 registers); head_dim 256: two warps of up to 255 registers,
// four CTAs (eight computing warps, no spills; measured faster than four warps x two CTAs).
constexpr int kQ8W128 = 4, kQ8S128 = 2, kQ8B128 = 4;
constexpr int kQ8W256 = 2, kQ8S256 = 2, kQ8B256 = 4;
// One-warp CTAs for the head_dim-256 single-query kernels (real head_dim 256 and KV-head
// pairs), eight per SM with the same 255 registers: a unit per warp, no end-of-unit exchange.
// Taken when a call's units overflow one wave of the two-warp CTAs but fit one wave of these
// (Q8_0 over 131072 cells, head_dim 128 as 1024 KV-head-pair units: 62.9 -> 59.7 us per op;
// Q8_0 + Q4_0 60.3 -> 56.8, Q4_0 59.6 -> 56.0); with more units the two-warp kernels measured
// better (Q8_0 head_dim 256, 2048 units: 108.9 against 114.1 us), and a third stage gained
// nothing (60.4 us).
constexpr int kQ8S256One = 2, kQ8B256One = 8;
// Q8_0 multi-query (head_dim 128, up to 16 query rows): two warps of up to 255 registers,
// four CTAs per SM -- the two output tiles and the 16-row query fragments do not fit the
// single-query kernel's 128 registers.
constexpr int kQ8WMQ = 2, kQ8SMQ = 2, kQ8BMQ = 4;

// One kernel per (KV type, head_dim), each with its own register budget.
__global__ void __launch_bounds__(kThreads) split_decode_f16_d128(const __grid_constant__ SplitDecodeParams p) {
    split_decode_body<KVATTN_KV_F16, 128>(p);
}
__global__ void __launch_bounds__(kThreads, KVATTN_F16_D256_MIN_CTAS)
    split_decode_f16_d256(const __grid_constant__ SplitDecodeParams p) {
    split_decode_body<KVATTN_KV_F16, 256>(p);
}
__global__ void __launch_bounds__(kThreads) split_decode_mq_f16_d128(const __grid_constant__ SplitDecodeParams p) {
    split_decode_body<KVATTN_KV_F16, 128, true>(p);
}
// Up to 8 query rows per unit on the single-query geometry (small verification batches).
// 33 to 48 query rows per KV head: three consumer warps of 16 rows read each tile once.
__global__ void __launch_bounds__(4 * 32, 3) split_decode_mq3_f16_d128(const __grid_constant__ SplitDecodeParams p) {
    split_decode_body<KVATTN_KV_F16, 128, true, false, 3>(p);
}
__global__ void __launch_bounds__(kThreads) split_decode_mq8_f16_d128(const __grid_constant__ SplitDecodeParams p) {
    split_decode_body<KVATTN_KV_F16, 128, false, true>(p);
}
__global__ void __launch_bounds__(kThreads, KVATTN_F16_D256_MIN_CTAS)
    split_decode_mq8_f16_d256(const __grid_constant__ SplitDecodeParams p) {
    split_decode_body<KVATTN_KV_F16, 256, false, true>(p);
}
__global__ void __launch_bounds__(kThreads, KVATTN_F16_D256_MIN_CTAS)
    split_decode_mq_f16_d256(const __grid_constant__ SplitDecodeParams p) {
    split_decode_body<KVATTN_KV_F16, 256, true>(p);
}
__global__ void __launch_bounds__(kQ8W128 * 32, kQ8B128)
    split_decode_q8_d128(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<128, kQ8W128, kQ8S128>(p);
}
__global__ void __launch_bounds__(kQ8W256 * 32, kQ8B256)
    split_decode_q8_d256(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<256, kQ8W256, kQ8S256>(p);
}
// Q8_0 keys, Q4_0 values: the Q8_0 kernels with the second dequantisation on the V side.
__global__ void __launch_bounds__(kQ8W128 * 32, kQ8B128)
    split_decode_q8q4_d128(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<128, kQ8W128, kQ8S128, true>(p);
}
__global__ void __launch_bounds__(kQ8W256 * 32, kQ8B256)
    split_decode_q8q4_d256(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<256, kQ8W256, kQ8S256, true>(p);
}
__global__ void __launch_bounds__(kQ8WMQ * 32, kQ8BMQ)
    split_decode_mq_q8_d128(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<128, kQ8WMQ, kQ8SMQ, false, false, true>(p);
}
__global__ void __launch_bounds__(kQ8WMQ * 32, kQ8BMQ)
    split_decode_mq_q8q4_d128(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<128, kQ8WMQ, kQ8SMQ, true, false, true>(p);
}
__global__ void __launch_bounds__(kQ8WMQ * 32, kQ8BMQ)
    split_decode_mq_q4_d128(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<128, kQ8WMQ, kQ8SMQ, true, true, true>(p);
}
// Multi-query decode over the quantised caches, 8-row units on the single-query geometry:
// every row count at head_dim 256, up to 8 rows at head_dim 128.
__global__ void __launch_bounds__(kQ8W128 * 32, kQ8B128)
    split_decode_mq8_q8_d128(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<128, kQ8W128, kQ8S128, false, false, false, true>(p);
}
__global__ void __launch_bounds__(kQ8W128 * 32, kQ8B128)
    split_decode_mq8_q8q4_d128(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<128, kQ8W128, kQ8S128, true, false, false, true>(p);
}
__global__ void __launch_bounds__(kQ8W128 * 32, kQ8B128)
    split_decode_mq8_q4_d128(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<128, kQ8W128, kQ8S128, true, true, false, true>(p);
}
__global__ void __launch_bounds__(kQ8W256 * 32, kQ8B256)
    split_decode_mq_q8_d256(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<256, kQ8W256, kQ8S256, false, false, false, true>(p);
}
__global__ void __launch_bounds__(kQ8W256 * 32, kQ8B256)
    split_decode_mq_q8q4_d256(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<256, kQ8W256, kQ8S256, true, false, false, true>(p);
}
__global__ void __launch_bounds__(kQ8W256 * 32, kQ8B256)
    split_decode_mq_q4_d256(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<256, kQ8W256, kQ8S256, true, true, false, true>(p);
}
// Q4_0 keys and values.
__global__ void __launch_bounds__(kQ8W128 * 32, kQ8B128)
    split_decode_q4_d128(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<128, kQ8W128, kQ8S128, true, true>(p);
}
__global__ void __launch_bounds__(kQ8W256 * 32, kQ8B256)
    split_decode_q4_d256(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<256, kQ8W256, kQ8S256, true, true>(p);
}

// One-warp head_dim-256 single-query kernels (mode 4).
__global__ void __launch_bounds__(32, kQ8B256One) split_decode_q8_d256_w1(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<256, 1, kQ8S256One>(p);
}
__global__ void __launch_bounds__(32, kQ8B256One)
    split_decode_q8q4_d256_w1(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<256, 1, kQ8S256One, true>(p);
}
__global__ void __launch_bounds__(32, kQ8B256One) split_decode_q4_d256_w1(const __grid_constant__ SplitDecodeParams p) {
    q8_self_body<256, 1, kQ8S256One, true, true>(p);
}

// mode: 0 single-query, 1 multi-query, 2 f16 multi-query of up to 8 rows per unit on the
// single-query geometry (same resources as mode 0), 3 the three-consumer f16 multi-query
// kernel, 4 the one-warp quantised head_dim-256 single-query kernels.
const void* kernel_for(int kv_type, int head_dim, int mode = 0) {
    if (mode == 3) return reinterpret_cast<const void*>(split_decode_mq3_f16_d128);
    if (mode == 4) {
        if (kv_type == KVATTN_KV_Q8_0_Q4_0) return reinterpret_cast<const void*>(split_decode_q8q4_d256_w1);
        if (kv_type == KVATTN_KV_Q4_0) return reinterpret_cast<const void*>(split_decode_q4_d256_w1);
        return reinterpret_cast<const void*>(split_decode_q8_d256_w1);
    }
    if (mode == 2) {
        if (kv_type == KVATTN_KV_Q8_0) return reinterpret_cast<const void*>(split_decode_mq8_q8_d128);
        if (kv_type == KVATTN_KV_Q8_0_Q4_0) return reinterpret_cast<const void*>(split_decode_mq8_q8q4_d128);
        if (kv_type == KVATTN_KV_Q4_0) return reinterpret_cast<const void*>(split_decode_mq8_q4_d128);
        return head_dim == 256 ? reinterpret_cast<const void*>(split_decode_mq8_f16_d256)
                               : reinterpret_cast<const void*>(split_decode_mq8_f16_d128);
    }
    const bool mq = mode == 1;
    if (mq) {
        const bool d256 = head_dim == 256;
        if (kv_type == KVATTN_KV_Q8_0)
            return d256 ? reinterpret_cast<const void*>(split_decode_mq_q8_d256)
                        : reinterpret_cast<const void*>(split_decode_mq_q8_d128);
        if (kv_type == KVATTN_KV_Q8_0_Q4_0)
            return d256 ? reinterpret_cast<const void*>(split_decode_mq_q8q4_d256)
                        : reinterpret_cast<const void*>(split_decode_mq_q8q4_d128);
        if (kv_type == KVATTN_KV_Q4_0)
            return d256 ? reinterpret_cast<const void*>(split_decode_mq_q4_d256)
                        : reinterpret_cast<const void*>(split_decode_mq_q4_d128);
        return head_dim == 256 ? reinterpret_cast<const void*>(split_decode_mq_f16_d256)
                               : reinterpret_cast<const void*>(split_decode_mq_f16_d128);
    }
    if (kv_type == KVATTN_KV_F16)
        return head_dim == 128 ? reinterpret_cast<const void*>(split_decode_f16_d128)
                               : reinterpret_cast<const void*>(split_decode_f16_d256);
    if (kv_type == KVATTN_KV_Q8_0_Q4_0)
        return head_dim == 128 ? reinterpret_cast<const void*>(split_decode_q8q4_d128)
                               : reinterpret_cast<const void*>(split_decode_q8q4_d256);
    if (kv_type == KVATTN_KV_Q4_0)
        return head_dim == 128 ? reinterpret_cast<const void*>(split_decode_q4_d128)
                               : reinterpret_cast<const void*>(split_decode_q4_d256);
    return head_dim == 128 ? reinterpret_cast<const void*>(split_decode_q8_d128)
                           : reinterpret_cast<const void*>(split_decode_q8_d256);
}

cudaError_t set_smem_attr(const void* fn) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
}

}  // namespace

int split_decode_max_smem() { return 227 * 1024; }

int split_decode_stage_bytes(int kv_type, int head_dim) {
    if (kv_type == KVATTN_KV_F16) return head_dim == 128 ? Geom<0, 128>::kBytes : Geom<0, 256>::kBytes;
    return head_dim == 128 ? Geom<1, 128>::kBytes : Geom<1, 256>::kBytes;
}

// Dynamic shared memory of one CTA: header, slack for aligning the ring to 1024 bytes,
// the end-of-unit exchange area and the stage ring.
// Q8_0 kernels have a fixed geometry (n_stages is ignored for them).
int split_decode_smem_bytes(int kv_type, int head_dim, int n_stages, int mode) {
    // (the head_dim-256 multi-query kernels run on the single-query geometry)
    const bool mq = mode == 1 || mode == 3;
    const bool mq128 = mq && head_dim == 128;
    if (mode == 4) {
        if (kv_type == KVATTN_KV_Q8_0_Q4_0) return q8_self_smem<256, 1, kQ8S256One, true>();
        if (kv_type == KVATTN_KV_Q4_0) return q8_self_smem<256, 1, kQ8S256One, true, true>();
        return q8_self_smem<256, 1, kQ8S256One>();
    }
    if (kv_type == KVATTN_KV_Q8_0 && mq128) return q8_self_smem<128, kQ8WMQ, kQ8SMQ, false, false, true>();
    if (kv_type == KVATTN_KV_Q8_0_Q4_0 && mq128) return q8_self_smem<128, kQ8WMQ, kQ8SMQ, true, false, true>();
    if (kv_type == KVATTN_KV_Q4_0 && mq128) return q8_self_smem<128, kQ8WMQ, kQ8SMQ, true, true, true>();
    if (kv_type == KVATTN_KV_Q8_0)
        return head_dim == 128 ? q8_self_smem<128, kQ8W128, kQ8S128>() : q8_self_smem<256, kQ8W256, kQ8S256>();
    if (kv_type == KVATTN_KV_Q8_0_Q4_0)
        return head_dim == 128 ? q8_self_smem<128, kQ8W128, kQ8S128, true>()
                               : q8_self_smem<256, kQ8W256, kQ8S256, true>();
    if (kv_type == KVATTN_KV_Q4_0)
        return head_dim == 128 ? q8_self_smem<128, kQ8W128, kQ8S128, true, true>()
                               : q8_self_smem<256, kQ8W256, kQ8S256, true, true>();
    const int xchg = mq && head_dim == 128 ? Geom<0, 128>::kXchgBytesMQ
                     : head_dim == 128       ? Geom<0, 128>::kXchgBytes
                                             : Geom<0, 256>::kXchgBytes;
    return kHeaderBytes + 1024 + xchg + n_stages * split_decode_stage_bytes(kv_type, head_dim);
}

int split_decode_block_threads(int kv_type, int head_dim, int mode) {
    const bool mq = mode == 1;
    if (mode == 3) return 4 * 32;
    if (mode == 4) return 32;
    if (kv_type != KVATTN_KV_F16 && mq && head_dim == 128) return kQ8WMQ * 32;
    if (kv_type != KVATTN_KV_F16) return (head_dim == 128 ? kQ8W128 : kQ8W256) * 32;
    return kThreads;
}

// Cells per TMA box of the kernel's tensor maps.
int split_decode_box_cells(int kv_type) { return kv_type == KVATTN_KV_F16 ? kTileCells : kChunkCells; }
int split_decode_max_stages() { return kMaxStages; }
int split_decode_threads() { return kThreads; }

cudaError_t split_decode_occupancy(int kv_type, int head_dim, int n_stages, int mode, int* blocks) {
    const void* fn = kernel_for(kv_type, head_dim, mode);
    cudaError_t err = set_smem_attr(fn);
    if (err != cudaSuccess) return err;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, fn, split_decode_block_threads(kv_type, head_dim, mode),
                                                         split_decode_smem_bytes(kv_type, head_dim, n_stages, mode));
}

cudaError_t launch_split_decode(const SplitDecodeParams& p, int kv_type, int head_dim, unsigned grid_ctas,
                                cudaStream_t stream, bool pdl) {
    const int res = p.mq == 2 ? 0 : p.mq;  // resources (mode 2 has the single-query ones)
    const void* fn = kernel_for(kv_type, head_dim, p.mq);
    static std::once_flag once[64][40];
    static cudaError_t attr_err[64][40];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const int which = 8 * p.mq + 2 * kv_type + (head_dim == 256 ? 1 : 0);
    std::call_once(once[dev & 63][which], [&] { attr_err[dev & 63][which] = set_smem_attr(fn); });
    if (attr_err[dev & 63][which] != cudaSuccess) return attr_err[dev & 63][which];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_ctas, 1, 1);
    cfg.blockDim = dim3((unsigned)split_decode_block_threads(kv_type, head_dim, res), 1, 1);
    cfg.dynamicSmemBytes = split_decode_smem_bytes(kv_type, head_dim, p.n_stages, res);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    void* args[] = {const_cast<SplitDecodeParams*>(&p)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace kvattn
