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
    // end-of-split merge area (aliases stage 0 once every tile is consumed)
    static constexpr int kOStride = D + 4;
    static constexpr int kCombineBytes = (2 * kConsumerWarps * 8 + kConsumerWarps * 8 * kOStride) * 4;
    static_assert(kCombineBytes <= kBytes, "combine area must fit in one stage");
};

// Byte address of (row r, byte b) of a K or V section in either layout.
template <bool SWZ, int PAD_ROW>
__device__ __forceinline__ uint32_t sec_addr(uint32_t base, int r, int b) {
    if (SWZ)
        return base + (b >> 7) * kPlaneBytes + r * 128 + ((((b >> 4) & 7) ^ (r & 7)) << 4) + (b & 15);
    return base + r * PAD_ROW + b;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3, %4}], [%5];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
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

// One consumer warp's 16 cells of a tile: scores, online softmax, P V.
template <int KVT, int D, bool SWZ>
__device__ __forceinline__ void consume_tile(uint32_t kb, uint32_t vb, const unsigned char* ks,
                                             const unsigned char* vs, uint32_t mask, int warp, int lane,
                                             const uint32_t (&qa)[D / 16][2], float (&oacc)[D / 16][4],
                                             float& m_run, float& l_run, float scale_log2) {
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
                ldsm_x4(sec_addr<SWZ, G::kPadRow>(kb, r0 + 8 * j + (lane & 7), (kk * 16 + 8 * (lane >> 3)) * 2),
                        b0, b1, b2, b3);
                mma_16816(sacc[j], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
                mma_16816(sacc[j], qa[kk + 1][0], 0u, qa[kk + 1][1], 0u, b2, b3);
            }
        }
    } else {
#pragma unroll
        for (int b = 0; b < D / 32; ++b) {
            float cb[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                cb[j][0] = cb[j][1] = cb[j][2] = cb[j][3] = 0.f;
                const int r = r0 + 8 * j + gq;
                // block b, half hb: d = 32b + 16hb + 4tq + {0,1 | 2,3}
                const uint32_t w0 = lds32(sec_addr<SWZ, G::kPadRow>(kb, r, 32 * b + 4 * tq)) ^ 0x80808080u;
                const uint32_t w1 = lds32(sec_addr<SWZ, G::kPadRow>(kb, r, 32 * b + 16 + 4 * tq)) ^ 0x80808080u;
                mma_16816(cb[j], qa[2 * b][0], 0u, qa[2 * b][1], 0u, i8x2_lo(w0), i8x2_hi(w0));
                mma_16816(cb[j], qa[2 * b + 1][0], 0u, qa[2 * b + 1][1], 0u, i8x2_lo(w1), i8x2_hi(w1));
            }
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int c = r0 + 8 * j + 2 * tq + e;
                    const __half dk = reinterpret_cast<const __half*>(ks + c * G::kSclBytes)[b];
                    sacc[j][e] = fmaf(cb[j][e], __half2float(dk), sacc[j][e]);
                }
        }
    }

    // ---- online softmax (log2 domain) ----
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
    const float m_new = fmaxf(m_run, tmax);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = fast_exp2(m_run - m_use);
    m_run = m_new;
    float pf[2][2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) pf[j][e] = fast_exp2(x[j][e] - m_use);

    const float alpha0 = __shfl_sync(0xffffffffu, alpha, 8 * tq);
    const float alpha1 = __shfl_sync(0xffffffffu, alpha, 8 * tq + 4);
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        oacc[mt][0] *= alpha0;
        oacc[mt][1] *= alpha1;
        oacc[mt][2] *= alpha0;
        oacc[mt][3] *= alpha1;
    }

    // ---- O^T += V^T P^T ----
    if (KVT == KVATTN_KV_F16) {
        uint32_t pb[2];
        float psum = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            pb[j] = pack_half2(pf[j][0], pf[j][1]);
            const float2 r = __half22float2(*reinterpret_cast<const __half2*>(&pb[j]));
            psum += r.x + r.y;
        }
        l_run = l_run * alpha + psum;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(sec_addr<SWZ, G::kPadRow>(vb, r0 + (lane & 7) + 8 * (lane >> 4),
                                                    (16 * mt + 8 * ((lane >> 3) & 1)) * 2),
                          a0, a1, a2, a3);
            mma_16816(oacc[mt], a0, a1, a2, a3, pb[0], pb[1]);
        }
    } else {
        l_run = l_run * alpha + (pf[0][0] + pf[0][1] + pf[1][0] + pf[1][1]);
        const __half* dv0 = reinterpret_cast<const __half*>(vs + (r0 + 2 * tq) * G::kSclBytes);
        const __half* dv1 = reinterpret_cast<const __half*>(vs + (r0 + 2 * tq + 1) * G::kSclBytes);
        const __half* dv2 = reinterpret_cast<const __half*>(vs + (r0 + 2 * tq + 8) * G::kSclBytes);
        const __half* dv3 = reinterpret_cast<const __half*>(vs + (r0 + 2 * tq + 9) * G::kSclBytes);
#pragma unroll
        for (int b = 0; b < D / 32; ++b) {
            const uint32_t pb0 = pack_half2(pf[0][0] * __half2float(dv0[b]), pf[0][1] * __half2float(dv1[b]));
            const uint32_t pb1 = pack_half2(pf[1][0] * __half2float(dv2[b]), pf[1][1] * __half2float(dv3[b]));
            const int off = 32 * b + 4 * gq;
            const uint32_t w00 = lds32(sec_addr<SWZ, G::kPadRow>(vb, r0 + 2 * tq, off)) ^ 0x80808080u;
            const uint32_t w01 = lds32(sec_addr<SWZ, G::kPadRow>(vb, r0 + 2 * tq + 1, off)) ^ 0x80808080u;
            const uint32_t w10 = lds32(sec_addr<SWZ, G::kPadRow>(vb, r0 + 2 * tq + 8, off)) ^ 0x80808080u;
            const uint32_t w11 = lds32(sec_addr<SWZ, G::kPadRow>(vb, r0 + 2 * tq + 9, off)) ^ 0x80808080u;
            // interleave the two cells of each pair: bytes 0,1 (hb 0) and bytes 2,3 (hb 1)
            const uint32_t u0[2] = {prmt_b32(w00, w01, 0x5140u), prmt_b32(w00, w01, 0x7362u)};
            const uint32_t u1[2] = {prmt_b32(w10, w11, 0x5140u), prmt_b32(w10, w11, 0x7362u)};
#pragma unroll
            for (int hb = 0; hb < 2; ++hb)
                mma_16816(oacc[2 * b + hb], i8x2_lo(u0[hb]), i8x2_hi(u0[hb]), i8x2_lo(u1[hb]), i8x2_hi(u1[hb]), pb0,
                          pb1);
        }
    }
}

// Online-softmax step shared by the consumer paths: masks the 2x2 scores a thread holds
// for query row gq, updates the running max, rescales O, returns the probabilities.
__device__ __forceinline__ void softmax_step(const float (&sacc)[2][4], uint32_t mask, int tq, float scale_log2,
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
    const float m_new = fmaxf(m_run, tmax);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    alpha = fast_exp2(m_run - m_use);
    m_run = m_new;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) pf[j][e] = fast_exp2(x[j][e] - m_use);
}

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

// head_dim 128: the warp copies every K/V fragment (and Q8_0 scale) of its 16 cells into
// registers, releases the stage to the producer at once, and only then computes, so the
// stage is refilled while the tensor-core work runs.
template <int KVT, bool SWZ>
__device__ __forceinline__ void consume_tile_staged(uint32_t kb, uint32_t vb, const unsigned char* ks,
                                                    const unsigned char* vs, uint32_t mask, int warp, int lane,
                                                    uint32_t empty_bar, const uint32_t (&qa)[8][2],
                                                    float (&oacc)[8][4], float& m_run, float& l_run,
                                                    float scale_log2) {
    constexpr int D = 128;
    using G = Geom<KVT, D>;
    const int gq = lane >> 2;
    const int tq = lane & 3;
    const int r0 = warp * kWarpCells;
    float sacc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;

    if (KVT == KVATTN_KV_F16) {
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
        softmax_step(sacc, mask, tq, scale_log2, m_run, alpha, pf);
        rescale_o<D>(oacc, alpha, tq);
        uint32_t pb[2];
        float psum = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            pb[j] = pack_half2(pf[j][0], pf[j][1]);
            const float2 r = __half22float2(*reinterpret_cast<const __half2*>(&pb[j]));
            psum += r.x + r.y;
        }
        l_run = l_run * alpha + psum;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) mma_16816(oacc[mt], vf[mt][0], vf[mt][1], vf[mt][2], vf[mt][3], pb[0], pb[1]);
    } else {
        uint32_t kw[4][2][2];   // [block][n-tile][half]
        uint32_t vw[4][4];      // [block][cell 2tq, 2tq+1, 2tq+8, 2tq+9]
        uint2 ksc[2][2];        // 4 half scales of cell r0 + 8j + 2tq + e
        uint2 vsc[4];           // 4 half scales of cells 2tq, 2tq+1, 2tq+8, 2tq+9
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int r = r0 + 8 * j + gq;
                kw[b][j][0] = lds32(sec_addr<SWZ, G::kPadRow>(kb, r, 32 * b + 4 * tq));
                kw[b][j][1] = lds32(sec_addr<SWZ, G::kPadRow>(kb, r, 32 * b + 16 + 4 * tq));
            }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int off = 32 * b + 4 * gq;
            vw[b][0] = lds32(sec_addr<SWZ, G::kPadRow>(vb, r0 + 2 * tq, off));
            vw[b][1] = lds32(sec_addr<SWZ, G::kPadRow>(vb, r0 + 2 * tq + 1, off));
            vw[b][2] = lds32(sec_addr<SWZ, G::kPadRow>(vb, r0 + 2 * tq + 8, off));
            vw[b][3] = lds32(sec_addr<SWZ, G::kPadRow>(vb, r0 + 2 * tq + 9, off));
        }
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                ksc[j][e] = *reinterpret_cast<const uint2*>(ks + (r0 + 8 * j + 2 * tq + e) * G::kSclBytes);
        vsc[0] = *reinterpret_cast<const uint2*>(vs + (r0 + 2 * tq) * G::kSclBytes);
        vsc[1] = *reinterpret_cast<const uint2*>(vs + (r0 + 2 * tq + 1) * G::kSclBytes);
        vsc[2] = *reinterpret_cast<const uint2*>(vs + (r0 + 2 * tq + 8) * G::kSclBytes);
        vsc[3] = *reinterpret_cast<const uint2*>(vs + (r0 + 2 * tq + 9) * G::kSclBytes);
        __syncwarp();
        mbar_arrive(empty_bar);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            float cb[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                cb[j][0] = cb[j][1] = cb[j][2] = cb[j][3] = 0.f;
                const uint32_t w0 = kw[b][j][0] ^ 0x80808080u, w1 = kw[b][j][1] ^ 0x80808080u;
                mma_16816(cb[j], qa[2 * b][0], 0u, qa[2 * b][1], 0u, i8x2_lo(w0), i8x2_hi(w0));
                mma_16816(cb[j], qa[2 * b + 1][0], 0u, qa[2 * b + 1][1], 0u, i8x2_lo(w1), i8x2_hi(w1));
            }
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const __half* sc = reinterpret_cast<const __half*>(&ksc[j][e]);
                    sacc[j][e] = fmaf(cb[j][e], __half2float(sc[b]), sacc[j][e]);
                }
        }
        float alpha, pf[2][2];
        softmax_step(sacc, mask, tq, scale_log2, m_run, alpha, pf);
        rescale_o<D>(oacc, alpha, tq);
        l_run = l_run * alpha + (pf[0][0] + pf[0][1] + pf[1][0] + pf[1][1]);
        const __half* dv0 = reinterpret_cast<const __half*>(&vsc[0]);
        const __half* dv1 = reinterpret_cast<const __half*>(&vsc[1]);
        const __half* dv2 = reinterpret_cast<const __half*>(&vsc[2]);
        const __half* dv3 = reinterpret_cast<const __half*>(&vsc[3]);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint32_t pb0 = pack_half2(pf[0][0] * __half2float(dv0[b]), pf[0][1] * __half2float(dv1[b]));
            const uint32_t pb1 = pack_half2(pf[1][0] * __half2float(dv2[b]), pf[1][1] * __half2float(dv3[b]));
            const uint32_t f0 = vw[b][0] ^ 0x80808080u, f1 = vw[b][1] ^ 0x80808080u;
            const uint32_t f2 = vw[b][2] ^ 0x80808080u, f3 = vw[b][3] ^ 0x80808080u;
            const uint32_t u0[2] = {prmt_b32(f0, f1, 0x5140u), prmt_b32(f0, f1, 0x7362u)};
            const uint32_t u1[2] = {prmt_b32(f2, f3, 0x5140u), prmt_b32(f2, f3, 0x7362u)};
#pragma unroll
            for (int hb = 0; hb < 2; ++hb)
                mma_16816(oacc[2 * b + hb], i8x2_lo(u0[hb]), i8x2_hi(u0[hb]), i8x2_lo(u1[hb]), i8x2_hi(u1[hb]), pb0,
                          pb1);
        }
    }
}

template <int KVT, int D>
__global__ void __launch_bounds__(kThreads) split_decode_kernel(const __grid_constant__ SplitDecodeParams p) {
    using G = Geom<KVT, D>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment of the stage ring (the 128-B swizzle repeats every 8 rows)
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty_bar = full_bar + kMaxStages;
    uint32_t* tile_mask = reinterpret_cast<uint32_t*>(empty_bar + kMaxStages);
    uint32_t* tile_swz = tile_mask + kMaxStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tile_swz + kMaxStages);
    unsigned char* stages = smem + kHeaderBytes;

    const int split_idx = blockIdx.x;
    const int g = blockIdx.y;
    const int s = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_stages = p.n_stages;

    if (threadIdx.x == 0) {
        for (int i = 0; i < n_stages; ++i) {
            mbar_init(smem_addr(&full_bar[i]), p.src_lsu ? 64 : G::kArrivals);
            mbar_init(smem_addr(&empty_bar[i]), kConsumerWarps * 32);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    __syncthreads();
    pdl_wait();

    // The split's range of plan entries / cells.
    // (the length and the descriptor are independent loads: issue both before using either)
    const int64_t cap = p.plan ? p.plan_stride : p.n_cells;
    int64_t L = p.seq_lens != nullptr ? (int64_t)p.seq_lens[s] : p.fixed_len;
    const int desc_valid = p.desc != nullptr ? p.desc[(int64_t)s * p.n_split + split_idx].x : 1;
    L = L < 0 ? 0 : L;
    L = L < p.max_len ? L : p.max_len;
    L = L < cap ? L : cap;
    const int64_t i0 = (int64_t)split_idx * p.split;
    const int64_t i1 = (i0 + p.split < L) ? i0 + p.split : L;
    const bool empty = i0 >= i1 || desc_valid == 0;
    const int n_tiles = empty ? 0 : (int)((i1 - i0 + kTileCells - 1) / kTileCells);
    if (empty) {
        // Nothing to read.  A fully masked split inside the length still reports (0, -inf)
        // for the merge; a split past the length writes only when the caller asked for
        // every partial slot.
        if (i0 < i1 || p.write_beyond) {
            const int64_t part = (int64_t)s * p.part_stride + p.part_base + split_idx;
            const int H = p.n_head;
            for (int idx = threadIdx.x; idx < p.group * D; idx += kThreads) {
                const int r = idx / D;
                const int d = idx - r * D;
                const int h = g * p.group + r;
                p.part_o[(part * H + h) * D + d] = 0.f;
                if (d == 0) p.part_lse[part * H + h] = -INFINITY;
            }
        }
        pdl_launch_dependents();
        return;
    }

    const int gq = lane >> 2;
    const int tq = lane & 3;
    float oacc[D / 16][4];
    float m_run = -INFINITY, l_run = 0.f;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

    if (warp == kConsumerWarps) {
        // ------------------------------- producer -------------------------------
        const int64_t Hk = p.n_head_kv;
        bool bad = false;
        // plan entries of this lane's cell, prefetched four tiles ahead
        const int32_t* prow = p.plan != nullptr ? p.plan + (int64_t)s * p.plan_stride : nullptr;
        auto plan_entry = [&](int tt) -> int32_t {
            const int64_t i = i0 + (int64_t)tt * kTileCells + lane;
            return (prow != nullptr && tt < n_tiles && i < i1) ? __ldg(prow + i) : -1;
        };
        int32_t e0 = plan_entry(0), e1 = plan_entry(1), e2 = plan_entry(2), e3 = plan_entry(3);
        for (int t = 0; t < n_tiles; ++t) {
            const int32_t e = e0;
            e0 = e1;
            e1 = e2;
            e2 = e3;
            e3 = plan_entry(t + 4);
            const int st = t % n_stages;
            const int use = t / n_stages;
            if (use > 0) {
                const bool ok =
                    mbar_wait_bounded(smem_addr(&empty_bar[st]), (uint32_t)((use - 1) & 1), abort_flag,
                                      p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, ok)) break;  // the whole warp agrees before any collective
            }
            const int64_t tile0 = i0 + (int64_t)t * kTileCells;
            const int64_t i = tile0 + lane;
            bool valid = i < i1;
            int64_t cell = 0;
            if (valid) {
                if (p.plan != nullptr) {
                    if (e < -1 || (int64_t)e >= p.n_cells) {
                        bad = true;
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
                mbar_expect_tx(bar, bytes + (t == 0 ? p.stall_tx : 0u));
            }
            __syncwarp();
            if (use_tma) {
                if (lane == 0) {
                    const uint32_t kdst = smem_addr(stage);
                    const uint32_t vdst = kdst + G::kSwzSection;
#pragma unroll
                    for (int pl = 0; pl < G::kPlanes; ++pl) {
                        const int x = pl * (KVT == KVATTN_KV_F16 ? 64 : 128);  // elements of 128 B
                        tma_load_3d(kdst + pl * kPlaneBytes, &p.tmap_k, x, g, (int)base, bar);
                        tma_load_3d(vdst + pl * kPlaneBytes, &p.tmap_v, x, g, (int)base, bar);
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
            if (KVT == KVATTN_KV_Q8_0) {
                const uint32_t ks = smem_addr(stage + G::kKsOff + lane * G::kSclBytes);
                unsigned char* vsp = stage + G::kVsOff + lane * G::kSclBytes;
                if (valid) {
                    const int64_t row = cell * Hk + g;
                    const __half* ksrc = p.k_scale + row * (D / 32);
                    const __half* vsrc = p.v_scale + row * (D / 32);
                    if (D == 128) {
                        cp_async_8(ks, ksrc);
                        cp_async_8(smem_addr(vsp), vsrc);
                    } else {
                        cp_async_16(ks, ksrc);
                        cp_async_16(smem_addr(vsp), vsrc);
                    }
                } else {
                    uint32_t* zs = reinterpret_cast<uint32_t*>(vsp);
#pragma unroll
                    for (int k = 0; k < G::kSclBytes / 4; ++k) zs[k] = 0u;
                    wrote = true;
                }
            }
            if (KVT == KVATTN_KV_Q8_0 || p.src_lsu) cp_async_arrive_noinc(bar);
            if (wrote) fence_proxy_async();  // zero-fills before later async writes to this stage
            mbar_arrive(bar);
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, KVATTN_DEVICE_BAD_PLAN_ENTRY);
    } else {
        // ------------------------------- consumers -------------------------------
        const int h = g * p.group + gq;
        const bool row_ok = gq < p.group;
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + ((int64_t)s * p.n_head + h) * D);
        uint32_t qa[D / 16][2];
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

        for (int t = 0; t < n_tiles; ++t) {
            const int st = t % n_stages;
            const int use = t / n_stages;
            const bool ok =
                mbar_wait_bounded(smem_addr(&full_bar[st]), (uint32_t)(use & 1), abort_flag, p.wait_limit_ns);
            if (!__all_sync(0xffffffffu, ok)) break;
            const uint32_t mask = (tile_mask[st] >> (warp * kWarpCells)) & 0xffffu;
            const bool swz = tile_swz[st] != 0u;
            unsigned char* stage = stages + st * G::kBytes;
            const uint32_t ebar = smem_addr(&empty_bar[st]);
            bool released = false;
            if (mask != 0u) {
                const unsigned char* ks = stage + G::kKsOff;
                const unsigned char* vs = stage + G::kVsOff;
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
                        consume_tile_staged<KVT, true>(kb, vb, ks, vs, mask, warp, lane, ebar, qa, oacc, m_run,
                                                       l_run, p.scale_log2);
                        released = true;
                    } else {
                        consume_tile<KVT, D, true>(kb, vb, ks, vs, mask, warp, lane, qa, oacc, m_run, l_run,
                                                   p.scale_log2);
                    }
                } else {
                    const uint32_t kb = smem_addr(stage);
                    const uint32_t vb = kb + G::kPadSection;
                    if constexpr (D == 128) {
                        consume_tile_staged<KVT, false>(kb, vb, ks, vs, mask, warp, lane, ebar, qa, oacc, m_run,
                                                        l_run, p.scale_log2);
                        released = true;
                    } else {
                        consume_tile<KVT, D, false>(kb, vb, ks, vs, mask, warp, lane, qa, oacc, m_run, l_run,
                                                    p.scale_log2);
                    }
                }
            }
            if (!released) {
                __syncwarp();
                mbar_arrive(ebar);
            }
        }
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    }

    // ------------------------- combine the consumer warps -------------------------
    __syncthreads();
    const bool aborted = *abort_flag != 0;
    const bool have = !aborted && n_tiles > 0;
    float* cm = reinterpret_cast<float*>(stages);       // [warps][8] running max (log2 units)
    float* cl = cm + kConsumerWarps * 8;                // [warps][8] running sum
    float* xm = cl + kConsumerWarps * 8;                // [8] this CTA's max (log2), -inf: no cell
    float* xl = xm + 8;                                 // [8] this CTA's sum
    float* co = xl + 8;                                 // [warps][8][D + 4]; warp 0's rows end up
                                                        // holding the CTA's unnormalised O
    if (have && warp < kConsumerWarps) {
        if (tq == 0) {
            cm[warp * 8 + gq] = m_run;
            cl[warp * 8 + gq] = l_run;
        }
        float* cw = co + warp * 8 * G::kOStride;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            const int d0 = out_dim<KVT>(mt, 0, gq);
            const int d1 = out_dim<KVT>(mt, 1, gq);
            cw[(2 * tq) * G::kOStride + d0] = oacc[mt][0];
            cw[(2 * tq + 1) * G::kOStride + d0] = oacc[mt][1];
            cw[(2 * tq) * G::kOStride + d1] = oacc[mt][2];
            cw[(2 * tq + 1) * G::kOStride + d1] = oacc[mt][3];
        }
    }
    __syncthreads();
    const int G_rows = p.group;
    if (threadIdx.x < 8) {
        const int r = threadIdx.x;
        float M = -INFINITY, den = 0.f;
        if (have && r < G_rows) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cm[w * 8 + r]);
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w)
                    if (cm[w * 8 + r] != -INFINITY) den = fmaf(fast_exp2(cm[w * 8 + r] - M), cl[w * 8 + r], den);
            }
        }
        xm[r] = den > 0.f ? M : -INFINITY;
        xl[r] = den;
    }
    if (have) {
        for (int idx = threadIdx.x; idx < G_rows * D; idx += kThreads) {
            const int r = idx / D;
            const int d = idx - r * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cm[w * 8 + r]);
            float o = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w)
                    if (cm[w * 8 + r] != -INFINITY)
                        o = fmaf(fast_exp2(cm[w * 8 + r] - M), co[(w * 8 + r) * G::kOStride + d], o);
            }
            co[r * G::kOStride + d] = o;  // warp 0's slot: read above by this thread only
        }
    }
    __syncthreads();

    constexpr float kLn2 = 0.69314718055994530942f;
    const int H = p.n_head;
    if (aborted) {
        if (threadIdx.x == 0) atomicOr(p.status, KVATTN_DEVICE_WAIT_TIMEOUT);
    } else {
        const int64_t part = (int64_t)s * p.part_stride + p.part_base + split_idx;
        for (int idx = threadIdx.x; idx < G_rows * D; idx += kThreads) {
            const int r = idx / D;
            const int d = idx - r * D;
            const int h = g * G_rows + r;
            const bool ok = xm[r] != -INFINITY;
            p.part_o[(part * H + h) * D + d] = ok ? co[r * G::kOStride + d] / xl[r] : 0.f;
            if (d == 0) p.part_lse[part * H + h] = ok ? (xm[r] + fast_log2(xl[r])) * kLn2 : -INFINITY;
        }
    }
    pdl_launch_dependents();
}

template <int KVT, int D>
const void* kernel_ptr() {
    return reinterpret_cast<const void*>(split_decode_kernel<KVT, D>);
}

const void* kernel_for(int kv_type, int head_dim) {
    if (kv_type == KVATTN_KV_F16) return head_dim == 128 ? kernel_ptr<0, 128>() : kernel_ptr<0, 256>();
    return head_dim == 128 ? kernel_ptr<1, 128>() : kernel_ptr<1, 256>();
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

// header + slack for aligning the ring to 1024 bytes
int split_decode_header_bytes() { return kHeaderBytes + 1024; }
int split_decode_max_stages() { return kMaxStages; }
int split_decode_threads() { return kThreads; }

cudaError_t split_decode_occupancy(int kv_type, int head_dim, int n_stages, int* blocks) {
    const void* fn = kernel_for(kv_type, head_dim);
    cudaError_t err = set_smem_attr(fn);
    if (err != cudaSuccess) return err;
    const int smem = split_decode_header_bytes() + n_stages * split_decode_stage_bytes(kv_type, head_dim);
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, fn, kThreads, smem);
}

cudaError_t launch_split_decode(const SplitDecodeParams& p, int kv_type, int head_dim, dim3 grid,
                                cudaStream_t stream, bool pdl) {
    const void* fn = kernel_for(kv_type, head_dim);
    static std::once_flag once[64][4];
    static cudaError_t attr_err[64][4];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const int which = (kv_type ? 2 : 0) + (head_dim == 256 ? 1 : 0);
    std::call_once(once[dev & 63][which], [&] { attr_err[dev & 63][which] = set_smem_attr(fn); });
    if (attr_err[dev & 63][which] != cudaSuccess) return attr_err[dev & 63][which];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes =
        split_decode_header_bytes() + p.n_stages * split_decode_stage_bytes(kv_type, head_dim);
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
