// Split-KV single-query decode attention: one CTA per (split, KV head, sequence).
//
// The computation is flash-decoding as the pages describe it ("Rolling-KV -- overflow
// throughput evaluations", sections 1 and 3: a decode op that emits its own LSE channel;
// "KVARN KV Performance optimizations", items 2, 6 and 9: GQA rows padded to eight
// physical rows, fully masked splits skipped, query rows sharing every decoded K/V
// byte, partials merged by max/numerator/denominator).  The kernel design is our own
// for sm_103a:
//
//  * warp 2 is the producer: each lane owns one cell of a 32-cell tile and moves that
//    cell's K row and V row (256 B each for f16, head_dim 128) from HBM into shared
//    memory with one 1-D bulk async copy (TMA engine) per row, completing on the
//    stage's mbarrier.  Holes (-1 plan entries, cells past the length, out-of-range
//    entries) issue no copy; their V row is zero-filled so that P = 0 never meets a
//    NaN.  A ring of n_stages stages keeps up to n_stages tiles in flight per CTA.
//  * warps 0 and 1 each consume 16 cells of every tile: S = q K^T on the tensor cores
//    (mma m16n8k16, the G <= 8 query rows of this KV head in the M dimension), an
//    online softmax in fp32 on exp2-scaled scores, and O^T += V^T P^T (head_dim in M,
//    query rows in N).  Each K/V byte is read from HBM once for all G query heads.
//  * Q8_0 is dequantised as it is consumed: int8 lanes become exact f16 with the
//    magic-number byte permutation, per-32 K scales multiply fp32 block dot products,
//    per-32 V scales are folded into the f16 P operand of each block.
//  * the two consumer warps merge their (m, l, O) through shared memory and write the
//    split's normalised partial O_p and its natural-log LSE_p.
//
// All waits are bounded (about 2 s of wall time); a wait that gives up sets a sticky
// status bit in the workspace and the CTA finishes without writing results.
#include <cmath>
#include <mutex>

#include "kvattn_internal.cuh"

namespace kvattn {

namespace {

constexpr int kMaxStages = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kHeaderBytes = 256;

template <int KVT, int D>
struct Geom;

template <int D>
struct Geom<KVATTN_KV_F16, D> {
    static constexpr int kRowK = D * 2 + 16;  // +16 B: ldmatrix rows land in distinct banks
    static constexpr int kRowV = D * 2 + 16;
    static constexpr int kSclK = 0;
    static constexpr int kSclV = 0;
    static constexpr int kRowBytes = D * 2;   // bytes copied per (cell, KV head) row
    static constexpr int kArrivals = 32;
};

template <int D>
struct Geom<KVATTN_KV_Q8_0, D> {
    static constexpr int kRowK = D + 32;      // 8-byte K fragment loads conflict-free
    static constexpr int kRowV = D + 16;      // 4-byte V fragment loads conflict-free
    static constexpr int kSclK = D / 16;      // D/32 half scales per row
    static constexpr int kSclV = D / 16;
    static constexpr int kRowBytes = D;
    static constexpr int kArrivals = 64;      // 32 lanes + 32 cp.async completion arrivals
};

template <int KVT, int D>
struct Stage {
    using G = Geom<KVT, D>;
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kTileCells * G::kRowK;
    static constexpr int kKsOff = kVOff + kTileCells * G::kRowV;
    static constexpr int kVsOff = kKsOff + kTileCells * G::kSclK;
    static constexpr int kBytes = ((kVsOff + kTileCells * G::kSclV) + 127) / 128 * 128;
    // end-of-split merge area (aliases stage 0 once every tile is consumed)
    static constexpr int kOStride = D + 4;
    static constexpr int kCombineBytes = (2 * kConsumerWarps * 8 + kConsumerWarps * 8 * kOStride) * 4;
    static_assert(kCombineBytes <= kBytes, "combine area must fit in one stage");
};

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

// Output head_dim index of accumulator slot (m-tile mt, upper half hi) for thread row gq.
template <int KVT>
__device__ __forceinline__ int out_dim(int mt, int hi, int gq) {
    if (KVT == KVATTN_KV_F16) return 16 * mt + 8 * hi + gq;
    // Q8_0: m-tile 2b+hb covers dims 32b + 4*gq + 2*hb + hi (block-aligned permutation)
    return 32 * (mt >> 1) + 4 * gq + 2 * (mt & 1) + hi;
}

template <int KVT, int D>
__global__ void __launch_bounds__(kThreads) split_decode_kernel(const SplitDecodeParams p) {
    using G = Geom<KVT, D>;
    using ST = Stage<KVT, D>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty_bar = full_bar + kMaxStages;
    uint32_t* tile_mask = reinterpret_cast<uint32_t*>(empty_bar + kMaxStages);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tile_mask + kMaxStages);
    unsigned char* stages = smem + kHeaderBytes;

    const int split_idx = blockIdx.x;
    const int g = blockIdx.y;
    const int s = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_stages = p.n_stages;

    if (threadIdx.x == 0) {
        for (int i = 0; i < n_stages; ++i) {
            mbar_init(smem_addr(&full_bar[i]), G::kArrivals);
            mbar_init(smem_addr(&empty_bar[i]), kConsumerWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    pdl_wait();

    // The split's range of plan entries / cells.
    const int64_t cap = p.plan ? p.plan_stride : p.n_cells;
    int64_t L = p.seq_lens != nullptr ? (int64_t)p.seq_lens[s] : p.fixed_len;
    L = L < 0 ? 0 : L;
    L = L < p.max_len ? L : p.max_len;
    L = L < cap ? L : cap;
    const int64_t i0 = (int64_t)split_idx * p.split;
    const int64_t i1 = (i0 + p.split < L) ? i0 + p.split : L;
    bool empty = i0 >= i1;
    if (!empty && p.desc != nullptr) empty = p.desc[(int64_t)s * p.n_split + split_idx].x == 0;
    const int n_tiles = empty ? 0 : (int)((i1 - i0 + kTileCells - 1) / kTileCells);

    // Per-consumer-thread state (unused by the producer warp).
    const int gq = lane >> 2;  // query row within the group (MMA row / N column)
    const int tq = lane & 3;
    float oacc[D / 16][4];
    float m_run = -INFINITY, l_run = 0.f;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

    if (warp == kConsumerWarps) {
        // ------------------------------- producer -------------------------------
        const int64_t Hk = p.n_head_kv;
        bool bad = false;
        for (int t = 0; t < n_tiles; ++t) {
            const int st = t % n_stages;
            const int use = t / n_stages;
            if (use > 0) {
                const bool ok =
                    mbar_wait_bounded(smem_addr(&empty_bar[st]), (uint32_t)((use - 1) & 1), abort_flag,
                                      p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, ok)) break;  // the whole warp agrees before any collective
            }
            const int64_t i = i0 + (int64_t)t * kTileCells + lane;
            bool valid = i < i1;
            int64_t cell = 0;
            if (valid) {
                if (p.plan != nullptr) {
                    const int32_t e = p.plan[(int64_t)s * p.plan_stride + i];
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
            unsigned char* stage = stages + st * ST::kBytes;
            const uint32_t bar = smem_addr(&full_bar[st]);
            if (lane == 0) {
                tile_mask[st] = mask;
                mbar_expect_tx(bar, (uint32_t)__popc(mask) * 2u * (uint32_t)G::kRowBytes +
                                        (t == 0 ? p.stall_tx : 0u));
            }
            __syncwarp();
            unsigned char* krow = stage + ST::kKOff + lane * G::kRowK;
            unsigned char* vrow = stage + ST::kVOff + lane * G::kRowV;
            if (valid) {
                const int64_t row = cell * Hk + g;
                bulk_g2s(smem_addr(krow), static_cast<const char*>(p.k) + row * G::kRowBytes,
                         G::kRowBytes, bar);
                bulk_g2s(smem_addr(vrow), static_cast<const char*>(p.v) + row * G::kRowBytes,
                         G::kRowBytes, bar);
                if (KVT == KVATTN_KV_Q8_0) {
                    const uint32_t ks = smem_addr(stage + ST::kKsOff + lane * G::kSclK);
                    const uint32_t vs = smem_addr(stage + ST::kVsOff + lane * G::kSclV);
                    const __half* ksrc = p.k_scale + row * (D / 32);
                    const __half* vsrc = p.v_scale + row * (D / 32);
                    if (D == 128) {
                        cp_async_8(ks, ksrc);
                        cp_async_8(vs, vsrc);
                    } else {
                        cp_async_16(ks, ksrc);
                        cp_async_16(vs, vsrc);
                    }
                }
            } else {
                uint4* z = reinterpret_cast<uint4*>(vrow);
#pragma unroll
                for (int k = 0; k < G::kRowBytes / 16; ++k) z[k] = make_uint4(0, 0, 0, 0);
                if (KVT == KVATTN_KV_Q8_0) {
                    uint32_t* zs = reinterpret_cast<uint32_t*>(stage + ST::kVsOff + lane * G::kSclV);
#pragma unroll
                    for (int k = 0; k < G::kSclV / 4; ++k) zs[k] = 0u;
                }
            }
            if (KVT == KVATTN_KV_Q8_0) cp_async_arrive_noinc(bar);
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
                d0 = 32 * (kk >> 1) + 8 * tq + 4 * (kk & 1);
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
            unsigned char* stage = stages + st * ST::kBytes;
            if (mask != 0u) {
                const uint32_t kb = smem_addr(stage + ST::kKOff) + warp * kWarpCells * G::kRowK;
                const uint32_t vb = smem_addr(stage + ST::kVOff) + warp * kWarpCells * G::kRowV;
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
                            ldsm_x4(kb + (8 * j + (lane & 7)) * G::kRowK + (kk * 16 + 8 * (lane >> 3)) * 2,
                                    b0, b1, b2, b3);
                            mma_16816(sacc[j], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
                            mma_16816(sacc[j], qa[kk + 1][0], 0u, qa[kk + 1][1], 0u, b2, b3);
                        }
                    }
                } else {
                    const unsigned char* ks = stage + ST::kKsOff + warp * kWarpCells * G::kSclK;
#pragma unroll
                    for (int b = 0; b < D / 32; ++b) {
                        float cb[2][4];
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            cb[j][0] = cb[j][1] = cb[j][2] = cb[j][3] = 0.f;
                            const uint2 w = lds64(kb + (8 * j + gq) * G::kRowK + 32 * b + 8 * tq);
                            const uint32_t b0 = i8pair_to_h2(w.x, w.x, 0x0100u);
                            const uint32_t b1 = i8pair_to_h2(w.x, w.x, 0x0302u);
                            const uint32_t b2 = i8pair_to_h2(w.y, w.y, 0x0100u);
                            const uint32_t b3 = i8pair_to_h2(w.y, w.y, 0x0302u);
                            mma_16816(cb[j], qa[2 * b][0], 0u, qa[2 * b][1], 0u, b0, b1);
                            mma_16816(cb[j], qa[2 * b + 1][0], 0u, qa[2 * b + 1][1], 0u, b2, b3);
                        }
#pragma unroll
                        for (int j = 0; j < 2; ++j)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int c = 8 * j + 2 * tq + e;
                                const __half dk = reinterpret_cast<const __half*>(ks + c * G::kSclK)[b];
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
                        x[j][e] = ((mask >> c) & 1u) ? sacc[j][e] * p.scale_log2 : -INFINITY;
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
                        ldsm_x4_trans(vb + ((lane & 7) + 8 * (lane >> 4)) * G::kRowV +
                                          (16 * mt + 8 * ((lane >> 3) & 1)) * 2,
                                      a0, a1, a2, a3);
                        mma_16816(oacc[mt], a0, a1, a2, a3, pb[0], pb[1]);
                    }
                } else {
                    l_run = l_run * alpha + (pf[0][0] + pf[0][1] + pf[1][0] + pf[1][1]);
                    const unsigned char* vs = stage + ST::kVsOff + warp * kWarpCells * G::kSclV;
                    const __half* dv0 = reinterpret_cast<const __half*>(vs + (2 * tq) * G::kSclV);
                    const __half* dv1 = reinterpret_cast<const __half*>(vs + (2 * tq + 1) * G::kSclV);
                    const __half* dv2 = reinterpret_cast<const __half*>(vs + (2 * tq + 8) * G::kSclV);
                    const __half* dv3 = reinterpret_cast<const __half*>(vs + (2 * tq + 9) * G::kSclV);
#pragma unroll
                    for (int b = 0; b < D / 32; ++b) {
                        const uint32_t pb0 = pack_half2(pf[0][0] * __half2float(dv0[b]),
                                                        pf[0][1] * __half2float(dv1[b]));
                        const uint32_t pb1 = pack_half2(pf[1][0] * __half2float(dv2[b]),
                                                        pf[1][1] * __half2float(dv3[b]));
                        const uint32_t off = 32 * b + 4 * gq;
                        const uint32_t w00 = lds32(vb + (2 * tq) * G::kRowV + off);
                        const uint32_t w01 = lds32(vb + (2 * tq + 1) * G::kRowV + off);
                        const uint32_t w10 = lds32(vb + (2 * tq + 8) * G::kRowV + off);
                        const uint32_t w11 = lds32(vb + (2 * tq + 9) * G::kRowV + off);
#pragma unroll
                        for (int hb = 0; hb < 2; ++hb) {
                            const uint32_t sel0 = ((4u + 2u * hb) << 8) | (2u * hb);
                            const uint32_t sel1 = ((5u + 2u * hb) << 8) | (2u * hb + 1u);
                            const uint32_t a0 = i8pair_to_h2(w00, w01, sel0);
                            const uint32_t a1 = i8pair_to_h2(w00, w01, sel1);
                            const uint32_t a2 = i8pair_to_h2(w10, w11, sel0);
                            const uint32_t a3 = i8pair_to_h2(w10, w11, sel1);
                            mma_16816(oacc[2 * b + hb], a0, a1, a2, a3, pb0, pb1);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&empty_bar[st]));
        }
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    }

    // ------------------------- merge the consumer warps -------------------------
    __syncthreads();
    const bool aborted = *abort_flag != 0;
    float* cm = reinterpret_cast<float*>(stages);       // [warps][8] running max (log2)
    float* cl = cm + kConsumerWarps * 8;                // [warps][8] running sum
    float* co = cl + kConsumerWarps * 8;                // [warps][8][D + 4] unnormalised O
    if (!aborted && n_tiles > 0 && warp < kConsumerWarps) {
        if (tq == 0) {
            cm[warp * 8 + gq] = m_run;
            cl[warp * 8 + gq] = l_run;
        }
        float* cw = co + warp * 8 * ST::kOStride;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            const int d0 = out_dim<KVT>(mt, 0, gq);
            const int d1 = out_dim<KVT>(mt, 1, gq);
            cw[(2 * tq) * ST::kOStride + d0] = oacc[mt][0];
            cw[(2 * tq + 1) * ST::kOStride + d0] = oacc[mt][1];
            cw[(2 * tq) * ST::kOStride + d1] = oacc[mt][2];
            cw[(2 * tq + 1) * ST::kOStride + d1] = oacc[mt][3];
        }
    }
    __syncthreads();
    if (aborted) {
        if (threadIdx.x == 0) atomicOr(p.status, KVATTN_DEVICE_WAIT_TIMEOUT);
    } else {
        const int64_t part = (int64_t)s * p.n_split + p.part_base + split_idx;
        const int H = p.n_head;
        for (int idx = threadIdx.x; idx < p.group * D; idx += kThreads) {
            const int r = idx / D;
            const int d = idx - r * D;
            const int h = g * p.group + r;
            float o = 0.f, lse = -INFINITY;
            if (n_tiles > 0) {
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cm[w * 8 + r]);
                float num = 0.f, den = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) {
                        const float mw = cm[w * 8 + r];
                        if (mw != -INFINITY) {
                            const float sc = fast_exp2(mw - M);
                            num = fmaf(sc, co[(w * 8 + r) * ST::kOStride + d], num);
                            den = fmaf(sc, cl[w * 8 + r], den);
                        }
                    }
                }
                if (den > 0.f) {
                    o = num / den;
                    lse = (M + fast_log2(den)) * 0.69314718055994530942f;
                }
            }
            p.part_o[(part * H + h) * D + d] = o;
            if (d == 0) p.part_lse[part * H + h] = lse;
        }
    }
    pdl_launch_dependents();
}

}  // namespace

int split_decode_max_smem() { return 227 * 1024; }

namespace {

template <int KVT, int D>
cudaError_t launch_typed(const SplitDecodeParams& p, dim3 grid, cudaStream_t stream, bool pdl) {
    using ST = Stage<KVT, D>;
    const int smem = kHeaderBytes + p.n_stages * ST::kBytes;
    static std::once_flag once[64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    static cudaError_t attr_err[64];
    std::call_once(once[dev & 63], [&] {
        attr_err[dev & 63] = cudaFuncSetAttribute(split_decode_kernel<KVT, D>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  split_decode_max_smem());
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, split_decode_kernel<KVT, D>, p);
}

}  // namespace

int split_decode_stage_bytes(int kv_type, int head_dim) {
    if (kv_type == KVATTN_KV_F16) return head_dim == 128 ? Stage<0, 128>::kBytes : Stage<0, 256>::kBytes;
    return head_dim == 128 ? Stage<1, 128>::kBytes : Stage<1, 256>::kBytes;
}

cudaError_t split_decode_occupancy(int kv_type, int head_dim, int n_stages, int* blocks) {
    int smem = kHeaderBytes + n_stages * split_decode_stage_bytes(kv_type, head_dim);
    const void* fn;
    if (kv_type == KVATTN_KV_F16)
        fn = head_dim == 128 ? (const void*)split_decode_kernel<0, 128> : (const void*)split_decode_kernel<0, 256>;
    else
        fn = head_dim == 128 ? (const void*)split_decode_kernel<1, 128> : (const void*)split_decode_kernel<1, 256>;
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           split_decode_max_smem());
    if (err != cudaSuccess) return err;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, fn, kThreads, smem);
}

int split_decode_header_bytes() { return kHeaderBytes; }
int split_decode_max_stages() { return kMaxStages; }
int split_decode_threads() { return kThreads; }

cudaError_t launch_split_decode(const SplitDecodeParams& p, int kv_type, int head_dim, dim3 grid,
                                cudaStream_t stream, bool pdl) {
    if (kv_type == KVATTN_KV_F16) {
        if (head_dim == 128) return launch_typed<KVATTN_KV_F16, 128>(p, grid, stream, pdl);
        return launch_typed<KVATTN_KV_F16, 256>(p, grid, stream, pdl);
    }
    if (head_dim == 128) return launch_typed<KVATTN_KV_Q8_0, 128>(p, grid, stream, pdl);
    return launch_typed<KVATTN_KV_Q8_0, 256>(p, grid, stream, pdl);
}

}  // namespace kvattn
