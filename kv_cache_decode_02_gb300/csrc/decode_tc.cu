// Causal multi-query decode (speculative verification: "Rolling-KV -- overflow throughput
// evaluations", section 3; "KVARN KV Performance optimizations", items 2 and 7) on the
// fifth-generation tensor cores: f16 cache, head_dim 128, all G x n_q query rows of a KV
// head (up to 128) in one work unit (sequence, split, KV head).
//
//  * one warp produces: 32-cell tiles of K and V into a ring of stages, each tile as two
//    128-byte-swizzled planes (dims 0-63, 64-127) of 32 rows -- four tensor-map boxes when
//    the tile's valid entries are one physical run, otherwise 16-byte cp.async copies of the
//    valid rows straight into their swizzled places.  Before a tile's P V the first row warp
//    zeros the V rows of the tile's other cells.
//  * another warp issues the MMAs (the whole warp walks the schedule and waits, one elected
//    lane issues with warp-uniform operands): S = Q K^T (M = 128 rows, N = 32 cells, K = 128
//    dims; A = Q from tensor memory, where the rows put it once per unit, B = K from shared
//    memory, K-major) into one of two 32-column TMEM buffers, and O += P V (A = P from the
//    first 16 columns of that buffer, B = V in shared memory with head_dim the contiguous
//    dimension, N = 128) into 128 columns that accumulate over the unit.  It
//    issues S of the next tile before waiting for this tile's probabilities, so the tensor
//    cores compute S(t+1) while the rows run the softmax of tile t; the commit after P V(t)
//    releases the tile's stage to the producer.
//  * warps 0-3 hold the rows: thread r owns query row r, which is TMEM lane r.  Warps whose
//    lanes hold no row of the unit take the producer's and the MMA thread's roles (on other
//    schedulers than the rows) or sit out.  Each row's online softmax is thread-local:
//    it reads its 32 scores, masks plan holes, cells past the split and its own causal
//    limit, keeps its running maximum (moved lazily, only when it grows by more than 2^8, as
//    in the mma.sync kernels) and sum, rescales its O row in TMEM on such a move (after the
//    previous P V is complete), and writes its 32 probabilities as f16 pairs over the first
//    16 columns of the tile's S.  (MMAs of one thread run in issue order: the S two tiles
//    later, written into the same columns, follows this tile's P V.)
//
// Every wait is bounded; a wait that gives up sets a flag that every other wait sees, the
// kernel reports KVATTN_DEVICE_WAIT_TIMEOUT and frees its tensor memory.
#include <climits>
#include <cmath>
#include <mutex>

#include "decode_tc.cuh"

namespace kvattn {

namespace {

constexpr int kTile = 32;                   // cells per stage
constexpr int kStages = 4;
constexpr int kWarpBuf = 8192;              // per row warp: query rows in, O rows out
constexpr int kThreads = 6 * 32;            // row warps (up to 4), a producer and an MMA warp
constexpr int kPlane = kTile * 128;         // one 128-byte-wide plane of a tile (4 KB)
constexpr int kStageBytes = 4 * kPlane;     // K planes 0, 1 then V planes 0, 1 (16 KB)
constexpr int kHeader = 1024;
constexpr int kSmem = kHeader + 1024 + kStages * kStageBytes + 4 * kWarpBuf;  // (+1024: slack to align the base)
// TMEM columns: two S buffers 0-31 and 32-63 (a tile's P is written over the first 16
// columns of its S), Q 64-127 (f16 pairs), O 128-255
constexpr uint32_t kCols = 256;
constexpr uint32_t kColS = 0, kColQ = 64, kColO = 128;
constexpr float kSlack = 8.f;               // lazy maximum, as in the mma.sync kernels
constexpr float kLn2 = 0.69314718055994530942f;

// Shared-memory matrix descriptor: start address, leading and stride byte offsets, the
// descriptor version of this architecture family, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor of kind::f16: f32 accumulator, f16 A and B, operand majors (1: the
// M/N dimension is contiguous), N and M.
constexpr uint32_t instr_desc(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kIdQK = instr_desc(128, kTile, 0, 0);
constexpr uint32_t kIdPV = instr_desc(128, 128, 0, 1);

// byte (row r, byte b) of a 128-byte-swizzled plane whose base is 1024-byte aligned
__device__ __forceinline__ uint32_t swz(int r, int b) {
    return (uint32_t)(r * 128 + ((((b >> 4) & 7) ^ (r & 7)) << 4) + (b & 15));
}

__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
                 "r"(a_tmem), "l"(b), "r"(id), "r"(acc)
                 : "memory");
}
// one lane of the (fully active) warp
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}" : "=r"(pred));
    return pred != 0;
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 consecutive 32-bit TMEM columns of the warp's 32 lanes (one per thread)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
                 "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
                 "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar,
                                        uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
        : "memory");
}

// A work unit (sequence, split, KV head), KV head fastest; units are numbered in 32 bits.
struct TcUnit {
    int s, g;
    int64_t split_idx, len, i0, i1;
    int n_tiles;
    bool write_empty;
};
__device__ __forceinline__ TcUnit tc_unit(const SplitDecodeParams& p, uint32_t u) {
    TcUnit x;
    const uint32_t hk = (uint32_t)p.n_head_kv, us = (uint32_t)p.unit_splits;
    const uint32_t r = u / hk;
    x.g = (int)(u - r * hk);
    const uint32_t si = r / us;
    x.s = (int)si;
    x.split_idx = (int64_t)(r - si * us);
    const int64_t cap = p.plan ? p.plan_stride : p.n_cells;
    int64_t L = p.seq_lens != nullptr ? (int64_t)__ldg(p.seq_lens + x.s) : p.fixed_len;
    L = L < 0 ? 0 : L;
    L = L < p.max_len ? L : p.max_len;
    L = L < cap ? L : cap;
    x.len = L;
    x.i0 = x.split_idx * p.split;
    x.i1 = (x.i0 + p.split < L) ? x.i0 + p.split : L;
    const bool empty = x.i0 >= x.i1;
    x.n_tiles = empty ? 0 : (int)((x.i1 - x.i0 + kTile - 1) / kTile);
    x.write_empty = empty && p.write_beyond;
    return x;
}

// The V rows of a tile's cells outside `mask` (plan holes, cells past the split, rows no
// copy brought) become zeros, so that their P = 0 never meets a non-finite value: 16 lanes
// a row, two rows per store; then the proxy fence that orders the stores before the P V.
__device__ __forceinline__ void zero_masked_v(unsigned char* stage, uint32_t mask, int lane) {
    unsigned char* zv = stage + 2 * kPlane;
    for (uint32_t m = ~mask; m != 0u;) {
        const int c = __ffs(m) - 1;
        const uint32_t m2 = m & (m - 1u);
        const int c2 = m2 != 0u ? __ffs(m2) - 1 : c;
        const int cz = lane < 16 ? c : c2;
        *reinterpret_cast<uint4*>(zv + ((lane >> 3) & 1) * kPlane + cz * 128 + (lane & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        m = m2 != 0u ? m2 & (m2 - 1u) : 0u;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, 2) split_decode_tc_f16_d128(const __grid_constant__ SplitDecodeParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem);  // [kStages] a tile has landed
    uint64_t* empty_bar = full_bar + kStages;                 // [kStages] its P V is done
    uint64_t* s_full = empty_bar + kStages;                   // [2] S of a tile is in TMEM
    uint64_t* p_full = s_full + 2;                            // [2] P of a tile is in TMEM
    uint64_t* q_full = p_full + 2;                            // a unit's Q rows are staged
    uint64_t* o_bar = q_full + 1;                             // a unit's last P V is done
    uint64_t* zero_bar = o_bar + 1;                           // [kStages] masked V rows zeroed
    uint32_t* tile_mask = reinterpret_cast<uint32_t*>(zero_bar + kStages);  // [kStages] valid entries
    uint32_t* tile_lsu = tile_mask + kStages;                      // [kStages] rows copied by the LSU
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tile_lsu + kStages);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tile_lsu + kStages + 1);
    unsigned char* stages = smem + kHeader;  // 1024-byte aligned
    unsigned char* qbuf = stages + kStages * kStageBytes;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int H = p.n_head, G = p.group, NQ = p.n_q;
    const int rows = G * NQ;
    const int row_warps = (rows + 31) >> 5;  // warps holding at least one row
    // Warp w reaches TMEM lanes 32 (w % 4) ..: rows 32q .. 32q + 31 belong to warp q.  The
    // producer and the MMA warp take warps no row needs, on other schedulers than the rows.
    const int prod_warp = row_warps <= 2 ? 2 : 4;
    const int mma_warp = row_warps <= 3 ? 3 : 5;
    // Through a plan with up to 64 rows a spare warp zeros the V rows of a tile's masked cells
    // (a plan hole inside a run may hold anything, and 0 x NaN is NaN on the tensor cores too)
    // before the tile's P V; otherwise -- more rows, or a contiguous cache, whose only masked
    // cells are past a sequence's end in its last tile -- the first row warp does.
    const int fix_warp = (row_warps <= 2 && p.plan != nullptr) ? 4 : -1;
    const uint32_t n_units = (uint32_t)((int64_t)p.n_seq * p.unit_splits * p.n_head_kv);

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_addr(&full_bar[i]), 64);  // 32 producer lanes + their copy completions
            mbar_init(smem_addr(&empty_bar[i]), 1);  // the MMA thread's commit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&s_full[i]), 1);
            mbar_init(smem_addr(&p_full[i]), 32 * row_warps);
        }
        mbar_init(smem_addr(q_full), 32 * row_warps);
        mbar_init(smem_addr(o_bar), 1);
        for (int i = 0; i < kStages; ++i) mbar_init(smem_addr(&zero_bar[i]), 32);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    bool bad = false;

    if (warp == prod_warp) {
        // ---------------------------------- producer ----------------------------------
        const uint64_t pol = evict_first_policy();
        const int64_t Hk = p.n_head_kv;
        uint32_t T = 0;
        bool stop = false;
        for (uint32_t u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
            const TcUnit x = tc_unit(p, u);
            // The split's descriptor (the same for every KV head) is written by its head-0 unit
            // from the plan entries read here anyway: count, smallest and largest valid cell,
            // whether every valid entry has the same (cell - position), out-of-range entries.
            const bool emit_desc = p.desc_out != nullptr && x.g == 0;
            if (x.n_tiles == 0) {
                if (emit_desc && lane == 0)
                    p.desc_out[(int64_t)x.s * p.n_split + x.split_idx] = make_int4(0, -1, -1, x.i0 >= x.len ? 9 : 1);
                continue;
            }
            int d_lo = INT_MAX, d_hi = -1, d_count = 0;
            long long d_off_lo = LLONG_MAX, d_off_hi = LLONG_MIN;
            bool d_bad = false;
            // this lane's plan entries, loaded four at a time four tiles ahead (a batch is only
            // touched once its loads are four tiles old)
            const int32_t* prow = p.plan != nullptr ? p.plan + (int64_t)x.s * p.plan_stride : nullptr;
            auto plan_entry = [&](int tt) -> int32_t {
                const int64_t i = x.i0 + (int64_t)tt * kTile + lane;
                return (prow != nullptr && tt < x.n_tiles && i < x.i1) ? __ldg(prow + i) : -1;
            };
            int32_t f0 = plan_entry(0), f1 = plan_entry(1), f2 = plan_entry(2), f3 = plan_entry(3);
            int32_t e0 = -1, e1 = -1, e2 = -1, e3 = -1;
            for (int t = 0; t < x.n_tiles; ++t, ++T) {
                if ((t & 3) == 0) {
                    e0 = f0;
                    e1 = f1;
                    e2 = f2;
                    e3 = f3;
                    f0 = plan_entry(t + 4);
                    f1 = plan_entry(t + 5);
                    f2 = plan_entry(t + 6);
                    f3 = plan_entry(t + 7);
                }
                const int32_t e = (t & 2) ? ((t & 1) ? e3 : e2) : ((t & 1) ? e1 : e0);
                const int st = (int)(T % kStages);
                const uint32_t use = T / kStages;
                if (use > 0) {
                    const bool ok = mbar_wait_bounded(smem_addr(&empty_bar[st]), (use - 1) & 1u, abort_flag,
                                                      p.wait_limit_ns);
                    if (!__all_sync(0xffffffffu, ok)) {
                        stop = true;
                        break;
                    }
                }
                const int64_t tile0 = x.i0 + (int64_t)t * kTile;
                const int64_t i = tile0 + lane;
                bool valid = i < x.i1;
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
                        cell = (int64_t)x.s * p.n_cells + i;
                    }
                }
                const uint32_t mask = __ballot_sync(0xffffffffu, valid);
                int64_t base = (int64_t)x.s * p.n_cells + tile0;
                bool run = true;
                if (p.plan != nullptr) {
                    // one physical run: the same (cell - position) in every valid lane; a 32-bit
                    // warp reduction unless some offset leaves that range
                    const long long off = (long long)(cell - i);
                    long long lo, hi;
                    if (!__any_sync(0xffffffffu, valid && (off < INT_MIN / 2 || off > INT_MAX / 2))) {
                        lo = __reduce_min_sync(0xffffffffu, valid ? (int)off : INT_MAX);
                        hi = __reduce_max_sync(0xffffffffu, valid ? (int)off : INT_MIN);
                        if (lo == INT_MAX) lo = LLONG_MAX;  // no valid lane
                        if (hi == INT_MIN) hi = LLONG_MIN;
                    } else {
                        lo = valid ? off : LLONG_MAX;
                        hi = valid ? off : LLONG_MIN;
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
                            lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
                            hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
                        }
                    }
                    run = mask != 0u && lo == hi;
                    base = lo + tile0;
                    if (emit_desc) {
                        d_off_lo = min(d_off_lo, lo);
                        d_off_hi = max(d_off_hi, hi);
                        d_count += __popc(mask);
                        if (valid) {
                            d_lo = min(d_lo, (int)cell);
                            d_hi = max(d_hi, (int)cell);
                        }
                    }
                }
                const bool use_tma = run && p.use_tma != 0 && base > INT_MIN / 2 && base < INT_MAX / 2;
                unsigned char* stage = stages + st * kStageBytes;
                const uint32_t bar = smem_addr(&full_bar[st]);
                if (lane == 0) {
                    tile_mask[st] = mask;
                    tile_lsu[st] = use_tma ? 0u : 1u;
                    mbar_expect_tx(bar, (use_tma ? (uint32_t)kStageBytes : 0u) + (T == 0 ? p.stall_tx : 0u));
                }
                __syncwarp();
                if (use_tma) {
                    if (lane == 0) {
                        const uint32_t d = smem_addr(stage);
                        tma_box(d, &p.tmap_k, 0, x.g, (int)base, bar, pol);
                        tma_box(d + kPlane, &p.tmap_k, 64, x.g, (int)base, bar, pol);
                        tma_box(d + 2 * kPlane, &p.tmap_v, 0, x.g, (int)base, bar, pol);
                        tma_box(d + 3 * kPlane, &p.tmap_v, 64, x.g, (int)base, bar, pol);
                    }
                } else {
                    // valid rows, each by the whole warp: lane l copies bytes 16 (l % 16) .. of the
                    // row's K (l < 16) or V (l >= 16) into its swizzled place
                    const int which = lane >> 4;
                    const int off = (lane & 15) * 16;
                    const char* src0 = static_cast<const char*>(which ? p.v : p.k);
                    const uint32_t dst0 = smem_addr(stage) + (uint32_t)(which * 2 * kPlane + (off >> 7) * kPlane);
                    for (int c = 0; c < kTile; ++c) {
                        if (!((mask >> c) & 1u)) continue;
                        const int64_t cc = __shfl_sync(0xffffffffu, cell, c);
                        const int64_t row = cc * Hk + x.g;
                        cp_async_16_cg(dst0 + swz(c, off & 127), src0 + row * 256 + off);
                    }
                }
                cp_async_arrive_noinc(bar);
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
                    p.desc_out[(int64_t)x.s * p.n_split + x.split_idx] =
                        make_int4(d_count, d_count ? d_lo : -1, d_count ? d_hi : -1, flags);
                }
            }
        }
    } else if (warp == mma_warp) {
        // ------------------------------------- MMA -------------------------------------
        // The whole warp walks the schedule and waits; one elected lane issues.  Every operand
        // is the same in all lanes (the TMEM base is broadcast from lane 0).
        const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
        auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort_flag, p.wait_limit_ns));
        };
        auto issue_s = [&](uint32_t T) -> bool {
            const int st = (int)(T % kStages);
            if (!wait_all(smem_addr(&full_bar[st]), (T / kStages) & 1u)) return false;
            if (tile_lsu[st] != 0u) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // rows the LSU wrote
            tc_fence_after();
            const uint64_t kd = smem_desc(smem_addr(stages + st * kStageBytes), 16, 1024);
            const uint32_t d = tm + kColS + 32 * (T & 1u);
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < 8; ++k)  // (start address in 16-byte units in the low bits)
                    mma_ts(d, tm + kColQ + 8 * k, kd + (uint64_t)(((k >> 2) * kPlane + 32 * (k & 3)) >> 4), kIdQK,
                           k > 0 ? 1u : 0u);
                mma_commit(smem_addr(&s_full[T & 1u]));
            }
            __syncwarp();
            return true;
        };
        uint32_t T = 0, U = 0;
        bool ok = true;
        int n_next = blockIdx.x < n_units ? tc_unit(p, blockIdx.x).n_tiles : 0;
        for (uint32_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            // (the next unit's tile count loads while this one runs)
            const int n_tiles = n_next;
            n_next = u + gridDim.x < n_units ? tc_unit(p, u + gridDim.x).n_tiles : 0;
            if (n_tiles == 0) continue;
            ok = wait_all(smem_addr(q_full), U & 1u);
            ++U;
            if (!ok) break;
            tc_fence_after();
            ok = issue_s(T);
            for (int t = 0; t < n_tiles && ok; ++t, ++T) {
                if (t + 1 < n_tiles && !issue_s(T + 1)) {
                    ok = false;
                    break;
                }
                if (!wait_all(smem_addr(&p_full[T & 1u]), (T >> 1) & 1u)) {
                    ok = false;
                    break;
                }
                // a tile with masked cells waits for its zeros (the zeros warp arrives for every
                // tile, so the phase is the tile's whatever tiles were not waited for)
                if (fix_warp >= 0 && tile_mask[T % kStages] != 0xffffffffu &&
                    !wait_all(smem_addr(&zero_bar[T % kStages]), (T / kStages) & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // O += P V over the tile's 32 cells (two k-steps of 16)
                const uint64_t vd = smem_desc(smem_addr(stages + (T % kStages) * kStageBytes) + 2 * kPlane, kPlane, 1024);
                const uint32_t a = tm + kColS + 32 * (T & 1u);
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < 2; ++k)
                        mma_ts(tm + kColO, a + 8 * k, vd + (uint64_t)((2048 * k) >> 4), kIdPV, (t > 0 || k > 0) ? 1u : 0u);
                    mma_commit(smem_addr(&empty_bar[T % kStages]));
                    if (t + 1 == n_tiles) mma_commit(smem_addr(o_bar));
                }
                __syncwarp();
            }
        }
    } else if (warp == fix_warp) {
        // ------------------------------------- zeros ------------------------------------
        uint32_t T = 0;
        bool ok = true;
        for (uint32_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const int n_tiles = tc_unit(p, u).n_tiles;
            for (int t = 0; t < n_tiles; ++t, ++T) {
                const int st = (int)(T % kStages);
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&full_bar[st]), (T / kStages) & 1u,
                                                                abort_flag, p.wait_limit_ns))) {
                    ok = false;
                    break;
                }
                const uint32_t mask = tile_mask[st];
                if (mask != 0xffffffffu) zero_masked_v(stages + st * kStageBytes, mask, lane);
                mbar_arrive(smem_addr(&zero_bar[st]));
            }
        }
    } else if (warp < row_warps) {
        // ------------------------------------- rows -------------------------------------
        const int r = tid;  // query row r of the unit = TMEM lane r
        const bool row_ok = r < rows;
        const int tok = row_ok ? r / G : 0;
        const int hj = row_ok ? r % G : 0;
        const int64_t HR = (int64_t)NQ * H;
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        const uint32_t t_s = tmem + kColS + lane_base, t_q = tmem + kColQ + lane_base, t_o = tmem + kColO + lane_base;
        // This warp's 8 KB: the next unit's 32 query rows (256 bytes each, 16-byte chunk k of
        // row l at k ^ (l % 16)), then the outgoing O rows (two 32-column halves of 128 bytes a
        // row, chunk j of row l at j ^ (l % 8)); the XOR keeps eight lanes on distinct banks.
        unsigned char* wbuf = qbuf + warp * kWarpBuf;
        const uint32_t wb = smem_addr(wbuf);
        auto fetch_q = [&](const TcUnit& y) {
            if (row_ok) {
                const char* src = reinterpret_cast<const char*>(p.q + (((int64_t)y.s * NQ + tok) * H + y.g * G + hj) * 128);
#pragma unroll
                for (int k = 0; k < 16; ++k) cp_async_16_cg(wb + lane * 256 + ((k ^ (lane & 15)) << 4), src + 16 * k);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        // the fetched row into this thread's TMEM lane (64 columns of f16 pairs, the A operand
        // of S; zeros beyond the unit's rows); the MMA thread learns of it from q_full
        auto stage_q = [&]() {
            asm volatile("cp.async.wait_all;" ::: "memory");
            uint32_t v[2][32];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const uint4 w = row_ok ? *reinterpret_cast<const uint4*>(wbuf + lane * 256 + ((k ^ (lane & 15)) << 4))
                                       : make_uint4(0u, 0u, 0u, 0u);
                v[k >> 3][4 * (k & 7)] = w.x;
                v[k >> 3][4 * (k & 7) + 1] = w.y;
                v[k >> 3][4 * (k & 7) + 2] = w.z;
                v[k >> 3][4 * (k & 7) + 3] = w.w;
            }
            tmem_st32(t_q, v[0]);
            tmem_st32(t_q + 32, v[1]);
            tc_wait_st();
            tc_fence_before();
            mbar_arrive(smem_addr(q_full));
            __syncwarp();  // every row read before the buffer is written again
        };
        auto no_unit = []() {
            TcUnit z = {};
            z.n_tiles = 0;
            z.write_empty = false;
            return z;
        };
        uint32_t T = 0, U = 0;
        bool ok = true;
        bool fetched = false, staged = false;  // the Q rows of unit x are in the buffer / in TMEM
        uint32_t u = blockIdx.x;
        TcUnit x = u < n_units ? tc_unit(p, u) : no_unit();
        while (u < n_units && ok) {
            // the next unit's lengths load while this one runs
            const uint32_t un = u + gridDim.x;
            const TcUnit xn = un < n_units ? tc_unit(p, un) : no_unit();
            const int64_t part = (int64_t)x.s * p.part_stride + p.part_base + x.split_idx;
            const int64_t prow = part * HR + (int64_t)tok * H + x.g * G + hj;  // this row's partial
            if (x.n_tiles == 0) {
                if (x.write_empty && row_ok) {
                    float4* o = reinterpret_cast<float4*>(p.part_o + prow * 128);
                    for (int k = 0; k < 32; ++k) o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                    p.part_lse[prow] = -INFINITY;
                }
                x = xn;
                u = un;
                continue;
            }
            if (!staged) {
                if (!fetched) fetch_q(x);
                stage_q();
            }
            fetched = staged = false;
            if (xn.n_tiles > 0) {  // the next unit's rows travel during this unit's tiles
                fetch_q(xn);
                fetched = true;
            }
            // causal limit of this row (logical position, exclusive)
            const int64_t lim = x.len - NQ + 1 + tok;
            float m_run = -INFINITY, l_run = 0.f;
            for (int t = 0; t < x.n_tiles; ++t, ++T) {
                const bool got = mbar_wait_bounded(smem_addr(&s_full[T & 1u]), (T >> 1) & 1u, abort_flag, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // (this wait has completed: it orders the producer's mask write before the read)
                const bool landed = mbar_wait_bounded(smem_addr(&full_bar[T % kStages]), (T / kStages) & 1u, abort_flag,
                                                      p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, landed)) {
                    ok = false;
                    break;
                }
                const uint32_t mask = tile_mask[T % kStages];
                if (mask != 0xffffffffu && warp == 0 && fix_warp < 0)
                    zero_masked_v(stages + (T % kStages) * kStageBytes, mask, lane);
                uint32_t sv[32];
                tmem_ld32(t_s + 32 * (T & 1u), sv);
                tc_wait_ld();
                const int64_t rel = lim - (x.i0 + (int64_t)t * kTile);
                const int lim_c = rel < 0 ? 0 : (rel > kTile ? kTile : (int)rel);
                float xs[32];
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                // the cells this row sees: in the tile and before its causal limit
                const uint32_t vm = mask & (lim_c >= kTile ? 0xffffffffu : ((1u << lim_c) - 1u));
                if (vm == 0xffffffffu) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        xs[c] = __uint_as_float(sv[c]) * p.scale_log2;
                        mx[c & 3] = fmaxf(mx[c & 3], xs[c]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        xs[c] = ((vm >> c) & 1u) ? __uint_as_float(sv[c]) * p.scale_log2 : -INFINITY;
                        mx[c & 3] = fmaxf(mx[c & 3], xs[c]);
                    }
                }
                const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                const bool grow = tmax > m_run + kSlack;
                if (__any_sync(0xffffffffu, grow)) {
                    float alpha = 1.f;
                    if (grow) {
                        const float m_new = fmaxf(m_run, tmax);
                        alpha = fast_exp2(m_run - ((m_new == -INFINITY) ? 0.f : m_new));
                        m_run = m_new;
                        l_run *= alpha;
                    }
                    // this warp's rows whose maximum moved rescale their O row once the previous
                    // tile's P V is complete (t > 0 only: the first tile's P V overwrites O)
                    if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                        // (the commit after P V(t-1) released its stage)
                        const bool done = mbar_wait_bounded(smem_addr(&empty_bar[(T - 1) % kStages]), ((T - 1) / kStages) & 1u,
                                                            abort_flag, p.wait_limit_ns);
                        if (!__all_sync(0xffffffffu, done)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll 1
                        for (int c0 = 0; c0 < 128; c0 += 32) {
                            uint32_t ov[32];
                            tmem_ld32(t_o + c0, ov);
                            tc_wait_ld();
#pragma unroll
                            for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
                            tmem_st32(t_o + c0, ov);
                        }
                    }
                }
                const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
                uint32_t pw[16];
                float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float p0 = fast_exp2(xs[2 * j] - m_use), p1 = fast_exp2(xs[2 * j + 1] - m_use);
                    ps[j & 3] += p0 + p1;
                    const __half2 hv = __floats2half2_rn(p0, p1);
                    pw[j] = *reinterpret_cast<const uint32_t*>(&hv);
                }
                l_run += (ps[0] + ps[1]) + (ps[2] + ps[3]);
                tmem_st16(t_s + 32 * (T & 1u), pw);  // over S(t), read above
                tc_wait_st();
                tc_fence_before();
                mbar_arrive(smem_addr(&p_full[T & 1u]));
            }
            if (!ok) break;
            // the next unit's Q rows go in now: every S MMA of this unit is complete
            if (fetched) {
                stage_q();
                staged = true;
            }
            // O is final once the unit's last P V is done
            const bool done = mbar_wait_bounded(smem_addr(o_bar), U & 1u, abort_flag, p.wait_limit_ns);
            ++U;
            if (!__all_sync(0xffffffffu, done)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const bool have = m_run != -INFINITY && l_run > 0.f;
            const float inv = have ? 1.f / l_run : 0.f;
            // O leaves through the buffer: each thread writes its row's 64 columns, then every
            // instruction of the warp stores four whole 128-byte row segments (lane l takes rows
            // 4 i + l / 8, whose partial rows it learns once)
            long long pr[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) pr[i] = __shfl_sync(0xffffffffu, (long long)prow, 4 * i + (lane >> 3));
            const int q4 = lane & 7;
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 64) {
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    uint32_t ov[32];
                    tmem_ld32(t_o + c0 + 32 * h2, ov);
                    tc_wait_ld();
                    float4* d = reinterpret_cast<float4*>(wbuf + h2 * 4096 + lane * 128);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        d[j ^ (lane & 7)] =
                            make_float4(__uint_as_float(ov[4 * j]) * inv, __uint_as_float(ov[4 * j + 1]) * inv,
                                        __uint_as_float(ov[4 * j + 2]) * inv, __uint_as_float(ov[4 * j + 3]) * inv);
                }
                __syncwarp();
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    float4 v[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int R = 4 * i + (lane >> 3);
                        v[i] = *reinterpret_cast<const float4*>(wbuf + h2 * 4096 + R * 128 + ((q4 ^ (R & 7)) << 4));
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (32 * warp + 4 * i + (lane >> 3) < rows)
                            __stcg(reinterpret_cast<float4*>(p.part_o + pr[i] * 128 + c0 + 32 * h2 + 4 * q4), v[i]);
                }
                __syncwarp();
            }
            if (row_ok) p.part_lse[prow] = have ? (m_run + fast_log2(l_run)) * kLn2 : -INFINITY;
            // (the next unit's first P V, which overwrites O, waits for this warp's next P)
            tc_fence_before();
            x = xn;
            u = un;
        }
    }
    if (warp == prod_warp && __any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, KVATTN_DEVICE_BAD_PLAN_ENTRY);
    tc_fence_before();
    __syncthreads();
    if (*abort_flag != 0) {
        if (threadIdx.x == 0) atomicOr(p.status, KVATTN_DEVICE_WAIT_TIMEOUT);
        // an MMA or copy issued before the wait that gave up finishes long before this
        const uint64_t t0 = global_ns();
        while (global_ns() - t0 < p.wait_limit_ns / 8) {
        }
    }
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
    pdl_launch_dependents();
}

// Per device, once: the kernel's shared-memory attributes and how many of its CTAs fit on an
// SM.  Shared memory decides (the runtime's occupancy query answers one CTA for this kernel
// although two fit); two CTAs of 256 tensor-memory columns fill an SM's 512.
struct TcSetup {
    cudaError_t err;
    int blocks;
};
TcSetup tc_setup() {
    static std::once_flag once[64];
    static TcSetup done[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return TcSetup{e, 1};
    std::call_once(once[dev & 63], [&] {
        TcSetup r{cudaSuccess, 1};
        r.err = cudaFuncSetAttribute(split_decode_tc_f16_d128, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        // the whole carve-out as shared memory: two CTAs of ~100 KB per SM
        if (r.err == cudaSuccess)
            r.err = cudaFuncSetAttribute(split_decode_tc_f16_d128, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
        int per_sm = 0, reserved = 0;
        if (r.err == cudaSuccess) r.err = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (r.err == cudaSuccess) r.err = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        const int fit = per_sm / (kSmem + reserved);
        r.blocks = fit < 1 ? 1 : (fit > 2 ? 2 : fit);
        done[dev & 63] = r;
    });
    return done[dev & 63];
}

}  // namespace

cudaError_t launch_split_decode_tc(const SplitDecodeParams& p, unsigned grid_ctas, cudaStream_t stream, bool pdl) {
    const TcSetup t = tc_setup();
    if (t.err != cudaSuccess) return t.err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_ctas, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    void* args[] = {const_cast<SplitDecodeParams*>(&p)};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(split_decode_tc_f16_d128), args);
}

cudaError_t split_decode_tc_occupancy(int* blocks) {
    const TcSetup t = tc_setup();
    *blocks = t.blocks;
    return t.err;
}

}  // namespace kvattn
