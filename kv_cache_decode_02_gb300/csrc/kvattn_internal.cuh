// Internal declarations and device helpers of the kvattn library (not installed).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>  // CUtensorMap (type only; the encoder is fetched through the runtime)
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kvattn.h"

namespace kvattn {

// ---------------------------------------------------------------------------------------
// Workspace layout shared by the decode entry points.
// ---------------------------------------------------------------------------------------
constexpr size_t kWsAlign = 256;
constexpr size_t kStatusBytes = 256;  // first bytes: sticky uint32 status word

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct DecodeWsLayout {
    size_t desc_off, lse_off, o_off, total;
};

// status word | descriptors | partial LSE | partial O
inline DecodeWsLayout decode_ws_layout(int n_seq, int n_head, int head_dim, int64_t n_split) {
    DecodeWsLayout L;
    size_t off = kStatusBytes;
    L.desc_off = off;
    off = align_up(off + (size_t)n_seq * (size_t)n_split * 16, kWsAlign);
    L.lse_off = off;
    off = align_up(off + (size_t)n_seq * (size_t)n_split * (size_t)n_head * 4, kWsAlign);
    L.o_off = off;
    off = align_up(off + (size_t)n_seq * (size_t)n_split * (size_t)n_head * (size_t)head_dim * 4,
                   kWsAlign);
    L.total = off;
    return L;
}

// ---------------------------------------------------------------------------------------
// Kernel parameter blocks.
// ---------------------------------------------------------------------------------------
struct SplitDecodeParams {
    CUtensorMap tmap_k;       // 3-D {row elements, KV heads, cells} views of the caches for
    CUtensorMap tmap_v;       // the TMA path (valid when use_tma != 0)
    CUtensorMap tmap_ks;      // 2-D {n_head_kv * head_dim / 32 halves, cells} views of the
    CUtensorMap tmap_vs;      // quantised caches' scales (valid when scl_tma != 0)
    const __half* q;          // [S][H][D]
    const void* k;            // [cells][Hk][D] (f16 or int8)
    const void* v;
    const __half* k_scale;    // Q8_0: [cells][Hk][D/32]
    const __half* v_scale;
    const int32_t* plan;      // nullable: [S][plan_stride]
    const int32_t* seq_lens;  // nullable: [S]; when NULL every sequence has fixed_len cells
    const int4* desc;         // nullable: [S][n_split]
    float* part_o;            // [S][n_split][H][D]
    float* part_lse;          // [S][n_split][H]
    uint32_t* status;         // sticky status word
    int64_t n_cells;
    int64_t plan_stride;
    int64_t max_len;
    int64_t n_split;          // splits per sequence (descriptor stride)
    int64_t unit_splits;      // splits per sequence in this launch: the kernel's work units are
                              // (sequence, split < unit_splits, KV head), KV head fastest
    int64_t part_stride;      // partial slots per sequence
    int64_t part_base;        // first partial index written (window + tail packs several calls)
    int64_t fixed_len;
    uint64_t wait_limit_ns;   // bound on every pipeline wait
    uint32_t stall_tx;        // test hook: extra bytes expected on the first tile (never arrive)
    int n_seq, n_head, n_head_kv, group, split;
    int n_q;                  // query tokens per sequence (multi-query decode; 1 otherwise)
    int mq;                   // 1: the multi-query kernels; 2: f16 multi-query units of up to 8
                              // rows on the single-query kernels (single-query resources); 3:
                              // the three-consumer f16 multi-query kernel; 4: the one-warp
                              // quantised head_dim-256 single-query kernels; 5: the tcgen05 kernel
    int n_rg;                 // multi-query row groups per KV head (0 or 1: one group holding
                              // every row); the units become (sequence, split, KV head, row
                              // group), row group fastest, so the groups of one split run side
                              // by side and share its K/V bytes through L2
    int rg_rows;              // query rows per row group (when n_rg > 1)
    int n_stages;
    int use_tma;              // tiles that are one physical run load through tmap_k/tmap_v
    int scl_tma;              // ... and their scale rows through tmap_ks/tmap_vs: one 16-byte
                              // box row per cell (for head_dim 128 the KV-head pair g & ~1,
                              // g | 1: the scale rows of one head are 8 bytes)
    int write_beyond;         // splits past a sequence's length still write (0, -inf)
    int src_lsu;              // K/V rows arrive by 16-byte cp.async (e.g. straight from pinned
                              // host memory) instead of the TMA engine
    int4* desc_out;           // nullable: per-split descriptors written by the f16 producer
                              // ([n_seq][n_split], as descriptor_kernel computes them)
    int no_dep_wait;          // 1: launched as a programmatic dependent of a grid whose results
                              // it does not read, and itself launched only after everything it
                              // does read was complete: skip the dependency wait (run beside it)
    int pair;                 // head-pair units (quantised head_dim-128 caches, G <= 4, an even
                              // number of KV heads): the head_dim-256 kernels read 256-byte rows
                              // of the KV-head pair 2g, 2g+1; n_head_kv and group count pairs and
                              // the pair's 2G query rows, q and the partials keep head_dim 128
    float scale_log2;         // scale * log2(e)
};

// Fill a 2-D tensor map {n_head_kv * head_dim / 32 halves, cells} over a scale plane with
// boxes of 8 halves (16 bytes) x the kernel's cells, no swizzle.  Returns false when the
// geometry does not allow it (the base not 16-byte aligned, rows not a multiple of 16
// bytes) or the encoder rejects it.
bool encode_scale_tensor_map(CUtensorMap* map, const void* base, int64_t cells, int n_head_kv, int head_dim,
                             int box_cells);
// Fill a 3-D tensor map {row elements, n_head_kv, cells} over a cell-major cache with
// boxes of the kernel's cells x 128 bytes (a whole 64- or 128-byte row for 4-bit V rows,
// v_side with KVATTN_KV_Q8_0_Q4_0) and the 128-byte swizzle; for 8-bit rows of 256 bytes
// a 4-D map {128 bytes, cells, plane, n_head_kv} whose box {128, the kernel's cells, 2, 1}
// brings both planes at once.  Returns false if the driver's encoder is unavailable or
// rejects the geometry (the caller then loads per cell).
bool encode_kv_tensor_map(CUtensorMap* map, const void* base, int kv_type, int64_t cells,
                          int n_head_kv, int head_dim, bool v_side);

struct MergeParams {
    const float* part_o;      // parts: o[(base + p) * row_stride_parts ...]
    const float* part_lse;
    float* out;
    float* lse;
    const int32_t* seq_lens;  // nullable: per-sequence part count = ceil(clamp(len)/split)
    int all_written;          // every part's O was written (0 for empty parts): read O and LSE
                              // in one round instead of gating O on the LSE
    int64_t n_parts;          // parts per sequence (fixed count when seq_lens == NULL)
    int64_t max_len;
    int64_t len_cap;          // clamp for seq_lens (n_cells or plan_stride)
    int n_seq, n_rows;        // rows per sequence (= n_head)
    int head_dim, split;
    int64_t wide_rows_max;    // decode partials of at most this many rows in all may merge with
                              // 16-warp CTAs (one per SM); 0: always 8 warps
    int allow_slices;         // decode partials of rows with many parts may spread each row's
                              // head_dim over several CTAs
};

// Launchers (return cudaError_t of the launch).
cudaError_t launch_split_decode(const SplitDecodeParams& p, int kv_type, int head_dim,
                                unsigned grid_ctas, cudaStream_t stream, bool pdl);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream, bool pdl);
// Copies `bytes` (a multiple of 16) of K and of V from device-visible (e.g. mapped pinned
// host) memory into device buffers with one kernel launch.
cudaError_t launch_tile_copy(const void* k_src, const void* v_src, void* k_dst, void* v_dst, size_t bytes,
                             cudaStream_t stream);
int split_decode_stage_bytes(int kv_type, int head_dim);
// mode: 0 single-query, 1 multi-query kernels, 3 the three-consumer multi-query kernel, 4 the
// one-warp quantised head_dim-256 single-query kernels (the multi-query units of up to 8
// rows, mode 2, use the single-query resources)
int split_decode_smem_bytes(int kv_type, int head_dim, int n_stages, int mode = 0);
int split_decode_block_threads(int kv_type, int head_dim, int mode = 0);
int split_decode_box_cells(int kv_type);
int split_decode_max_stages();
int split_decode_max_smem();
int split_decode_threads();
cudaError_t split_decode_occupancy(int kv_type, int head_dim, int n_stages, int mode, int* blocks);
cudaError_t launch_descriptors(const int32_t* plan, int64_t plan_stride, const int32_t* seq_lens,
                               int n_seq, int64_t max_len, int split, int64_t n_cells,
                               int64_t n_split, int4* desc, uint32_t* status,
                               cudaStream_t stream);

// Scratch the library owns (a file-scope device array), for callers that cannot allocate:
// its size, and a host function that yields its device address on the current device.
struct LibraryScratch {
    size_t bytes;
    cudaError_t (*address)(void** ptr);
};

// kvattn_decode with the workspace taken from `scratch` (api.cu): every argument check,
// the size check included, runs before the address lookup and before any device work; the
// status word is then cleared on the stream, because the array keeps the last call's bytes.
int decode_with_library_scratch(const void* q, const void* k_cache, const void* v_cache, const void* k_scales,
                                const void* v_scales, int kv_type, int64_t n_cells, const int32_t* cell_plan,
                                int64_t plan_stride, const int32_t* seq_lens, int n_seq, int64_t max_len,
                                int n_head, int n_head_kv, int head_dim, int split, float scale, float* out,
                                float* lse, const LibraryScratch& scratch, void* stream);

// Host plan builder (plan.cpp).
int build_cell_plan_host(const int64_t* cells, const int64_t* offsets, int n_seq,
                         int64_t capacity_cells, int32_t* plan, int64_t plan_stride,
                         int32_t* seq_lens);

// Tile geometry of the split-decode kernel.
constexpr int kConsumerWarps = 2;
constexpr int kWarpCells = 16;
constexpr int kTileCells = kConsumerWarps * kWarpCells;  // cells per pipeline stage
constexpr int kMaxGroup = 8;

// ---------------------------------------------------------------------------------------
// Device helpers: mbarrier, bulk async copies, bounded waits, tensor-core fragments.
// ---------------------------------------------------------------------------------------
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

#endif  // __CUDACC__

// Default bound on a pipeline wait (wall time).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

#if defined(__CUDACC__)

// Bounded wait on an mbarrier phase.  Gives up after `limit_ns` of wall time, or early
// when another thread of the CTA has already given up (`*abort` set).  Returns false on
// give-up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int* abort, uint64_t limit_ns) {
    if (mbar_test(bar, parity)) return true;
    uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_test(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (*abort) return false;
            if (global_ns() - t0 > limit_ns) {
                *abort = 1;
                return false;
            }
        }
    }
}

// 1-D bulk async copy global -> shared, completion counted on an mbarrier (bytes).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Small LSU async copies (8 or 16 bytes) and their mbarrier completion arrive.
__device__ __forceinline__ void cp_async_8(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_16_cg(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col)
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fast_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// int8 -> exact f16 lanes with the magic-number method of Kim et al. 2022 ("Who Says
// Elephants Can't Run"), on words whose sign bits were flipped once (w ^ 0x80808080): a
// byte u = x + 128 paired with 0x64 is the f16 1024 + u, and subtracting 1152 as f16x2
// leaves x.  _lo converts bytes 0,1 and _hi bytes 2,3.
__device__ __forceinline__ uint32_t prmt_b32(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t t;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(t) : "r"(a), "r"(b), "r"(sel));
    return t;
}
__device__ __forceinline__ uint32_t magic_bias_h2(uint32_t t) {
    uint32_t r;
    const uint32_t bias = 0x64806480u;  // (1152, 1152) in f16
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(bias));
    return r;
}
__device__ __forceinline__ uint32_t i8x2_lo(uint32_t flipped) {
    return magic_bias_h2(prmt_b32(flipped, 0x64646464u, 0x4140u));
}
__device__ __forceinline__ uint32_t i8x2_hi(uint32_t flipped) {
    return magic_bias_h2(prmt_b32(flipped, 0x64646464u, 0x4342u));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

#endif  // __CUDACC__

}  // namespace kvattn
