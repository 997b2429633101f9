// C-ABI entry points of kvattn: host-side validation, workspace carving, launch order,
// and the window + host-tail pipeline.  No entry point allocates device memory.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <thread>

#include "decode_tc.cuh"
#include "kvattn_internal.cuh"

using namespace kvattn;

namespace {

constexpr int kMaxDevices = 64;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int env_int(const char* name, int dflt) {
    const char* v = std::getenv(name);
    if (v == nullptr || *v == 0) return dflt;
    return std::atoi(v);
}

bool use_pdl() {
    static const bool on = env_int("KVATTN_PDL", 1) != 0;
    return on;
}

// Opt-in trace of launch decisions: with KVATTN_LOG=1 (read on every call) each entry point
// that launches work prints one line on stderr.  Otherwise the library never prints.
bool log_on() { return env_int("KVATTN_LOG", 0) != 0; }

void log_line(const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    std::fprintf(stderr, "kvattn: %s\n", buf);
}

int sm_count() {
    static std::once_flag once[kMaxDevices];
    static int count[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::call_once(once[dev % kMaxDevices], [&] {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        count[dev % kMaxDevices] = n > 0 ? n : 1;
    });
    return count[dev % kMaxDevices];
}

// Resident CTAs per SM of the split-decode kernel for (kv_type, head_dim, n_stages,
// multi-query kernel).
// mode: the launch's resources (0 single-query, 1 multi-query kernels, 3 the three-consumer
// multi-query kernel).
int occupancy(int kv_type, int head_dim, int n_stages, int mode = 0) {
    static std::mutex mu;
    static int cache[kMaxDevices][4][2][5][16];
    static bool have[kMaxDevices][4][2][5][16];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    const int d = dev % kMaxDevices, t = kv_type, h = head_dim == 256 ? 1 : 0, m = mode < 0 || mode > 4 ? 0 : mode;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[d][t][h][m][n_stages]) {
        int blocks = 0;
        if (split_decode_occupancy(kv_type, head_dim, n_stages, mode, &blocks) != cudaSuccess) blocks = 0;
        cache[d][t][h][m][n_stages] = blocks;
        have[d][t][h][m][n_stages] = true;
    }
    return cache[d][t][h][m][n_stages];
}

// Pipeline depth per CTA ("launch bounds and occupancy-aware selection", KVARN item 6).
// The kernel is persistent, so the aim is the most resident CTAs the register budget allows
// (up to the number of work units), then the deepest ring (at most 4 stages) that keeps that
// many resident.  Deeper rings measured slower on GB300 for the multi-wave Q8_0 and plan
// workloads (111 vs 91 us at 8 vs 4 stages for Q8_0 over 131072 cells).
int pick_stages(int kv_type, int head_dim, int64_t n_units, int mq = 0) {
    const int forced = env_int("KVATTN_STAGES", 0);
    const int max_st = split_decode_max_stages();
    const int limit = split_decode_max_smem();
    if (forced >= 2 && forced <= max_st && split_decode_smem_bytes(kv_type, head_dim, forced, mq) <= limit)
        return forced;
    const int64_t n_sm = sm_count();
    const int64_t want = std::min(n_units, (int64_t)occupancy(kv_type, head_dim, 2, mq) * n_sm);
    for (int st = 4; st >= 3; --st) {
        if (split_decode_smem_bytes(kv_type, head_dim, st, mq) > limit) continue;
        if ((int64_t)occupancy(kv_type, head_dim, st, mq) * n_sm >= want) return st;
    }
    return 2;
}

// Split selection ("split-size auto-selector" re-measured on GB300): the smallest power of
// two >= 64 whose work units (sequences x splits x KV heads) fit in one wave of resident
// CTAs.  On the Qwen3-8B-shaped decode (32/8 heads, head_dim 128) that choice was the
// fastest of splits 64-4096 at 1 and 4 sequences of 1K-256K cells (e.g. 16K cells: split
// 256, 14.9 us against 18.7 us at 128; 64K cells: split 1024, 44.5 us against 48.4 us at 256).
constexpr int64_t kMinAutoSplit = 64;
constexpr int64_t kMaxAutoSplit = int64_t(1) << 30;

int64_t auto_split_slots(int kv_type, int head_dim) {
    const int st = kv_type == KVATTN_KV_F16 ? 3 : 2;  // the one-wave f16 ring; quantised geometry is fixed
    return (int64_t)std::max(occupancy(kv_type, head_dim, st), 1) * sm_count();
}

// Launches the persistent split-decode kernel over n_seq x unit_splits x n_head_kv work
// units: one CTA per unit, at most as many CTAs as fit on the device at once.
cudaError_t launch_decode_units(SplitDecodeParams p, int kv_type, int head_dim, int64_t unit_splits,
                                cudaStream_t stream, bool pdl) {
    p.unit_splits = unit_splits;
    const int64_t n_units = (int64_t)p.n_seq * unit_splits * p.n_head_kv * (p.n_rg > 1 ? p.n_rg : 1);
    if (n_units > (int64_t)INT32_MAX) return cudaErrorInvalidValue;  // units are numbered in 32 bits
    if (p.mq == 5) {  // the tcgen05 multi-query kernel
        int blocks = 0;
        if (split_decode_tc_occupancy(&blocks) != cudaSuccess) blocks = 1;
        const int64_t grid = std::min(n_units, (int64_t)std::max(blocks, 1) * sm_count());
        if (grid < 1) return cudaSuccess;
        return launch_split_decode_tc(p, (unsigned)grid, stream, pdl);
    }
    const int64_t resident =
        (int64_t)std::max(occupancy(kv_type, head_dim, p.n_stages, p.mq == 2 ? 0 : p.mq), 1) * sm_count();
    const int64_t grid = std::min(n_units, resident);
    if (grid < 1) return cudaSuccess;
    return launch_split_decode(p, kv_type, head_dim, (unsigned)grid, stream, pdl);
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? KVATTN_OK : KVATTN_ERR_CUDA; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn tensor_map_encoder() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

bool use_tma_env() {
    static const bool on = env_int("KVATTN_TMA", 1) != 0;
    return on;
}

// Tensor maps of the K and V caches for the TMA path of the split-decode kernel.
void set_kv_maps(SplitDecodeParams& p, int kv_type, int64_t cells, int n_head_kv, int head_dim) {
    p.use_tma = 0;
    p.scl_tma = 0;
    if (!use_tma_env()) return;
    if (encode_kv_tensor_map(&p.tmap_k, p.k, kv_type, cells, n_head_kv, head_dim, false) &&
        encode_kv_tensor_map(&p.tmap_v, p.v, kv_type, cells, n_head_kv, head_dim, true))
        p.use_tma = 1;
    // quantised caches: the scale rows of a one-run chunk arrive by one TMA box per plane
    // instead of one 8- or 16-byte copy per cell (KVATTN_SCL_TMA=0 keeps the per-cell copies)
    if (p.use_tma && kv_type != KVATTN_KV_F16 && env_int("KVATTN_SCL_TMA", 1) != 0 &&
        encode_scale_tensor_map(&p.tmap_ks, p.k_scale, cells, n_head_kv, head_dim, split_decode_box_cells(kv_type)) &&
        encode_scale_tensor_map(&p.tmap_vs, p.v_scale, cells, n_head_kv, head_dim, split_decode_box_cells(kv_type)))
        p.scl_tma = 1;
}

bool valid_kv_type(int kv_type) {
    return kv_type == KVATTN_KV_F16 || kv_type == KVATTN_KV_Q8_0 || kv_type == KVATTN_KV_Q8_0_Q4_0 ||
           kv_type == KVATTN_KV_Q4_0;
}

// Failure-detection test hook (host-side switch, read on every call): with
// KVATTN_DEBUG_STALL_TX=<bytes> the first tile of every split expects that many extra
// bytes that no copy delivers, so its pipeline wait runs out after KVATTN_DEBUG_WAIT_MS
// milliseconds (default 20) and the kernel reports KVATTN_DEVICE_WAIT_TIMEOUT.  All real
// copies still complete; nothing faults or hangs.
void apply_debug_hooks(SplitDecodeParams& p) {
    p.wait_limit_ns = kWaitLimitNs;
    p.stall_tx = 0;
    const int stall = env_int("KVATTN_DEBUG_STALL_TX", 0);
    if (stall > 0) {
        p.stall_tx = (uint32_t)stall;
        p.wait_limit_ns = (uint64_t)env_int("KVATTN_DEBUG_WAIT_MS", 20) * 1000000ull;
    }
}

struct DecodeShape {
    int n_seq, n_head, n_head_kv, head_dim, split;
    int64_t max_len;
};

// Shape checks shared by the decode entry points.
int check_shape(const DecodeShape& s) {
    if (s.n_seq < 0 || s.n_head < 1 || s.n_head_kv < 1 || s.max_len < 0 || s.split < 1)
        return KVATTN_ERR_INVALID_ARG;
    if (s.n_head % s.n_head_kv != 0) return KVATTN_ERR_INVALID_ARG;
    if (s.n_head / s.n_head_kv > kMaxGroup) return KVATTN_ERR_UNSUPPORTED;
    if (s.head_dim != 128 && s.head_dim != 256) return KVATTN_ERR_UNSUPPORTED;
    if (s.split % kTileCells != 0) return KVATTN_ERR_UNSUPPORTED;
    // merge rows (sequence, head) are numbered in 32 bits
    if ((int64_t)s.n_seq * s.n_head > (int64_t)INT32_MAX) return KVATTN_ERR_UNSUPPORTED;
    // work units (sequence, split, KV head) are numbered in 32 bits on the device
    if ((s.max_len + s.split - 1) / s.split * s.n_head_kv * std::max(s.n_seq, 1) > (int64_t)INT32_MAX)
        return KVATTN_ERR_UNSUPPORTED;
    return KVATTN_OK;
}

}  // namespace

bool kvattn::encode_scale_tensor_map(CUtensorMap* map, const void* base, int64_t cells, int n_head_kv,
                                     int head_dim, int box_cells) {
    EncodeTiledFn enc = tensor_map_encoder();
    const cuuint64_t row_halves = (cuuint64_t)n_head_kv * (cuuint64_t)(head_dim / 32);
    if (enc == nullptr || base == nullptr || cells < 1 || !aligned(base, 16) || (row_halves * 2) % 16 != 0)
        return false;
    const cuuint64_t dims[2] = {row_halves, (cuuint64_t)cells};
    const cuuint64_t strides[1] = {row_halves * 2};
    const cuuint32_t box[2] = {8u, (cuuint32_t)box_cells};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool kvattn::encode_kv_tensor_map(CUtensorMap* map, const void* base, int kv_type, int64_t cells,
                                  int n_head_kv, int head_dim, bool v_side) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (enc == nullptr || base == nullptr || cells < 1 || !aligned(base, 16)) return false;
    const bool f16 = kv_type == KVATTN_KV_F16;
    const bool q4 = kv_type == KVATTN_KV_Q4_0 || (v_side && kv_type == KVATTN_KV_Q8_0_Q4_0);  // 4-bit rows
    const cuuint64_t row_elems = q4 ? (cuuint64_t)head_dim / 2 : (cuuint64_t)head_dim;
    const cuuint64_t row_bytes = row_elems * (f16 ? 2 : 1);
    const cuuint32_t box_cells = (cuuint32_t)split_decode_box_cells(kv_type);
    if (!f16 && !q4 && row_bytes > 128 && row_bytes % 128 == 0) {
        // 8-bit rows wider than one 128-byte swizzle span (head_dim 256, KV-head pairs): 4-D
        // {128 bytes, cells, plane, KV head}, so that one box brings all the 128-byte planes
        // of the box's cells, [plane][cell][128 bytes] in shared memory as with one box per
        // plane (two TMA issues per chunk fewer: Q8_0 over 131072 cells, head_dim 256, 113.1
        // -> 109.3 us per op; head_dim 128 as KV-head pairs 64.8 -> 63.1 us)
        const cuuint64_t planes = row_bytes / 128;
        const cuuint64_t dims4[4] = {128u, (cuuint64_t)cells, planes, (cuuint64_t)n_head_kv};
        const cuuint64_t strides4[3] = {row_bytes * (cuuint64_t)n_head_kv, 128u, row_bytes};
        const cuuint32_t box4[4] = {128u, box_cells, (cuuint32_t)planes, 1u};
        const cuuint32_t estr4[4] = {1, 1, 1, 1};
        return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims4, strides4, box4, estr4,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    const cuuint64_t dims[3] = {row_elems, (cuuint64_t)n_head_kv, (cuuint64_t)cells};
    const cuuint64_t strides[2] = {row_bytes, row_bytes * (cuuint64_t)n_head_kv};
    // box: 128 bytes of a row (64 or 128 bytes for a whole 4-bit row), one head, the kernel's
    // cells; the swizzle spans the box's width (64-byte rows take the 64-byte swizzle)
    const cuuint32_t inner = f16 ? 64u : (q4 ? (cuuint32_t)row_elems : 128u);
    const cuuint32_t box[3] = {inner, 1u, box_cells};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                           const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           inner == 64u && !f16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Everything a captured window + tail graph depends on; a call with the same key replays it.
struct TailGraphKey {
    const void *q, *k_win, *v_win, *k_tail, *v_tail, *k_tail_dev, *v_tail_dev;
    int64_t n_win, n_tail, tile_cells;
    int n_head, n_head_kv, head_dim, split, tail_split;
    float scale;
    float *out, *lse;
    void* ws;
    size_t ws_bytes;
    uint32_t stall_tx;
    uint64_t wait_limit_ns;
    int pdl, device;
    bool operator==(const TailGraphKey& o) const { return std::memcmp(this, &o, sizeof(*this)) == 0; }
};

// Recorded pipelines kept per context: a model with one context for all its layers replays
// one graph per layer instead of recording a new one on every call.
constexpr int kTailGraphSlots = 64;

struct TailGraphEntry {
    TailGraphKey key;
    cudaGraphExec_t exec;
    uint64_t last_use;
};

struct kvattn_tail_ctx {
    cudaEvent_t copied[2];
    cudaEvent_t consumed[2];
    cudaEvent_t start;
    cudaEvent_t done;
    cudaEvent_t joined;
    cudaEvent_t joined2;
    cudaStream_t copy2;     // private copy stream for odd tiles (the caller's carries even ones)
    cudaStream_t cap_main;  // private streams the pipeline is recorded on
    cudaStream_t cap_fork;
    cudaStream_t cap_fork2;
    TailGraphEntry graphs[kTailGraphSlots];
    int n_graphs;
    uint64_t use_clock;
    uint32_t flags;          // KVATTN_TAIL_*
    uint64_t tiles_issued;   // staging-slot sequence carried from call to call (prefetch mode)
    bool carry_valid;        // consumed[] hold the last readers of both slots (prefetch mode)
    unsigned long long carry_capture;  // the stream capture those records belong to (0: none)
    int device;
    bool pending;
};

extern "C" {

const char* kvattn_status_string(int status) {
    switch (status) {
    case KVATTN_OK: return "KVATTN_OK";
    case KVATTN_ERR_INVALID_ARG: return "KVATTN_ERR_INVALID_ARG";
    case KVATTN_ERR_UNSUPPORTED: return "KVATTN_ERR_UNSUPPORTED";
    case KVATTN_ERR_WORKSPACE: return "KVATTN_ERR_WORKSPACE";
    case KVATTN_ERR_CAPACITY: return "KVATTN_ERR_CAPACITY";
    case KVATTN_ERR_CUDA: return "KVATTN_ERR_CUDA";
    case KVATTN_ERR_TIMEOUT: return "KVATTN_ERR_TIMEOUT";
    default: return "KVATTN_ERR_UNKNOWN";
    }
}

int kvattn_version(void) { return (1 << 16) | 0; }

int kvattn_build_cell_plan(const int64_t* cells, const int64_t* offsets, int n_seq,
                           int64_t capacity_cells, int32_t* plan, int64_t plan_stride,
                           int32_t* seq_lens) {
    return build_cell_plan_host(cells, offsets, n_seq, capacity_cells, plan, plan_stride, seq_lens);
}

int kvattn_build_descriptors(const int32_t* cell_plan, int64_t plan_stride, const int32_t* seq_lens,
                             int n_seq, int64_t max_len, int split, int64_t n_cells, int32_t* desc,
                             void* stream) {
    if (n_seq < 0 || split < 1 || max_len < 0 || n_cells < 1 || plan_stride < 1)
        return KVATTN_ERR_INVALID_ARG;
    const int64_t n_split = (max_len + split - 1) / split;
    if (n_seq == 0 || n_split == 0) return KVATTN_OK;
    if (cell_plan == nullptr || seq_lens == nullptr || desc == nullptr || !aligned(desc, 16))
        return KVATTN_ERR_INVALID_ARG;
    return cuda_status(launch_descriptors(cell_plan, plan_stride, seq_lens, n_seq, max_len, split,
                                          n_cells, n_split, reinterpret_cast<int4*>(desc), nullptr,
                                          static_cast<cudaStream_t>(stream)));
}

size_t kvattn_decode_multi_workspace_bytes(int n_seq, int n_q, int n_head, int head_dim, int64_t max_len,
                                           int split) {
    if (n_q < 1 || split < 0 || n_head < 1) return 0;
    const int64_t rows = (int64_t)n_q * n_head;
    if (rows > INT32_MAX) return 0;
    return kvattn_decode_workspace_bytes(n_seq, (int)rows, head_dim, max_len, split);
}

size_t kvattn_decode_workspace_bytes(int n_seq, int n_head, int head_dim, int64_t max_len,
                                     int split) {
    if (n_seq < 0 || n_head < 1 || head_dim < 1 || max_len < 0 || split < 0) return 0;
    if (split == 0) split = kMinAutoSplit;  // covers whichever split the call selects
    const int64_t n_split = (max_len + split - 1) / split;
    return decode_ws_layout(n_seq, n_head, head_dim, n_split).total;
}

int kvattn_select_split_for(int n_seq, int64_t max_len, int n_head_kv, int64_t resident_ctas) {
    if (n_seq < 0 || max_len < 0 || n_head_kv < 1 || resident_ctas < 1) return KVATTN_ERR_INVALID_ARG;
    int64_t split = kMinAutoSplit;
    for (;;) {
        const int64_t units = (int64_t)n_seq * ((max_len + split - 1) / split) * n_head_kv;
        if (units <= resident_ctas || split >= max_len || split >= kMaxAutoSplit) return (int)split;
        split *= 2;
    }
}

int kvattn_select_split(int kv_type, int n_seq, int64_t max_len, int n_head_kv, int head_dim) {
    if (!valid_kv_type(kv_type)) return KVATTN_ERR_INVALID_ARG;
    if (head_dim != 128 && head_dim != 256) return KVATTN_ERR_UNSUPPORTED;
    return kvattn_select_split_for(n_seq, max_len, n_head_kv, auto_split_slots(kv_type, head_dim));
}

}  // extern "C"

namespace {

// kvattn_decode and kvattn_decode_partials: split-decode into partials (the workspace's
// or the caller's), then -- for kvattn_decode -- the merge.
int decode_impl(const void* q, const void* k_cache, const void* v_cache, const void* k_scales,
                const void* v_scales, int kv_type, int64_t n_cells, const int32_t* cell_plan,
                int64_t plan_stride, const int32_t* seq_lens, int n_seq, int64_t max_len, int n_head,
                int n_head_kv, int head_dim, int split, float scale, float* out, float* lse,
                float* part_o_user, float* part_lse_user, void* ws, size_t ws_bytes, void* stream,
                int n_q = 0, const kvattn::LibraryScratch* lib_scratch = nullptr) {
    // n_q = 0: single-query decode; n_q >= 1: causal multi-query decode
    // lib_scratch: the workspace is the library's own array (ws and ws_bytes are unused)
    // One token is single-query decode (its causal window is the whole sequence, and the
    // output and partial layouts coincide): the single-query kernels, which carry one 8-row
    // output tile instead of two (four GQA-6 sequences through a plan: 139.8 -> 98.8 us).
    const bool multi = n_q > 1;
    if (!multi) n_q = 1;
    const bool merge = part_o_user == nullptr;
    // multi-query rows per KV head beyond one unit's (f16: 32 at head_dim 128, 16 at 256;
    // quantised: 16 at head_dim 128, 8 at 256) run as row groups of that size, units of their
    // own
    const int mq_rows = (n_head_kv >= 1 && n_head >= n_head_kv) ? (n_head / n_head_kv) * n_q : 0;
    // (f16 head_dim 128 in groups of 16 instead, each group a cell-split unit: 33.4 against
    // 29.3 us for 32 rows, 49.8 against 41.6 us for 64, on a 16384-cell 8-KV-head layer)
    // f16 head_dim 128 with 33 to 48 rows, when the tcgen05 kernel below does not take them
    // (KVATTN_TC=0, q not 16-byte aligned): one unit whose three consumer warps take 16 rows
    // each, so every tile is read once for all the rows instead of once per row group of 32
    // (four GQA-6 sequences through a plan verifying 8 tokens, 48 rows: 276 -> 202 us).  Four
    // consumer warps for 49 to 64 rows measured slower than two row groups (39.4 against
    // 37.9 us on a 16384-cell layer), which keep that range.
    // f16 head_dim 128 with more than 16 rows (to 128): the tcgen05 kernel, every row of a KV
    // head in one unit (rows in TMEM lanes, S and O accumulated in tensor memory).  Measured on
    // the Qwen3-8B-shaped layer (16384 cells): at split 256, 48 rows 33.5 -> 25.2 us, 64 rows
    // 38.0 -> 26.7 us, the four-sequence GQA-6 plan verifying 8 tokens (split 512) 202 -> 147
    // us.  With 17 to 32 rows it pays only when the call's units fit about one wave of its
    // CTAs (split 512 there: 32 rows 20.1 us against 21.2 us for the mma.sync kernels at
    // their best split, 256; at split 256 the tcgen05 kernel takes 22.0 us).
    const bool tc_ok = multi && kv_type == KVATTN_KV_F16 && head_dim == 128 && mq_rows > 16 &&
                       mq_rows <= kTcMaxRows && aligned(q, 16) && env_int("KVATTN_TC", 1) != 0;
    int64_t tc_slots = 1;  // its resident CTAs
    if (tc_ok) {
        int tc_blocks = 0;
        if (split_decode_tc_occupancy(&tc_blocks) != cudaSuccess) tc_blocks = 1;
        tc_slots = (int64_t)std::max(tc_blocks, 1) * sm_count();
    }
    // split 0 (kvattn_decode_multi picks it): one wave of the tcgen05 kernel's units
    const int tc_split = (tc_ok && split == 0 && merge && max_len >= 0 && n_seq >= 0 && n_head_kv >= 1)
                             ? kvattn_select_split_for(n_seq, max_len, n_head_kv, tc_slots)
                             : split;
    const bool mq_tc =
        tc_ok && (mq_rows > 32 ||
                  (tc_split > 0 && (int64_t)n_seq * ((max_len + tc_split - 1) / tc_split) * n_head_kv * 4 <= tc_slots * 5));
    const int mq_wide = (!mq_tc && multi && kv_type == KVATTN_KV_F16 && head_dim == 128 && mq_rows > 32 &&
                         mq_rows <= 48 && env_int("KVATTN_MQ_WIDE", 1) != 0)
                            ? 3
                            : 0;
    const int rg_rows = mq_tc ? kTcMaxRows : mq_wide ? 16 * mq_wide
                        : kv_type == KVATTN_KV_F16 ? (head_dim == 256 ? 16 : 32)
                                                   : (head_dim == 256 ? 8 : 16);
    const int n_rg = (multi && mq_rows > rg_rows) ? (mq_rows + rg_rows - 1) / rg_rows : 1;
    if (split == 0 && merge) {  // kvattn_decode picks the split (partials need it fixed)
        if (!valid_kv_type(kv_type)) return KVATTN_ERR_INVALID_ARG;
        if (head_dim != 128 && head_dim != 256) return KVATTN_ERR_UNSUPPORTED;
        if (n_head_kv < 1 || n_seq < 0 || max_len < 0) return KVATTN_ERR_INVALID_ARG;
        if (mq_tc) {
            // one wave of the tcgen05 kernel's units: on the Qwen3-8B-shaped layer (16384
            // cells, 8 KV heads) split 512 -- 48 rows 22.6 us, 64 rows 24.7 us, against 24.5 /
            // 27.0 us at the single-query kernels' 256
            split = tc_split;
        } else {
            split = n_rg > 1 ? kvattn_select_split_for(n_seq, max_len, n_head_kv * n_rg,
                                                       auto_split_slots(kv_type, head_dim))
                             : kvattn_select_split(kv_type, n_seq, max_len, n_head_kv, head_dim);
        }
        if (split < 0) return split;
    }
    const DecodeShape shape{n_seq, n_head, n_head_kv, head_dim, split, max_len};
    int st = check_shape(shape);
    if (st != KVATTN_OK) return st;
    if (multi && (int64_t)n_seq * n_q * n_head > (int64_t)INT32_MAX) return KVATTN_ERR_UNSUPPORTED;
    // multi-query: up to 128 query rows per KV head (16 tokens at 8 query heads per KV head),
    // any cache type, head_dim 128 or 256
    if (multi) {
        const int rows = mq_rows;
        const bool ok = valid_kv_type(kv_type) && rows <= 128 && (head_dim == 128 || head_dim == 256);
        if (!ok) return KVATTN_ERR_UNSUPPORTED;
        if ((int64_t)n_seq * ((max_len + split - 1) / split) * n_head_kv * n_rg > (int64_t)INT32_MAX)
            return KVATTN_ERR_UNSUPPORTED;
    }
    if (q == nullptr || k_cache == nullptr || v_cache == nullptr || seq_lens == nullptr ||
        (ws == nullptr && lib_scratch == nullptr))
        return KVATTN_ERR_INVALID_ARG;
    if (merge && (out == nullptr || lse == nullptr)) return KVATTN_ERR_INVALID_ARG;
    if (!merge && (part_lse_user == nullptr || !aligned(part_o_user, 16) || !aligned(part_lse_user, 4)))
        return KVATTN_ERR_INVALID_ARG;
    if (!valid_kv_type(kv_type)) return KVATTN_ERR_INVALID_ARG;
    if (kv_type != KVATTN_KV_F16 && (k_scales == nullptr || v_scales == nullptr))
        return KVATTN_ERR_INVALID_ARG;
    if (kv_type == KVATTN_KV_F16 && (k_scales != nullptr || v_scales != nullptr))
        return KVATTN_ERR_INVALID_ARG;
    if (n_cells < 1 || (cell_plan != nullptr && plan_stride < 1) || !std::isfinite(scale))
        return KVATTN_ERR_INVALID_ARG;
    if (!aligned(q, 4) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        (merge && (!aligned(out, 16) || !aligned(lse, 4))) || (lib_scratch == nullptr && !aligned(ws, kWsAlign)) ||
        (cell_plan && !aligned(cell_plan, 4)) || !aligned(seq_lens, 4))
        return KVATTN_ERR_INVALID_ARG;
    if (kv_type != KVATTN_KV_F16) {
        const size_t sa = head_dim == 128 ? 8 : 16;
        if (!aligned(k_scales, sa) || !aligned(v_scales, sa)) return KVATTN_ERR_INVALID_ARG;
    }
    const int64_t n_split = (max_len + split - 1) / split;
    const DecodeWsLayout lay = decode_ws_layout(n_seq, n_q * n_head, head_dim, n_split);
    if ((lib_scratch != nullptr ? lib_scratch->bytes : ws_bytes) < lay.total) return KVATTN_ERR_WORKSPACE;
    if (n_seq == 0) return KVATTN_OK;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (lib_scratch != nullptr) {
        // every check passed: only now the array's address, and the status word cleared (the
        // array keeps the previous call's bytes; descriptors and partials are rewritten)
        if (lib_scratch->address(&ws) != cudaSuccess || ws == nullptr) return KVATTN_ERR_CUDA;
        if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), s) != cudaSuccess) return KVATTN_ERR_CUDA;
    }
    char* wsb = static_cast<char*>(ws);
    uint32_t* status = reinterpret_cast<uint32_t*>(wsb);
    float* part_o = merge ? reinterpret_cast<float*>(wsb + lay.o_off) : part_o_user;
    float* part_lse = merge ? reinterpret_cast<float*>(wsb + lay.lse_off) : part_lse_user;
    int4* desc = nullptr;
    const bool pdl = use_pdl();
    if (n_split > 0) {
        // Per-split descriptors of a plan.  The f16 kernels compute them in their producer warp
        // from the plan entries it reads anyway (no launch on the critical path; a fully
        // masked split then costs its plan reads and no K/V load); the quantised kernels,
        // whose warps each see a part of a split, read them from a descriptor launch first
        // and skip fully masked splits before touching their plan entries.
        int4* desc_out = nullptr;
        if (cell_plan != nullptr) {
            int4* d = reinterpret_cast<int4*>(wsb + lay.desc_off);
            if (kv_type == KVATTN_KV_F16) {
                desc_out = d;
            } else {
                desc = d;
                cudaError_t e = launch_descriptors(cell_plan, plan_stride, seq_lens, n_seq, max_len,
                                                   split, n_cells, n_split, desc, status, s);
                if (e != cudaSuccess) return KVATTN_ERR_CUDA;
            }
        }
        SplitDecodeParams p = {};
        p.q = static_cast<const __half*>(q);
        p.k = k_cache;
        p.v = v_cache;
        p.k_scale = static_cast<const __half*>(k_scales);
        p.v_scale = static_cast<const __half*>(v_scales);
        p.plan = cell_plan;
        p.seq_lens = seq_lens;
        p.desc = desc;
        p.desc_out = desc_out;
        p.part_o = part_o;
        p.part_lse = part_lse;
        p.status = status;
        p.n_cells = n_cells;
        p.plan_stride = plan_stride;
        p.max_len = max_len;
        p.n_split = n_split;
        p.part_base = 0;
        p.part_stride = n_split;
        p.write_beyond = merge ? 0 : 1;  // the merge reads only splits inside each length
        p.fixed_len = 0;
        p.n_seq = n_seq;
        p.n_head = n_head;
        p.n_head_kv = n_head_kv;
        p.group = n_head / n_head_kv;
        p.split = split;
        p.n_q = n_q;
        // up to 8 query rows per KV head: the single-query kernels with per-row causal masks
        // (one 8-row output tile instead of two; the quantised head_dim-256 multi-query kernels
        // are of that form already)
        const bool mq8 = multi && mq_rows <= 8 && (kv_type == KVATTN_KV_F16 || head_dim == 128);
        p.mq = multi ? (mq_tc ? 5 : mq_wide ? mq_wide : mq8 ? 2 : 1) : 0;
        p.n_rg = n_rg;
        p.rg_rows = rg_rows;
        // Quantised head_dim-128 caches with at most four query heads per KV head and an even
        // number of KV heads run on the head_dim-256 kernels as KV-head pairs: the K/V rows of
        // heads 2g and 2g+1 are adjacent, so a pair's rows are 256-byte rows; the pair's 2G
        // query rows hold each head's query in its own half of the 256 dimensions and zeros
        // in the other, so every score is that head's q.K; P.V computes the cross halves too
        // and the partial keeps only each row's own half.  Twice the bytes per chunk for the
        // same per-chunk loop and exchange work: 29 % fewer instructions per cell and head
        // (684 -> 481 per 16 cells on Q8_0 over 131072 cells), 62.0 -> 61.8 us there and
        // 58.7 -> 55.9 us for Q4_0 (KVATTN_PAIR=0 keeps one KV head per unit).
        const bool pair = !multi && kv_type != KVATTN_KV_F16 && head_dim == 128 && n_head_kv % 2 == 0 &&
                          n_head / n_head_kv <= 4 && env_int("KVATTN_PAIR", 1) != 0;
        const int k_hd = pair ? 256 : head_dim;           // kernel geometry
        const int k_hkv = pair ? n_head_kv / 2 : n_head_kv;
        p.pair = pair ? 1 : 0;
        p.n_head_kv = k_hkv;
        p.group = (n_head / n_head_kv) * (pair ? 2 : 1);
        // Quantised head_dim-256 kernels (and KV-head pairs) whose units overflow one wave of
        // the two-warp CTAs but fit one wave of the one-warp ones: a unit per warp, eight CTAs
        // per SM, no end-of-unit exchange (KVATTN_ONE_WARP=0 keeps two warps per CTA)
        if (!multi && kv_type != KVATTN_KV_F16 && k_hd == 256 && env_int("KVATTN_ONE_WARP", 1) != 0) {
            const int64_t units = (int64_t)n_seq * n_split * k_hkv;
            const int64_t two = (int64_t)std::max(occupancy(kv_type, 256, 2, 0), 1) * sm_count();
            const int64_t one = (int64_t)std::max(occupancy(kv_type, 256, 2, 4), 1) * sm_count();
            if (units > two && units <= one) p.mq = 4;
        }
        p.n_stages = p.mq == 5 ? 4 : pick_stages(kv_type, k_hd, n_split * k_hkv * n_rg * n_seq, p.mq == 2 ? 0 : p.mq);
        p.scale_log2 = (float)((double)scale * 1.4426950408889634074);
        apply_debug_hooks(p);
        set_kv_maps(p, kv_type, cell_plan != nullptr ? n_cells : n_cells * (int64_t)n_seq, k_hkv, k_hd);
        cudaError_t e = launch_decode_units(p, kv_type, k_hd, n_split, s, pdl);
        if (e != cudaSuccess) return KVATTN_ERR_CUDA;
        if (log_on()) {
            const int64_t units = (int64_t)n_seq * n_split * k_hkv * n_rg;
            int tc_blocks = 0;
            if (p.mq == 5 && split_decode_tc_occupancy(&tc_blocks) != cudaSuccess) tc_blocks = 1;
            const int64_t resident =
                (int64_t)std::max(p.mq == 5 ? tc_blocks : occupancy(kv_type, k_hd, p.n_stages, p.mq == 2 ? 0 : p.mq), 1) *
                sm_count();
            log_line("%s kv_type=%d n_seq=%d n_q=%d n_head=%d/%d head_dim=%d max_len=%lld split=%d n_split=%lld "
                     "plan=%d descriptors=%s units=%lld grid=%lld stages=%d tma=%d scale_tma=%d head_pairs=%d merge=%d "
                     "mode=%d",
                     multi ? "decode_multi" : (merge ? "decode" : "decode_partials"), kv_type, n_seq, n_q, n_head,
                     n_head_kv, head_dim, (long long)max_len, split, (long long)n_split, cell_plan != nullptr,
                     cell_plan == nullptr ? "none" : (desc_out != nullptr ? "in-kernel" : "kernel"),
                     (long long)units, (long long)std::min(units, resident), p.n_stages, p.use_tma, p.scl_tma, p.pair,
                     merge ? 1 : 0, p.mq);
        }
    }
    if (!merge) return KVATTN_OK;
    MergeParams m = {};
    m.part_o = part_o;
    m.part_lse = part_lse;
    m.out = out;
    m.lse = lse;
    m.seq_lens = seq_lens;
    m.n_parts = n_split;
    m.max_len = max_len;
    m.len_cap = cell_plan != nullptr ? plan_stride : n_cells;
    m.n_seq = n_seq;
    m.n_rows = n_q * n_head;  // rows (token t, head h) = t * n_head + h
    m.head_dim = head_dim;
    m.split = split;
    m.all_written = 1;
    m.allow_slices = env_int("KVATTN_MERGE_SLICES", 1) != 0;
    m.wide_rows_max = sm_count();
    return cuda_status(launch_merge(m, s, pdl && n_split > 0));
}

}  // namespace

extern "C" {

int kvattn_decode(const void* q, const void* k_cache, const void* v_cache, const void* k_scales,
                  const void* v_scales, int kv_type, int64_t n_cells, const int32_t* cell_plan,
                  int64_t plan_stride, const int32_t* seq_lens, int n_seq, int64_t max_len,
                  int n_head, int n_head_kv, int head_dim, int split, float scale, float* out,
                  float* lse, void* ws, size_t ws_bytes, void* stream) {
    if (out == nullptr || lse == nullptr) return KVATTN_ERR_INVALID_ARG;
    return decode_impl(q, k_cache, v_cache, k_scales, v_scales, kv_type, n_cells, cell_plan,
                       plan_stride, seq_lens, n_seq, max_len, n_head, n_head_kv, head_dim, split,
                       scale, out, lse, nullptr, nullptr, ws, ws_bytes, stream);
}

int kvattn_decode_partials(const void* q, const void* k_cache, const void* v_cache,
                           const void* k_scales, const void* v_scales, int kv_type,
                           int64_t n_cells, const int32_t* cell_plan, int64_t plan_stride,
                           const int32_t* seq_lens, int n_seq, int64_t max_len, int n_head,
                           int n_head_kv, int head_dim, int split, float scale, float* part_o,
                           float* part_lse, void* ws, size_t ws_bytes, void* stream) {
    if (part_o == nullptr || part_lse == nullptr) return KVATTN_ERR_INVALID_ARG;
    return decode_impl(q, k_cache, v_cache, k_scales, v_scales, kv_type, n_cells, cell_plan,
                       plan_stride, seq_lens, n_seq, max_len, n_head, n_head_kv, head_dim, split,
                       scale, nullptr, nullptr, part_o, part_lse, ws, ws_bytes, stream);
}

int kvattn_decode_multi(const void* q, const void* k_cache, const void* v_cache, const void* k_scales,
                        const void* v_scales, int kv_type, int64_t n_cells, const int32_t* cell_plan,
                        int64_t plan_stride, const int32_t* seq_lens, int n_seq, int64_t max_len, int n_q, int n_head,
                        int n_head_kv, int head_dim, int split, float scale, float* out, float* lse, void* ws,
                        size_t ws_bytes, void* stream) {
    if (n_q < 1) return KVATTN_ERR_INVALID_ARG;
    return decode_impl(q, k_cache, v_cache, k_scales, v_scales, kv_type, n_cells, cell_plan, plan_stride, seq_lens,
                       n_seq, max_len, n_head, n_head_kv, head_dim, split, scale, out, lse, nullptr, nullptr, ws,
                       ws_bytes, stream, n_q);
}

}  // extern "C"

int kvattn::decode_with_library_scratch(const void* q, const void* k_cache, const void* v_cache,
                                        const void* k_scales, const void* v_scales, int kv_type, int64_t n_cells,
                                        const int32_t* cell_plan, int64_t plan_stride, const int32_t* seq_lens,
                                        int n_seq, int64_t max_len, int n_head, int n_head_kv, int head_dim,
                                        int split, float scale, float* out, float* lse,
                                        const LibraryScratch& scratch, void* stream) {
    if (out == nullptr || lse == nullptr) return KVATTN_ERR_INVALID_ARG;
    return decode_impl(q, k_cache, v_cache, k_scales, v_scales, kv_type, n_cells, cell_plan, plan_stride, seq_lens,
                       n_seq, max_len, n_head, n_head_kv, head_dim, split, scale, out, lse, nullptr, nullptr,
                       nullptr, 0, stream, 0, &scratch);
}

extern "C" {

int kvattn_merge(const float* partials, const float* lses, int n_parts, int n_rows, int head_dim,
                 float* out, float* lse, void* stream) {
    if (n_parts < 0 || n_rows < 0 || head_dim < 4 || head_dim % 4 != 0 || head_dim > 1024)
        return KVATTN_ERR_INVALID_ARG;
    if (n_rows == 0) return KVATTN_OK;
    if (out == nullptr || lse == nullptr || (n_parts > 0 && (partials == nullptr || lses == nullptr)))
        return KVATTN_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(lse, 4) || (partials && !aligned(partials, 16)) ||
        (lses && !aligned(lses, 4)))
        return KVATTN_ERR_INVALID_ARG;
    MergeParams m = {};
    m.part_o = partials;
    m.part_lse = lses;
    m.out = out;
    m.lse = lse;
    m.seq_lens = nullptr;
    m.n_parts = n_parts;
    m.max_len = 0;
    m.len_cap = 0;
    m.n_seq = 1;
    m.n_rows = n_rows;
    m.head_dim = head_dim;
    m.split = 1;
    return cuda_status(launch_merge(m, static_cast<cudaStream_t>(stream), false));
}

// ------------------------------- window + host tail -------------------------------

int kvattn_tail_ctx_create(kvattn_tail_ctx** ctx) {
    if (ctx == nullptr) return KVATTN_ERR_INVALID_ARG;
    *ctx = nullptr;
    kvattn_tail_ctx* c = new (std::nothrow) kvattn_tail_ctx();
    if (c == nullptr) return KVATTN_ERR_INVALID_ARG;
    cudaError_t e = cudaGetDevice(&c->device);
    cudaEvent_t* evs[8] = {&c->copied[0], &c->copied[1], &c->consumed[0], &c->consumed[1],
                           &c->start,     &c->done,      &c->joined,      &c->joined2};
    int made = 0;  // events created so far
    for (; e == cudaSuccess && made < 8; ++made) {
        e = cudaEventCreateWithFlags(evs[made], cudaEventDisableTiming);
        if (e != cudaSuccess) break;
    }
    cudaStream_t* sts[4] = {&c->copy2, &c->cap_main, &c->cap_fork, &c->cap_fork2};
    for (cudaStream_t* st : sts) *st = nullptr;
    for (cudaStream_t* st : sts)
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(st, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
        for (int i = 0; i < made; ++i) cudaEventDestroy(*evs[i]);
        for (cudaStream_t* st : sts)
            if (*st) cudaStreamDestroy(*st);
        delete c;
        return KVATTN_ERR_CUDA;
    }
    c->pending = false;
    c->n_graphs = 0;
    c->use_clock = 0;
    c->flags = 0;
    c->tiles_issued = 0;
    c->carry_valid = false;
    c->carry_capture = 0;
    *ctx = c;
    return KVATTN_OK;
}

int kvattn_tail_ctx_set_flags(kvattn_tail_ctx* ctx, uint32_t flags) {
    if (ctx == nullptr || (flags & ~(uint32_t)KVATTN_TAIL_PREFETCH) != 0u) return KVATTN_ERR_INVALID_ARG;
    ctx->flags = flags;
    return KVATTN_OK;
}

int kvattn_tail_ctx_destroy(kvattn_tail_ctx* ctx) {
    if (ctx == nullptr) return KVATTN_ERR_INVALID_ARG;
    cudaEvent_t evs[8] = {ctx->copied[0], ctx->copied[1], ctx->consumed[0], ctx->consumed[1],
                          ctx->start,     ctx->done,      ctx->joined,      ctx->joined2};
    int rc = KVATTN_OK;
    for (int i = 0; i < ctx->n_graphs; ++i)
        if (cudaGraphExecDestroy(ctx->graphs[i].exec) != cudaSuccess) rc = KVATTN_ERR_CUDA;
    for (cudaStream_t st : {ctx->copy2, ctx->cap_main, ctx->cap_fork, ctx->cap_fork2})
        if (cudaStreamDestroy(st) != cudaSuccess) rc = KVATTN_ERR_CUDA;
    for (cudaEvent_t ev : evs)
        if (cudaEventDestroy(ev) != cudaSuccess) rc = KVATTN_ERR_CUDA;
    delete ctx;
    return rc;
}

namespace {

struct TailLayout {
    size_t stage_off[2][2];  // [slot][k|v]
    DecodeWsLayout parts;    // partials of all window splits and tail tiles (n_seq = 1)
    size_t parts_base;
    int64_t n_split_win, n_tiles, splits_per_tile, n_parts;
    size_t total;
};

bool tail_layout(int n_head, int n_head_kv, int head_dim, int64_t n_win, int64_t n_tail, int split,
                 int64_t tile_cells, int tail_split, TailLayout* L) {
    if (n_head < 1 || n_head_kv < 1 || head_dim < 1 || n_win < 0 || n_tail < 0 || split < 1 ||
        tile_cells < 1 || tail_split < 1 || tile_cells % tail_split != 0)
        return false;
    const size_t tile_bytes = (size_t)tile_cells * n_head_kv * head_dim * 2;
    size_t off = kStatusBytes;
    for (int s = 0; s < 2; ++s)
        for (int kv = 0; kv < 2; ++kv) {
            L->stage_off[s][kv] = off;
            off = align_up(off + tile_bytes, kWsAlign);
        }
    L->n_split_win = (n_win + split - 1) / split;
    L->n_tiles = (n_tail + tile_cells - 1) / tile_cells;
    L->splits_per_tile = tile_cells / tail_split;
    L->n_parts = L->n_split_win + L->n_tiles * L->splits_per_tile;
    L->parts = decode_ws_layout(1, n_head, head_dim, L->n_parts);
    L->parts_base = off;
    L->total = off + L->parts.total;
    return true;
}

int fault_tile() {
    // KVATTN_FAULT=copy@<t>: pretend the host-to-device copy of tail tile t failed
    // (host-side fault injection for tests; no GPU fault is involved).
    const char* v = std::getenv("KVATTN_FAULT");
    if (v == nullptr || std::strncmp(v, "copy@", 5) != 0) return -1;
    return std::atoi(v + 5);
}

}  // namespace

}  // extern "C"

namespace {

bool use_tail_graph() {
    static const bool on = env_int("KVATTN_TAIL_GRAPH", 1) != 0;
    return on;
}

// Tail tiles move by a copy kernel reading mapped pinned memory (default) or by
// cudaMemcpyAsync on the copy engine (KVATTN_TAIL_COPY=0, and whenever the host buffers are
// not mapped into the device's address space).
bool use_copy_kernel() { return env_int("KVATTN_TAIL_COPY", 1) != 0; }

// Kernel parameters of one window + tail call, fixed before any enqueue or capture.
struct TailPlan {
    TailLayout L;
    SplitDecodeParams base;     // common fields
    SplitDecodeParams window;   // the resident window
    SplitDecodeParams slot[2];  // the two staging slots (tensor maps over tile_cells rows)
    MergeParams merge;
    size_t row_bytes;
    char* wsb;
    bool pdl;
};

void prepare_window_tail(TailPlan& t, const void* q, const void* k_win, const void* v_win, int64_t n_win,
                         int64_t n_tail, int64_t tile_cells, int n_head, int n_head_kv, int head_dim, int split,
                         int tail_split, float scale, float* out, float* lse, void* ws, const TailLayout& L) {
    t.L = L;
    t.wsb = static_cast<char*>(ws);
    t.pdl = use_pdl();
    t.row_bytes = (size_t)n_head_kv * head_dim * 2;
    char* parts = t.wsb + L.parts_base;
    SplitDecodeParams& p = t.base;
    p = SplitDecodeParams{};
    p.q = static_cast<const __half*>(q);
    p.part_o = reinterpret_cast<float*>(parts + L.parts.o_off);
    p.part_lse = reinterpret_cast<float*>(parts + L.parts.lse_off);
    p.status = reinterpret_cast<uint32_t*>(t.wsb);
    p.n_split = L.n_parts;
    p.part_stride = L.n_parts;
    p.write_beyond = 1;  // the final merge reads every part slot
    p.n_seq = 1;
    p.n_head = n_head;
    p.n_head_kv = n_head_kv;
    p.group = n_head / n_head_kv;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634074);
    apply_debug_hooks(p);
    t.window = p;
    if (L.n_split_win > 0) {
        SplitDecodeParams& w = t.window;
        w.k = k_win;
        w.v = v_win;
        w.n_cells = n_win;
        w.max_len = n_win;
        w.fixed_len = n_win;
        w.split = split;
        w.part_base = 0;
        w.n_stages = pick_stages(KVATTN_KV_F16, head_dim, (int64_t)L.n_split_win * n_head_kv);
        set_kv_maps(w, KVATTN_KV_F16, n_win, n_head_kv, head_dim);
    }
    const int tile_stages = pick_stages(KVATTN_KV_F16, head_dim, L.splits_per_tile * n_head_kv);
    for (int sl = 0; sl < 2; ++sl) {
        SplitDecodeParams& tp = t.slot[sl];
        tp = p;
        tp.k = t.wsb + L.stage_off[sl][0];
        tp.v = t.wsb + L.stage_off[sl][1];
        tp.max_len = tile_cells;
        tp.split = tail_split;
        tp.n_stages = tile_stages;
        set_kv_maps(tp, KVATTN_KV_F16, tile_cells, n_head_kv, head_dim);
    }
    MergeParams& m = t.merge;
    m = MergeParams{};
    m.part_o = p.part_o;
    m.part_lse = p.part_lse;
    m.out = out;
    m.lse = lse;
    m.seq_lens = nullptr;
    m.n_parts = L.n_parts;
    m.n_seq = 1;
    m.n_rows = n_head;
    m.head_dim = head_dim;
    m.split = 1;
    m.all_written = 1;
    m.allow_slices = env_int("KVATTN_MERGE_SLICES", 1) != 0;
    m.wide_rows_max = sm_count();
    (void)n_tail;
}

// Enqueue the window decode, the double-buffered tile pipeline and the final merge.
//
// carry = false: every copy is ordered after all work enqueued before the call on the
// compute stream (so no staging slot is overwritten while an earlier call still reads it),
// and tile i goes to slot i % 2.
// carry = true (prefetch mode): copies are ordered only after earlier work on the copy
// stream and after the decode that last read their slot -- possibly one of an earlier call,
// whose consumed[] record is the newest -- and the slot sequence continues from the earlier
// call (first tile -> slot slot0).  The next layer's tiles then cross the link while this
// layer's window, tiles and merge still run on the compute stream.
int enqueue_window_tail(kvattn_tail_ctx* ctx, const TailPlan& t, const void* k_tail_host, const void* v_tail_host,
                        const void* k_tail_dev, const void* v_tail_dev, int64_t n_tail, int64_t tile_cells,
                        cudaStream_t cs, cudaStream_t xs, cudaStream_t xs2, int fault, bool prefetch = false,
                        bool carry = false, int slot0 = 0, bool capturing = false) {
    const TailLayout& L = t.L;
    const int head_dim = t.merge.head_dim;
    const int n_head_kv = t.base.n_head_kv;
    if (!carry) {
        // The copy stream may not overwrite a staging slot that an earlier call's tile decode
        // on the compute stream still reads.
        if (cudaEventRecord(ctx->start, cs) != cudaSuccess) return KVATTN_ERR_CUDA;
        if (cudaStreamWaitEvent(xs, ctx->start, 0) != cudaSuccess) return KVATTN_ERR_CUDA;
        if (cudaStreamWaitEvent(xs2, ctx->start, 0) != cudaSuccess) return KVATTN_ERR_CUDA;
        if (prefetch) {
            // Start the carried slot sequence: a slot this call leaves unused must still be
            // guarded for the next call by a record that follows every earlier reader (a
            // replayed graph's readers never record the context's events, and a record made
            // before a stream capture cannot be waited on inside it).
            if (cudaEventRecord(ctx->consumed[0], cs) != cudaSuccess) return KVATTN_ERR_CUDA;
            if (cudaEventRecord(ctx->consumed[1], cs) != cudaSuccess) return KVATTN_ERR_CUDA;
        }
    } else if (L.n_tiles > 0) {
        // the context's copy stream follows the caller's: whatever the caller ordered before
        // the call on copy_stream (a write into the tail, say) precedes every copy
        if (cudaEventRecord(ctx->start, xs) != cudaSuccess) return KVATTN_ERR_CUDA;
        if (cudaStreamWaitEvent(xs2, ctx->start, 0) != cudaSuccess) return KVATTN_ERR_CUDA;
    }
    // window: resident cells, attended while the first tail tiles are in flight
    if (L.n_split_win > 0) {
        if (launch_decode_units(t.window, KVATTN_KV_F16, head_dim, L.n_split_win, cs, t.pdl) != cudaSuccess)
            return KVATTN_ERR_CUDA;
    }
    // tail: tile i -> staging slot i % 2, copied on copy stream i % 2 (so one tile's copy
    // ramps up while the previous one drains), decoded on the compute stream
    SplitDecodeParams slot[2] = {t.slot[0], t.slot[1]};
    for (int64_t i = 0; i < L.n_tiles; ++i) {
        const int sl = (int)((i + slot0) & 1);
        cudaStream_t xsi = sl ? xs2 : xs;
        const int64_t c0 = i * tile_cells;
        const int64_t len = (c0 + tile_cells <= n_tail) ? tile_cells : n_tail - c0;
        const size_t bytes = (size_t)len * t.row_bytes;
        if ((i >= 2 || carry) && cudaStreamWaitEvent(xsi, ctx->consumed[sl], 0) != cudaSuccess)
            return KVATTN_ERR_CUDA;
        if (i == fault) return KVATTN_ERR_CUDA;
        if (k_tail_dev != nullptr) {
            if (launch_tile_copy(static_cast<const char*>(k_tail_dev) + (size_t)c0 * t.row_bytes,
                                 static_cast<const char*>(v_tail_dev) + (size_t)c0 * t.row_bytes,
                                 const_cast<void*>(slot[sl].k), const_cast<void*>(slot[sl].v), bytes,
                                 xsi) != cudaSuccess)
                return KVATTN_ERR_CUDA;
        } else {
            if (cudaMemcpyAsync(const_cast<void*>(slot[sl].k),
                                static_cast<const char*>(k_tail_host) + (size_t)c0 * t.row_bytes, bytes,
                                cudaMemcpyHostToDevice, xsi) != cudaSuccess)
                return KVATTN_ERR_CUDA;
            if (cudaMemcpyAsync(const_cast<void*>(slot[sl].v),
                                static_cast<const char*>(v_tail_host) + (size_t)c0 * t.row_bytes, bytes,
                                cudaMemcpyHostToDevice, xsi) != cudaSuccess)
                return KVATTN_ERR_CUDA;
        }
        if (cudaEventRecord(ctx->copied[sl], xsi) != cudaSuccess) return KVATTN_ERR_CUDA;
        if (cudaStreamWaitEvent(cs, ctx->copied[sl], 0) != cudaSuccess) return KVATTN_ERR_CUDA;
        SplitDecodeParams& tp = slot[sl];
        tp.n_cells = len;
        tp.fixed_len = len;
        tp.part_base = L.n_split_win + i * L.splits_per_tile;
        if (launch_decode_units(tp, KVATTN_KV_F16, head_dim, L.splits_per_tile, cs, false) != cudaSuccess)
            return KVATTN_ERR_CUDA;
        if (cudaEventRecord(ctx->consumed[sl], cs) != cudaSuccess) return KVATTN_ERR_CUDA;
    }
    if (!carry || capturing) {
        // join both copy streams back into the compute stream (a recorded graph must end
        // on the stream it began on; otherwise, with carry, the compute stream already
        // waited for every copy of this call through copied[])
        if (cudaEventRecord(ctx->joined, xs) != cudaSuccess) return KVATTN_ERR_CUDA;
        if (cudaEventRecord(ctx->joined2, xs2) != cudaSuccess) return KVATTN_ERR_CUDA;
        if (cudaStreamWaitEvent(cs, ctx->joined, 0) != cudaSuccess) return KVATTN_ERR_CUDA;
        if (cudaStreamWaitEvent(cs, ctx->joined2, 0) != cudaSuccess) return KVATTN_ERR_CUDA;
    }
    if (launch_merge(t.merge, cs, t.pdl) != cudaSuccess) return KVATTN_ERR_CUDA;
    return KVATTN_OK;
}

}  // namespace

extern "C" {

size_t kvattn_window_tail_workspace_bytes(int n_head, int n_head_kv, int head_dim, int64_t n_win,
                                          int64_t n_tail, int split, int64_t tile_cells,
                                          int tail_split) {
    TailLayout L;
    if (!tail_layout(n_head, n_head_kv, head_dim, n_win, n_tail, split, tile_cells, tail_split, &L))
        return 0;
    return L.total;
}

int kvattn_decode_window_tail(kvattn_tail_ctx* ctx, const void* q, const void* k_win,
                              const void* v_win, int64_t n_win, const void* k_tail_host,
                              const void* v_tail_host, int64_t n_tail, int64_t tile_cells,
                              int n_head, int n_head_kv, int head_dim, int split, int tail_split,
                              float scale, float* out, float* lse, void* ws, size_t ws_bytes,
                              void* compute_stream, void* copy_stream) {
    if (ctx == nullptr || q == nullptr || out == nullptr || lse == nullptr || ws == nullptr)
        return KVATTN_ERR_INVALID_ARG;
    const DecodeShape sw{1, n_head, n_head_kv, head_dim, split, n_win};
    int st = check_shape(sw);
    if (st != KVATTN_OK) return st;
    const DecodeShape stl{1, n_head, n_head_kv, head_dim, tail_split, tile_cells};
    st = check_shape(stl);
    if (st != KVATTN_OK) return st;
    if (n_win < 0 || n_tail < 0 || tile_cells < 1 || tile_cells % tail_split != 0 ||
        !std::isfinite(scale) || compute_stream == copy_stream)
        return KVATTN_ERR_INVALID_ARG;
    if ((n_win > 0 && (k_win == nullptr || v_win == nullptr)) ||
        (n_tail > 0 && (k_tail_host == nullptr || v_tail_host == nullptr)))
        return KVATTN_ERR_INVALID_ARG;
    if (!aligned(q, 4) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(ws, kWsAlign) ||
        (k_win && !aligned(k_win, 16)) || (v_win && !aligned(v_win, 16)))
        return KVATTN_ERR_INVALID_ARG;
    TailLayout L;
    if (!tail_layout(n_head, n_head_kv, head_dim, n_win, n_tail, split, tile_cells, tail_split, &L))
        return KVATTN_ERR_INVALID_ARG;
    if (ws_bytes < L.total) return KVATTN_ERR_WORKSPACE;

    cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
    cudaStream_t xs = static_cast<cudaStream_t>(copy_stream);
    TailPlan plan;
    prepare_window_tail(plan, q, k_win, v_win, n_win, n_tail, tile_cells, n_head, n_head_kv, head_dim, split,
                        tail_split, scale, out, lse, ws, L);
    const int fault = fault_tile();
    // device view of the pinned tail (copy kernel), when the buffers are mapped and aligned
    const void* k_dev = nullptr;
    const void* v_dev = nullptr;
    if (n_tail > 0 && use_copy_kernel() && aligned(k_tail_host, 16) && aligned(v_tail_host, 16) &&
        ((size_t)tile_cells * plan.row_bytes) % 16 == 0) {
        void* dk = nullptr;
        void* dv = nullptr;
        if (cudaHostGetDevicePointer(&dk, const_cast<void*>(k_tail_host), 0) == cudaSuccess &&
            cudaHostGetDevicePointer(&dv, const_cast<void*>(v_tail_host), 0) == cudaSuccess) {
            k_dev = dk;
            v_dev = dv;
        } else {
            cudaGetLastError();  // not mapped: clear the query's error, copy on the copy engine
        }
    }
    // Pageable (unregistered) tail memory still works through cudaMemcpyAsync, which then
    // stages it through the driver, but such copies cannot be recorded into a graph.
    bool tail_pinned = true;
    for (const void* ptr : {k_tail_host, v_tail_host}) {
        if (n_tail == 0 || ptr == nullptr) continue;
        cudaPointerAttributes attr;
        if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
            cudaGetLastError();
            tail_pinned = false;
        } else if (attr.type == cudaMemoryTypeUnregistered) {
            tail_pinned = false;
        }
    }

    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    unsigned long long capture_id = 0;
    if (cudaStreamGetCaptureInfo(cs, &cap, &capture_id) != cudaSuccess) return KVATTN_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusActive) capture_id = 0;
    // Prefetch mode enqueues directly: a graph launched on the compute stream could not
    // start its copies before the compute stream reached it.  Its first call through a
    // context (or the first after a call in the other mode) still orders its copies after
    // the compute stream, since the slots' last readers are not known yet; so does the first
    // call of a stream capture (the readers' records lie outside it) -- a whole decode step
    // captured with its layers in this mode replays as one graph whose copies run ahead
    // across layers.
    const bool prefetch = (ctx->flags & KVATTN_TAIL_PREFETCH) != 0u;
    const bool carry = prefetch && ctx->carry_valid && ctx->carry_capture == capture_id;
    const bool use_graph =
        !prefetch && tail_pinned && use_tail_graph() && cap == cudaStreamCaptureStatusNone && fault < 0;
    if (!use_graph) {
        const int slot0 = prefetch ? (int)(ctx->tiles_issued & 1u) : 0;
        ctx->carry_valid = false;  // until this call's records are all enqueued
        const int rc = enqueue_window_tail(ctx, plan, k_tail_host, v_tail_host, k_dev, v_dev, n_tail, tile_cells, cs,
                                           xs, ctx->copy2, fault, prefetch, carry, slot0, capture_id != 0);
        if (rc != KVATTN_OK) return rc;
        if (prefetch) {
            ctx->tiles_issued += (uint64_t)plan.L.n_tiles;
            ctx->carry_valid = true;
            ctx->carry_capture = capture_id;
        }
    } else {
        ctx->carry_valid = false;
        TailGraphKey key;
        std::memset(&key, 0, sizeof(key));
        key.q = q;
        key.k_win = k_win;
        key.v_win = v_win;
        key.k_tail = k_tail_host;
        key.v_tail = v_tail_host;
        key.k_tail_dev = k_dev;
        key.v_tail_dev = v_dev;
        key.n_win = n_win;
        key.n_tail = n_tail;
        key.tile_cells = tile_cells;
        key.n_head = n_head;
        key.n_head_kv = n_head_kv;
        key.head_dim = head_dim;
        key.split = split;
        key.tail_split = tail_split;
        key.scale = scale;
        key.out = out;
        key.lse = lse;
        key.ws = ws;
        key.ws_bytes = ws_bytes;
        key.stall_tx = plan.base.stall_tx;
        key.wait_limit_ns = plan.base.wait_limit_ns;
        key.pdl = plan.pdl ? 1 : 0;
        cudaGetDevice(&key.device);
        TailGraphEntry* hit = nullptr;
        for (int i = 0; i < ctx->n_graphs && hit == nullptr; ++i)
            if (ctx->graphs[i].key == key) hit = &ctx->graphs[i];
        if (hit == nullptr) {
            // a free entry, or the least recently used one
            TailGraphEntry* slot = nullptr;
            if (ctx->n_graphs < kTailGraphSlots) {
                slot = &ctx->graphs[ctx->n_graphs];
            } else {
                slot = &ctx->graphs[0];
                for (int i = 1; i < ctx->n_graphs; ++i)
                    if (ctx->graphs[i].last_use < slot->last_use) slot = &ctx->graphs[i];
                cudaGraphExecDestroy(slot->exec);
                *slot = ctx->graphs[--ctx->n_graphs];
                slot = &ctx->graphs[ctx->n_graphs];
            }
            // Record the pipeline once as a graph: ~3 operations per tile would otherwise
            // cost more host time per call than the host-to-device copies themselves.
            // (recorded on private streams: the caller's may be the legacy default stream)
            if (cudaStreamBeginCapture(ctx->cap_main, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
                return KVATTN_ERR_CUDA;
            const int rc = enqueue_window_tail(ctx, plan, k_tail_host, v_tail_host, k_dev, v_dev, n_tail, tile_cells,
                                               ctx->cap_main, ctx->cap_fork, ctx->cap_fork2, -1);
            cudaGraph_t graph = nullptr;
            const cudaError_t ec = cudaStreamEndCapture(ctx->cap_main, &graph);
            if (rc != KVATTN_OK || ec != cudaSuccess || graph == nullptr) {
                if (graph != nullptr) cudaGraphDestroy(graph);
                return rc != KVATTN_OK ? rc : KVATTN_ERR_CUDA;
            }
            cudaGraphExec_t exec = nullptr;
            const cudaError_t ei = cudaGraphInstantiate(&exec, graph, 0);
            cudaGraphDestroy(graph);
            if (ei != cudaSuccess) return KVATTN_ERR_CUDA;
            slot->key = key;
            slot->exec = exec;
            ++ctx->n_graphs;
            hit = slot;
        }
        hit->last_use = ++ctx->use_clock;
        if (cudaGraphLaunch(hit->exec, cs) != cudaSuccess) return KVATTN_ERR_CUDA;
    }
    if (log_on())
        log_line("window_tail n_win=%lld n_tail=%lld tiles=%lld tile_cells=%lld mode=%s copy=%s graphs_cached=%d",
                 (long long)n_win, (long long)n_tail, (long long)plan.L.n_tiles, (long long)tile_cells,
                 use_graph ? "graph" : (prefetch ? (carry ? "prefetch-carried" : "prefetch-first") : "direct-enqueue"),
                 k_dev != nullptr ? "kernel" : "engine", ctx->n_graphs);
    if (cudaEventRecord(ctx->done, cs) != cudaSuccess) return KVATTN_ERR_CUDA;
    ctx->pending = true;
    return KVATTN_OK;
}

size_t kvattn_window_tail_direct_workspace_bytes(int n_head, int n_head_kv, int head_dim, int64_t n_win,
                                                 int64_t n_tail, int split, int tail_split) {
    if (n_head < 1 || n_head_kv < 1 || head_dim < 1 || n_win < 0 || n_tail < 0 || split < 1 || tail_split < 1)
        return 0;
    const int64_t parts = (n_win + split - 1) / split + (n_tail + tail_split - 1) / tail_split;
    return decode_ws_layout(1, n_head, head_dim, parts).total;
}

int kvattn_decode_window_tail_direct(const void* q, const void* k_win, const void* v_win, int64_t n_win,
                                     const void* k_tail_host, const void* v_tail_host, int64_t n_tail, int n_head,
                                     int n_head_kv, int head_dim, int split, int tail_split, float scale, float* out,
                                     float* lse, void* ws, size_t ws_bytes, void* stream) {
    if (q == nullptr || out == nullptr || lse == nullptr || ws == nullptr) return KVATTN_ERR_INVALID_ARG;
    int st = check_shape(DecodeShape{1, n_head, n_head_kv, head_dim, split, n_win});
    if (st != KVATTN_OK) return st;
    st = check_shape(DecodeShape{1, n_head, n_head_kv, head_dim, tail_split, n_tail});
    if (st != KVATTN_OK) return st;
    if (!std::isfinite(scale)) return KVATTN_ERR_INVALID_ARG;
    if ((n_win > 0 && (k_win == nullptr || v_win == nullptr)) ||
        (n_tail > 0 && (k_tail_host == nullptr || v_tail_host == nullptr)))
        return KVATTN_ERR_INVALID_ARG;
    if (!aligned(q, 4) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(ws, kWsAlign) ||
        (k_win && !aligned(k_win, 16)) || (v_win && !aligned(v_win, 16)) ||
        (k_tail_host && !aligned(k_tail_host, 16)) || (v_tail_host && !aligned(v_tail_host, 16)))
        return KVATTN_ERR_INVALID_ARG;
    const int64_t n_split_win = (n_win + split - 1) / split;
    const int64_t n_split_tail = (n_tail + tail_split - 1) / tail_split;
    const int64_t n_parts = n_split_win + n_split_tail;
    const DecodeWsLayout lay = decode_ws_layout(1, n_head, head_dim, n_parts);
    if (ws_bytes < lay.total) return KVATTN_ERR_WORKSPACE;
    // the device's view of the pinned tail (fails for memory that is not pinned and mapped)
    void* dk = nullptr;
    void* dv = nullptr;
    if (n_tail > 0) {
        if (cudaHostGetDevicePointer(&dk, const_cast<void*>(k_tail_host), 0) != cudaSuccess ||
            cudaHostGetDevicePointer(&dv, const_cast<void*>(v_tail_host), 0) != cudaSuccess) {
            cudaGetLastError();  // clear the error the failed query leaves behind
            return KVATTN_ERR_INVALID_ARG;
        }
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    char* wsb = static_cast<char*>(ws);
    const bool pdl = use_pdl();
    SplitDecodeParams p = {};
    p.q = static_cast<const __half*>(q);
    p.part_o = reinterpret_cast<float*>(wsb + lay.o_off);
    p.part_lse = reinterpret_cast<float*>(wsb + lay.lse_off);
    p.status = reinterpret_cast<uint32_t*>(wsb);
    p.n_split = n_parts;
    p.part_stride = n_parts;
    p.write_beyond = 1;
    p.n_seq = 1;
    p.n_head = n_head;
    p.n_head_kv = n_head_kv;
    p.group = n_head / n_head_kv;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634074);
    apply_debug_hooks(p);
    SplitDecodeParams w = p;
    if (n_split_win > 0) {
        w.k = k_win;
        w.v = v_win;
        w.n_cells = n_win;
        w.max_len = n_win;
        w.fixed_len = n_win;
        w.split = split;
        w.part_base = 0;
        w.n_stages = pick_stages(KVATTN_KV_F16, head_dim, n_split_win * n_head_kv);
        set_kv_maps(w, KVATTN_KV_F16, n_win, n_head_kv, head_dim);
    }
    SplitDecodeParams t = p;
    if (n_split_tail > 0) {
        // the tail's rows cross the host link once, straight into shared memory
        t.k = dk;
        t.v = dv;
        t.n_cells = n_tail;
        t.max_len = n_tail;
        t.fixed_len = n_tail;
        t.split = tail_split;
        t.part_base = n_split_win;
        t.use_tma = 0;
        t.src_lsu = 1;
        t.n_stages = pick_stages(KVATTN_KV_F16, head_dim, n_split_tail * n_head_kv);
    }
    // When the tail's units fit in one wave, its decode (bound by the host link) goes first
    // with a full dependency on the work before it, triggers its dependents at entry, and the
    // window's decode (bound by HBM) follows as that programmatic dependent: reading nothing
    // the tail writes, it skips the dependency wait, so both run at once; the merge then
    // waits for both (ordinary launch).  Otherwise the window goes first and each launch
    // waits for the one before it.
    const bool overlap =
        pdl && n_split_win > 0 && n_split_tail > 0 &&
        n_split_tail * n_head_kv <= (int64_t)occupancy(KVATTN_KV_F16, head_dim, t.n_stages) * sm_count();
    if (overlap) {
        if (launch_decode_units(t, KVATTN_KV_F16, head_dim, n_split_tail, cs, false) != cudaSuccess)
            return KVATTN_ERR_CUDA;
        w.no_dep_wait = 1;
        if (launch_decode_units(w, KVATTN_KV_F16, head_dim, n_split_win, cs, true) != cudaSuccess)
            return KVATTN_ERR_CUDA;
    } else {
        if (n_split_win > 0 && launch_decode_units(w, KVATTN_KV_F16, head_dim, n_split_win, cs, pdl) != cudaSuccess)
            return KVATTN_ERR_CUDA;
        if (n_split_tail > 0 &&
            launch_decode_units(t, KVATTN_KV_F16, head_dim, n_split_tail, cs, false) != cudaSuccess)
            return KVATTN_ERR_CUDA;
    }
    if (log_on())
        log_line("window_tail_direct n_win=%lld n_tail=%lld window_splits=%lld tail_splits=%lld overlap=%d",
                 (long long)n_win, (long long)n_tail, (long long)n_split_win, (long long)n_split_tail, overlap ? 1 : 0);
    MergeParams m = {};
    m.part_o = p.part_o;
    m.part_lse = p.part_lse;
    m.out = out;
    m.lse = lse;
    m.n_parts = n_parts;
    m.n_seq = 1;
    m.n_rows = n_head;
    m.head_dim = head_dim;
    m.split = 1;
    m.all_written = 1;
    m.allow_slices = env_int("KVATTN_MERGE_SLICES", 1) != 0;
    m.wide_rows_max = sm_count();
    // after the overlapped decodes the merge must follow both: an ordinary launch
    return cuda_status(launch_merge(m, cs, pdl && n_parts > 0 && !overlap));
}

int kvattn_tail_wait(kvattn_tail_ctx* ctx, int timeout_ms) {
    if (ctx == nullptr || timeout_ms < 0) return KVATTN_ERR_INVALID_ARG;
    if (!ctx->pending) return KVATTN_OK;
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        const cudaError_t e = cudaEventQuery(ctx->done);
        if (e == cudaSuccess) {
            ctx->pending = false;
            return KVATTN_OK;
        }
        if (e != cudaErrorNotReady) return KVATTN_ERR_CUDA;
        const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                            std::chrono::steady_clock::now() - t0)
                            .count();
        if (ms >= timeout_ms) return KVATTN_ERR_TIMEOUT;
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
}

int kvattn_workspace_status(void* ws, uint32_t* flags, int clear, void* stream) {
    if (ws == nullptr || flags == nullptr) return KVATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return KVATTN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVATTN_ERR_CUDA;
    *flags = v;
    if (clear) {
        if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), s) != cudaSuccess) return KVATTN_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return KVATTN_ERR_CUDA;
    }
    return KVATTN_OK;
}

}  // extern "C"
