/*
 * kvattn -- single-query (n_q = 1) split-KV decode attention for GB300 (sm_103a).
 *
 * C ABI: plain pointers and sizes only.  "device" pointers are CUDA device memory of
 * the current device, "host" pointers are ordinary (or pinned, where stated) host
 * memory.  Streams are passed as `void*` holding a cudaStream_t (NULL = the legacy
 * default stream).  The caller owns every buffer; the library allocates no device
 * memory on any decode path.  Every call validates its arguments on the host before
 * it touches CUDA and returns a kvattn_status; it never aborts, and it prints nothing
 * unless the environment variable KVATTN_LOG=1 asks for one line on stderr per launching
 * call (the chosen split, grid, ring depth, descriptor path, tail mode).
 * Device calls are asynchronous on the given stream(s).
 *
 * Host threads: every entry point may be called from several threads at once (the
 * library's per-device caches -- SM count, occupancy, kernel attributes, the tensor-map
 * encoder -- are filled once under a lock), except that one kvattn_tail_ctx serves one
 * thread at a time: it holds the window + tail pipeline's events, slot sequence and
 * recorded graphs.  Work that shares a workspace must be ordered on the device by the
 * caller (one stream, or events).
 *
 * Sources (web pages, cited by title and section):
 *  [RKV]  "Rolling-KV -- overflow throughput evaluations (consolidated)",
 *         opencoti-llamafile docs/evaluations/rolling_kv.md
 *  [KVN]  "KVARN KV Performance optimizations", beellama.cpp issue #140
 *
 * Attention definition (what every decode entry point computes, up to floating-point
 * reduction order): for sequence s and query head h, G = n_head / n_head_kv,
 * g = floor(h / G), over the valid cells c of the sequence
 *     x_c = scale * q[s][h] . K[c][g],   O[s][h] = sum_c softmax(x)_c V[c][g],
 *     LSE[s][h] = ln sum_c exp(x_c)      (-inf and O = 0 when no cell is valid).
 * Split-KV: cells are cut into splits; each split yields a partial (O_p, LSE_p) and
 * the partials are merged with weights exp(LSE_p - max LSE) ([RKV] section 3, the
 * decode-emitted LSE channel; [KVN] item 9, partial windows keep max, numerator and
 * denominator and are merged afterwards).
 *
 * Cache layouts
 *  f16  : K, V  half  [n_cells][n_head_kv][head_dim]          (cell-major rows)
 *  Q8_0 : K, V  int8  [n_cells][n_head_kv][head_dim] and scales
 *         half [n_cells][n_head_kv][head_dim / 32]; value = scale * int8, one scale
 *         per 32 consecutive head_dim elements (structure-of-arrays planes, chosen so
 *         that every row starts on a 16-byte boundary).
 *  Q8_0_Q4_0 : K as Q8_0; V uint8 [n_cells][n_head_kv][head_dim / 2] and scales half
 *         [n_cells][n_head_kv][head_dim / 32].  V is q4_0 ([RKV] resident-compression
 *         anchors, the "q8_0K/q4_0V" cache): 32 consecutive head_dim elements share one
 *         scale and 16 bytes; byte j of block b (byte 16b + j of the row) holds element
 *         32b + j in its low nibble and 32b + 16 + j in its high nibble; value =
 *         scale * (nibble - 8) (the llama.cpp q4_0 block, values and scales in two planes).
 *  Q4_0 : K and V both as the Q4_0 values above ([RKV] section 5a, the q4_0 cache).
 *  q    : half  [n_seq][n_head][head_dim];  out: float [n_seq][n_head][head_dim];
 *  lse  : float [n_seq][n_head] (natural log).
 */
#ifndef KVATTN_H
#define KVATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVATTN_OK = 0,
    KVATTN_ERR_INVALID_ARG = -1,   /* null pointer, bad size, misaligned buffer */
    KVATTN_ERR_UNSUPPORTED = -2,   /* valid but not built: head_dim, group size, split */
    KVATTN_ERR_WORKSPACE = -3,     /* workspace smaller than the *_workspace_bytes query */
    KVATTN_ERR_CAPACITY = -4,      /* a cell beyond the cache, or a plan row too long */
    KVATTN_ERR_CUDA = -5,          /* a CUDA call or launch failed */
    KVATTN_ERR_TIMEOUT = -6        /* a bounded host wait ran out */
} kvattn_status;

typedef enum {
    KVATTN_KV_F16 = 0,
    KVATTN_KV_Q8_0 = 1,
    KVATTN_KV_Q8_0_Q4_0 = 2,
    KVATTN_KV_Q4_0 = 3
} kvattn_kv_type;

/* Sticky device-side status bits, read with kvattn_workspace_status. */
#define KVATTN_DEVICE_WAIT_TIMEOUT 1u   /* a bounded pipeline wait gave up; results invalid */
#define KVATTN_DEVICE_BAD_PLAN_ENTRY 2u /* a plan entry outside [-1, n_cells) was masked */

/* Human-readable name of a kvattn_status (static storage, never NULL). */
const char* kvattn_status_string(int status);

/* ABI version of this header: (major << 16) | minor. */
int kvattn_version(void);

/*
 * kvattn_build_cell_plan -- host.  The compact indirect cell plan of [KVN] item 4
 * ("physical record-group-safe compact plans") with the duplicate handling of item 3
 * and the encoded-index rule of item 5.
 *
 *  cells    host int64 [offsets[n_seq]]: the concatenated per-sequence lists of encoded
 *           cell indices; low 32 bits (unsigned) = physical cell, high 32 bits = a
 *           stage-slot tag that the read plan ignores.  Order and duplicates are free.
 *  offsets  host int64 [n_seq + 1], non-decreasing, offsets[0] = 0.
 *  capacity_cells  physical cells in the cache (> 0).
 *  plan     host int32 [n_seq][plan_stride] output, or NULL to only compute seq_lens.
 *  seq_lens host int32 [n_seq] output: 128 x (number of distinct records selected).
 *
 * Each sequence's row is its selected physical 128-cell records in ascending order,
 * one complete 128-entry segment per record, entry j = record*128 + j when that cell
 * was selected and -1 (a hole) otherwise; the rest of the row is -1.
 * Errors: INVALID_ARG (null cells/offsets/seq_lens with work to do, bad offsets,
 * n_seq < 0, capacity < 1, plan_stride < 0); CAPACITY (a physical cell >= capacity,
 * or a row longer than plan_stride).  On error the outputs are unspecified.
 */
int kvattn_build_cell_plan(const int64_t* cells, const int64_t* offsets, int n_seq,
                           int64_t capacity_cells, int32_t* plan, int64_t plan_stride,
                           int32_t* seq_lens);

/*
 * kvattn_build_descriptors -- device.  Per-split descriptors of a cell plan ([KVN]
 * item 5, "descriptor setup"; item 6, "fully masked split skipping").
 *
 *  cell_plan  device int32 [n_seq][plan_stride];  seq_lens device int32 [n_seq].
 *  desc       device int32 [n_seq][ceil(max_len / split)][4] output:
 *             {n_valid, lo, hi, flags} over plan entries [p*split, min((p+1)*split, L))
 *             with L = min(seq_lens[s], max_len, plan_stride); an entry e is valid when
 *             0 <= e < n_cells; lo/hi = smallest/largest valid cell (-1 if none);
 *             flags: 1 = no valid entry, 2 = linear (e - i constant over valid entries),
 *             4 = an entry outside [-1, n_cells) was seen, 8 = split starts at/after L.
 * Errors: INVALID_ARG (null pointers, n_seq < 0, split < 1, max_len < 0, n_cells < 1,
 * plan_stride < 1); CUDA.
 */
int kvattn_build_descriptors(const int32_t* cell_plan, int64_t plan_stride,
                             const int32_t* seq_lens, int n_seq, int64_t max_len, int split,
                             int64_t n_cells, int32_t* desc, void* stream);

/* Bytes of workspace kvattn_decode needs (partials, descriptors, status word).  split 0:
 * enough for whichever split kvattn_decode selects (it sizes for split 64).  Returns 0 on
 * invalid arguments. */
size_t kvattn_decode_workspace_bytes(int n_seq, int n_head, int head_dim, int64_t max_len,
                                     int split);

/*
 * kvattn_select_split_for -- host, pure.  The split kvattn_decode uses when it is given
 * split 0 ("split-size auto-selector", [KVN] item 6 and its split-64 / split-128 geometry,
 * re-measured for GB300): the smallest power of two >= 64 such that the work units
 * n_seq x ceil(max_len / split) x n_head_kv fit in resident_ctas (one wave of the decode
 * kernel's CTAs); a split that reaches max_len (one split per sequence) or 2^30 ends the
 * search.  Returns the split, or INVALID_ARG (n_seq < 0, max_len < 0, n_head_kv < 1,
 * resident_ctas < 1).
 */
int kvattn_select_split_for(int n_seq, int64_t max_len, int n_head_kv, int64_t resident_ctas);

/*
 * kvattn_select_split -- host.  kvattn_select_split_for with the resident CTA count of the
 * decode kernel for (kv_type, head_dim) on the current device (queries the device; no
 * work is enqueued).  Errors: INVALID_ARG, UNSUPPORTED (head_dim not 128 or 256).
 */
int kvattn_select_split(int kv_type, int n_seq, int64_t max_len, int n_head_kv, int head_dim);

/*
 * kvattn_decode -- device.  Split-KV decode attention ([RKV] sections 1 and 3; [KVN]
 * items 2, 4, 6 and 9): per (sequence, KV head, split) one CTA streams the split's
 * K/V rows through shared memory once for all G query heads of that KV head, and
 * emits a partial (O_p, LSE_p); a second kernel merges the partials.
 *
 *  q        device half [n_seq][n_head][head_dim].
 *  k_cache, v_cache  device, 16-byte aligned.  f16: half rows.  Q8_0: int8 rows.
 *           Q8_0_Q4_0: int8 K rows, packed 4-bit V rows of head_dim / 2 bytes.  Q4_0: packed
 *           4-bit K and V rows.
 *  k_scales, v_scales  device half scale planes of the quantised types (8-byte aligned
 *           for head_dim 128, 16-byte for 256); must be NULL for f16.
 *  kv_type  a kvattn_kv_type.
 *  n_cells  rows per sequence when cell_plan is NULL (sequence s reads rows
 *           [s*n_cells, s*n_cells + seq_len)), or rows of the unified cache otherwise.
 *  cell_plan  NULL, or device int32 [n_seq][plan_stride]: sequence s reads the cells
 *           cell_plan[s][0 .. seq_len) with -1 holes (see kvattn_build_cell_plan).
 *           Entries outside [-1, n_cells) are masked and flagged in the workspace.
 *  seq_lens device int32 [n_seq]; each is clamped to [0, max_len] and to n_cells (no
 *           plan) or plan_stride (plan).
 *  max_len  host bound on the lengths; sizes the grid and the workspace.
 *  n_head, n_head_kv  n_head % n_head_kv == 0 and n_head / n_head_kv <= 8.
 *  head_dim 128 or 256.   split  cells per partial, a positive multiple of 32, or 0 to
 *           use kvattn_select_split (kvattn_decode and kvattn_decode_noalloc only).
 *  scale    softmax scale applied to q . k in fp32 (1/sqrt(head_dim) is usual).
 *  out, lse device float outputs.   ws/ws_bytes  device workspace of at least
 *           kvattn_decode_workspace_bytes(...) bytes, 256-byte aligned, zeroed once
 *           after allocation (its first word is the sticky status word).  After a call
 *           with a cell_plan, bytes [256, 256 + 16 n_seq n_split) hold the per-split
 *           descriptors int32 {n_valid, lo, hi, flags} [n_seq][n_split] (n_split =
 *           ceil(max_len / split)) exactly as kvattn_build_descriptors computes them.
 *  stream   cudaStream_t.
 *  Size limits (UNSUPPORTED beyond them): n_seq x n_head output rows and n_seq x
 *  ceil(max_len / split) x n_head_kv work units each below 2^31.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE (before any launch); CUDA.
 */
int kvattn_decode(const void* q, const void* k_cache, const void* v_cache,
                  const void* k_scales, const void* v_scales, int kv_type, int64_t n_cells,
                  const int32_t* cell_plan, int64_t plan_stride, const int32_t* seq_lens,
                  int n_seq, int64_t max_len, int n_head, int n_head_kv, int head_dim,
                  int split, float scale, float* out, float* lse, void* ws, size_t ws_bytes,
                  void* stream);

/*
 * kvattn_decode_partials -- device.  The split step of kvattn_decode alone: the same
 * arguments and checks, but every split's normalised partial and its LSE are written to
 * caller buffers instead of being merged, so that they can be merged with partials from
 * elsewhere (another device, a host tail) by kvattn_merge.
 *  part_o    device float [n_seq][ceil(max_len / split)][n_head][head_dim], 16-byte aligned.
 *  part_lse  device float [n_seq][ceil(max_len / split)][n_head].
 * Splits past a sequence's length, and splits with no valid cell, are written as
 * O_p = 0, LSE_p = -inf.  ws: as for kvattn_decode (status word and descriptors).
 * Errors: as kvattn_decode.
 */
int kvattn_decode_partials(const void* q, const void* k_cache, const void* v_cache,
                           const void* k_scales, const void* v_scales, int kv_type,
                           int64_t n_cells, const int32_t* cell_plan, int64_t plan_stride,
                           const int32_t* seq_lens, int n_seq, int64_t max_len, int n_head,
                           int n_head_kv, int head_dim, int split, float scale, float* part_o,
                           float* part_lse, void* ws, size_t ws_bytes, void* stream);

/* Bytes of workspace kvattn_decode_multi needs (split 0: as kvattn_decode_workspace_bytes). */
size_t kvattn_decode_multi_workspace_bytes(int n_seq, int n_q, int n_head, int head_dim, int64_t max_len,
                                           int split);

/*
 * kvattn_decode_multi -- device.  Causal multi-query decode ("small multi-query decode,
 * n_q <= 8/16 with a mask", the speculative-verify case of [RKV] section 3 and [KVN] items
 * 2 and 7, split decode eligible through n_q <= 8 with an attention mask): n_q new query
 * tokens per sequence, whose own K/V cells are already in the cache.  seq_lens[s] = L
 * counts them, token t sits at logical position L - n_q + t and attends to the logical
 * positions 0 .. L - n_q + t (plan entries or cells, -1 holes masked); a token whose window
 * is empty gets O = 0, LSE = -inf.  The G x n_q query rows of each KV head share every K/V
 * byte read from HBM (one or two 16-row MMA tiles, up to 32 rows; f16 at head_dim 128 with
 * q 16-byte aligned, 33 to 128 rows -- and 17 to 32 when the call's work units fit about
 * one wave of its CTAs, as the automatic split arranges -- one tcgen05 tile of all the
 * rows).  n_q = 1 is
 * exactly kvattn_decode (and runs its kernels); up to 8 rows per KV head (f16, and the
 * quantised types at head_dim 128) run on the single-query kernels with per-row causal
 * masks.
 *  q        device half [n_seq][n_q][n_head][head_dim].
 *  out, lse device float [n_seq][n_q][n_head][head_dim], [n_seq][n_q][n_head].
 *  Other arguments: as kvattn_decode.
 *  Limits (UNSUPPORTED otherwise): n_q >= 1 and (n_head / n_head_kv) * n_q <= 128 query
 *  rows per KV head (n_q <= 16 at up to 8 query heads per KV head); any kv_type; head_dim
 *  128 or 256.  Rows beyond one unit's share (f16: 32 at head_dim 128 when the tcgen05
 *  tile does not serve them, 16 at 256; the quantised types: 16 at head_dim 128, 8 at 256)
 *  run as row groups, units of their own that read the split's K/V again, mostly from L2
 *  (the groups of a split run side by side).
 *  ws: kvattn_decode_multi_workspace_bytes(...) bytes.
 * Errors: as kvattn_decode.
 */
int kvattn_decode_multi(const void* q, const void* k_cache, const void* v_cache,
                        const void* k_scales, const void* v_scales, int kv_type, int64_t n_cells,
                        const int32_t* cell_plan, int64_t plan_stride, const int32_t* seq_lens,
                        int n_seq, int64_t max_len, int n_q, int n_head, int n_head_kv, int head_dim,
                        int split, float scale, float* out, float* lse, void* ws, size_t ws_bytes,
                        void* stream);

/*
 * kvattn_merge -- device.  LSE-weighted merge of partial attention results ([KVN]
 * item 9; [RKV] section 3):  M = max_p LSE_p, w_p = exp(LSE_p - M),
 * out = sum_p w_p O_p / sum_p w_p, lse = M + ln sum_p w_p.  Parts with LSE = -inf hold
 * no cells and are skipped without reading their O; if every part is -inf the row is
 * O = 0, LSE = -inf.
 *  partials device float [n_parts][n_rows][head_dim];  lses device float [n_parts][n_rows].
 *  out      device float [n_rows][head_dim];  lse device float [n_rows].
 *  head_dim a positive multiple of 4, at most 1024.  n_parts >= 0.  All 16-byte aligned.
 * Errors: INVALID_ARG; CUDA.
 */
int kvattn_merge(const float* partials, const float* lses, int n_parts, int n_rows, int head_dim,
                 float* out, float* lse, void* stream);

/*
 * kvattn_decode_noalloc -- device.  kvattn_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart of this entry point; it exists for code that is
 * not allowed to call cudaMalloc where it runs decode attention -- inside a fixed memory
 * pool's budget, as a plugin that is handed only its inputs and outputs, or on a path that
 * must not wait on the driver's allocator.  It allocates nothing: the caller passes the
 * same inputs and outputs as kvattn_decode (no workspace), and the scratch lives in an
 * array of KVATTN_NOALLOC_SCRATCH_BYTES bytes that the library keeps in device memory on
 * every GPU that loads it, until the process exits.
 *
 *  Arguments, layouts and results: as kvattn_decode.
 *  Limit: a call whose kvattn_decode_workspace_bytes(n_seq, n_head, head_dim, max_len,
 *         split) exceeds KVATTN_NOALLOC_SCRATCH_BYTES returns KVATTN_ERR_WORKSPACE and
 *         launches nothing; use kvattn_decode with a caller workspace for such shapes.
 *  Set-up: the first call on a device looks up the array's device address on that device
 *         (cudaGetSymbolAddress) and remembers it; make that first call before any stream
 *         capture begins on the device.
 *  Sharing: every call on a device uses the same array, which keeps the previous call's
 *         contents (each call clears the status word it needs at zero).  Calls whose work
 *         overlaps on the GPU -- on different streams, or from different threads without
 *         ordering -- race on the array and give wrong results; order them on one stream.
 *  Device: the array used is the current device's, so `stream` must belong to the current
 *         device (as for every entry point of this library).
 *  Device-side status bits of this path are not reported.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE (all checked before the array's address is
 *         looked up and before anything is enqueued); CUDA.
 */
#define KVATTN_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

int kvattn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                          const void* k_scales, const void* v_scales, int kv_type, int64_t n_cells,
                          const int32_t* cell_plan, int64_t plan_stride, const int32_t* seq_lens,
                          int n_seq, int64_t max_len, int n_head, int n_head_kv, int head_dim,
                          int split, float scale, float* out, float* lse, void* stream);

/*
 * Window + host tail ([RKV] sections 1 and 5c: "POSITION_WINDOW keeps a resident window of
 * recent cells and streams the older tail from host RAM every decode step"; the window is
 * attended on the device and the tail streamed once, one tile ahead, and the partials are
 * merged).  One sequence, f16 cache.
 *
 * A tail context owns only CUDA events (no memory).
 */
typedef struct kvattn_tail_ctx kvattn_tail_ctx;

int kvattn_tail_ctx_create(kvattn_tail_ctx** ctx);
int kvattn_tail_ctx_destroy(kvattn_tail_ctx* ctx);

/*
 * kvattn_tail_ctx_set_flags -- host.  Mode of the later kvattn_decode_window_tail calls
 * through ctx (0 by default).
 *
 * KVATTN_TAIL_PREFETCH: cross-layer prefetch ([RKV] section 1, the cross-layer barrier
 * between the compute stream and the tail copies; the step-prefetch design).  A model calls
 * kvattn_decode_window_tail once per layer through one context.  Without the flag every
 * copy of a call waits for all work enqueued before it on compute_stream, so layer l+1's
 * tail cannot cross the link while layer l still computes.  With the flag a copy waits only
 * for
 *   - the work enqueued before the call on copy_stream (order a device-side write into the
 *     tail before the call there), and
 *   - the tile decode that last read its staging slot, in this call or an earlier one
 *     through the same context,
 * and the two staging slots alternate across calls, so the next layer's first two tiles
 * are copied while this layer's window, tiles and merge run.  The first call after the
 * flag is set, or after a call without it, still orders its copies after compute_stream.
 * Calls in this mode enqueue the pipeline directly (no CUDA graph), about six operations
 * per tile: use tiles large enough that a tile's copy outlasts that host work (a whole
 * layer's tail per tile is a fine choice when two of them fit in device memory).
 * Contract: a context's calls in this mode run on the same compute_stream and copy_stream,
 * and a workspace's staging slots are used through one context only.
 * Errors: INVALID_ARG (null ctx, unknown flag bits).
 */
#define KVATTN_TAIL_PREFETCH 1u

int kvattn_tail_ctx_set_flags(kvattn_tail_ctx* ctx, uint32_t flags);

/* Bytes of workspace for kvattn_decode_window_tail: two staging slots of tile_cells rows
 * of K and of V, the partials of the window splits and of every tail tile, status word. */
size_t kvattn_window_tail_workspace_bytes(int n_head, int n_head_kv, int head_dim,
                                          int64_t n_win, int64_t n_tail, int split,
                                          int64_t tile_cells, int tail_split);

/*
 *  q          device half [n_head][head_dim].
 *  k_win, v_win  device half [n_win][n_head_kv][head_dim] -- the resident window.
 *  k_tail_host, v_tail_host  PINNED host half [n_tail][n_head_kv][head_dim] -- the older
 *             tail (cudaHostAlloc / cudaHostRegister memory).  Pageable memory is accepted
 *             but slow: its copies stage through the driver and are never recorded into a
 *             graph.
 *  tile_cells tail cells per host-to-device tile (a positive multiple of tail_split);
 *             tiles are copied into two device staging slots, one tile ahead of the
 *             compute (double buffering), each copy ordered after the decode that last
 *             read its slot.  A tile moves by one copy kernel that reads the pinned
 *             buffers through their device mapping (cudaHostGetDevicePointer), or by two
 *             cudaMemcpyAsync when they are not mapped (or KVATTN_TAIL_COPY=0 is set);
 *             even tiles go on copy_stream, odd tiles on a stream of the context, so one
 *             copy ramps up while the previous drains.  The first call with a given set of
 *             arguments records the whole pipeline as a CUDA graph (on the context's own
 *             streams) and launches it on compute_stream; later calls with the same
 *             arguments replay that graph, so the host enqueues one launch instead of about
 *             six operations per tile.  A context keeps the graphs of its 64 most recently
 *             used argument sets (one per layer of a model that shares the context).  A
 *             call on a compute_stream that is itself being captured, or in
 *             KVATTN_TAIL_PREFETCH mode, enqueues the pipeline on compute_stream and
 *             copy_stream directly.
 *  split      cells per partial over the window; tail_split  cells per partial inside a
 *             tile.  Both positive multiples of 32.
 *  out, lse   device float [n_head][head_dim], [n_head].
 *  compute_stream, copy_stream  cudaStream_t; must differ.  On return every kernel and
 *             copy is enqueued; out/lse are ready when compute_stream reaches this point.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE (before any CUDA call); CUDA (work already
 * enqueued stays enqueued; outputs are then unspecified).
 */
int kvattn_decode_window_tail(kvattn_tail_ctx* ctx, const void* q,
                              const void* k_win, const void* v_win, int64_t n_win,
                              const void* k_tail_host, const void* v_tail_host, int64_t n_tail,
                              int64_t tile_cells, int n_head, int n_head_kv, int head_dim,
                              int split, int tail_split, float scale, float* out, float* lse,
                              void* ws, size_t ws_bytes, void* compute_stream,
                              void* copy_stream);

/*
 * kvattn_decode_window_tail_direct -- device.  The same window + host tail attention
 * ([RKV] sections 1 and 5c), but the decode kernel reads the tail's rows straight from
 * pinned host memory with 16-byte asynchronous loads, with no staging copies and no copy
 * stream.  Attention reads every tail byte exactly once, so reading host memory in place
 * costs no more link traffic than copying it first ([KVN], the note that plain zero-copy
 * lost only because a GEMM re-reads each weight tile), and it avoids the fixed per-copy
 * cost of many 1 MiB host-to-device copies.
 *
 *  q, k_win, v_win, n_win, split, scale, out, lse: as kvattn_decode_window_tail.
 *  k_tail_host, v_tail_host  pinned, device-mapped host memory (cudaHostAlloc,
 *             torch pin_memory(), or cudaHostRegister with mapping), 16-byte aligned,
 *             half [n_tail][n_head_kv][head_dim].
 *  tail_split cells per partial over the tail (a positive multiple of 32).
 *  ws         at least kvattn_window_tail_direct_workspace_bytes(...) bytes.
 *  stream     everything runs on this stream.
 * Errors: INVALID_ARG (including tail memory the device cannot address), UNSUPPORTED,
 * WORKSPACE (before any launch); CUDA.
 */
size_t kvattn_window_tail_direct_workspace_bytes(int n_head, int n_head_kv, int head_dim,
                                                 int64_t n_win, int64_t n_tail, int split,
                                                 int tail_split);

int kvattn_decode_window_tail_direct(const void* q, const void* k_win, const void* v_win,
                                     int64_t n_win, const void* k_tail_host,
                                     const void* v_tail_host, int64_t n_tail, int n_head,
                                     int n_head_kv, int head_dim, int split, int tail_split,
                                     float scale, float* out, float* lse, void* ws,
                                     size_t ws_bytes, void* stream);

/* Wait (host, bounded) until everything the last kvattn_decode_window_tail on this ctx
 * enqueued has finished.  Polls an event; returns TIMEOUT after timeout_ms, CUDA if the
 * work failed. */
int kvattn_tail_wait(kvattn_tail_ctx* ctx, int timeout_ms);

/* Read (and optionally clear) the sticky KVATTN_DEVICE_* bits of a decode or window+tail
 * workspace.  Synchronises `stream`. */
int kvattn_workspace_status(void* ws, uint32_t* flags, int clear, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVATTN_H */
