// Per-split descriptors of a compact cell plan ("KVARN KV Performance optimizations",
// item 5, descriptor setup with low-32-bit physical cells; item 6, fully masked split
// skipping).  For split p of sequence s, over plan entries [p*split, min((p+1)*split, L)):
//     {n_valid, lo, hi, flags}
// with an entry e valid when 0 <= e < n_cells, lo/hi the smallest/largest valid cell,
// flags 1 = no valid entry, 2 = linear (e - i is the same for every valid entry: one
// physical run with positional holes), 4 = an entry outside [-1, n_cells) seen,
// 8 = the split starts at or beyond L.  The quantised decode kernels read n_valid to skip a
// split before touching its plan entries or its K/V rows; the f16 decode kernels build the
// same descriptors in their producer warp instead (split_decode_body, desc_out).
//
// One warp per descriptor: lanes stride over the split's entries and reduce count,
// min, max and the min/max of (e - i) with shuffles, so no division sits in the scan.
#include <climits>

#include "kvattn_internal.cuh"

namespace kvattn {

namespace {

constexpr int kDescWarps = 8;

__global__ void __launch_bounds__(kDescWarps * 32)
    descriptor_kernel(const int32_t* __restrict__ plan, int64_t plan_stride,
                      const int32_t* __restrict__ seq_lens, int n_seq, int64_t max_len, int split,
                      int64_t n_cells, int64_t n_split, int4* __restrict__ desc, uint32_t* status) {
    pdl_launch_dependents();  // the decode kernel waits for this grid before reading desc
    pdl_wait();
    const int64_t id = (int64_t)blockIdx.x * kDescWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (id >= (int64_t)n_seq * n_split) return;
    const int s = (int)(id / n_split);
    const int64_t sp = id - (int64_t)s * n_split;
    int64_t L = seq_lens[s];
    L = L < 0 ? 0 : L;
    L = L < max_len ? L : max_len;
    L = L < plan_stride ? L : plan_stride;
    const int64_t i0 = sp * split;
    const int64_t i1 = (i0 + split < L) ? i0 + split : L;

    int count = 0;
    int lo = INT_MAX, hi = -1;
    long long off_lo = LLONG_MAX, off_hi = LLONG_MIN;
    bool bad = false;
    const int32_t* row = plan + (int64_t)s * plan_stride;
    for (int64_t i = i0 + lane; i < i1; i += 32) {
        const int32_t e = row[i];
        if (e >= 0 && (int64_t)e < n_cells) {
            ++count;
            lo = min(lo, e);
            hi = max(hi, e);
            const long long o = (long long)e - (long long)i;
            off_lo = min(off_lo, o);
            off_hi = max(off_hi, o);
        } else if (e != -1) {
            bad = true;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        count += __shfl_xor_sync(0xffffffffu, count, o);
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        off_lo = min(off_lo, __shfl_xor_sync(0xffffffffu, off_lo, o));
        off_hi = max(off_hi, __shfl_xor_sync(0xffffffffu, off_hi, o));
    }
    const bool any_bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
        int flags = 0;
        if (count == 0) flags |= 1;
        else if (off_lo == off_hi) flags |= 2;
        if (any_bad) flags |= 4;
        if (i0 >= L) flags |= 8;
        desc[id] = make_int4(count, count ? lo : -1, count ? hi : -1, flags);
        if (any_bad && status != nullptr) atomicOr(status, KVATTN_DEVICE_BAD_PLAN_ENTRY);
    }
}

}  // namespace

cudaError_t launch_descriptors(const int32_t* plan, int64_t plan_stride, const int32_t* seq_lens,
                               int n_seq, int64_t max_len, int split, int64_t n_cells,
                               int64_t n_split, int4* desc, uint32_t* status, cudaStream_t stream) {
    const int64_t total = (int64_t)n_seq * n_split;
    if (total == 0) return cudaSuccess;
    const int64_t blocks = (total + kDescWarps - 1) / kDescWarps;
    if (blocks > INT_MAX) return cudaErrorInvalidConfiguration;
    descriptor_kernel<<<(unsigned)blocks, kDescWarps * 32, 0, stream>>>(
        plan, plan_stride, seq_lens, n_seq, max_len, split, n_cells, n_split, desc, status);
    return cudaGetLastError();
}

}  // namespace kvattn
