// LSE-weighted merge of partial attention results ("KVARN KV Performance optimizations",
// item 9: partial windows keep the online-softmax maximum, numerator and denominator and
// are merged afterwards; "Rolling-KV -- overflow throughput evaluations", section 3: the
// decode op's LSE channel).  For one output row:
//     M = max_p LSE_p,  w_p = exp(LSE_p - M),
//     O = sum_p w_p O_p / sum_p w_p,  LSE = M + ln sum_p w_p.
// Parts with LSE = -inf carry no cells; they get weight 0 and their O is never read.
//
// One CTA of 8 warps per row.  Latency, not bandwidth, bounds this kernel (a row has a
// few KB to a few MB of partials sitting in L2), so it avoids dependent load chains.
//  * partials written by the decode kernels (every O written, 0 for empty parts): warp w
//    reads parts w, w+8, ... eight (head_dim 256: four) at a time, LSE and O in the same
//    round, and keeps a running (max, sum, O); the warps are then combined with the same
//    rescaling.
//  * caller partials (kvattn_merge: an empty part's O may be anything): pass 1 loads every
//    LSE in parallel and reduces the maximum, pass 2 turns them into weights in shared
//    memory, pass 3 sums the O rows of non-empty parts only, several loads in flight.
#include <cmath>

#include "kvattn_internal.cuh"

namespace kvattn {

namespace {

constexpr int kMergeWarps = 8;
constexpr int kMergeThreads = kMergeWarps * 32;
constexpr int kMaxChunks = 8;      // head_dim <= 1024: float4 chunks per lane (public merge)
constexpr int kWeightCache = 4096; // parts whose weights stay in shared memory

// Partials written by the decode kernels: warp w reads parts w, w + 8, ... BATCH at a time,
// LSE and O in the same round of independent loads (an empty part's O is 0), and folds
// them into a running (max, sum, O) with the decode kernel's rescaling.  CPL: float4 chunks
// of a row per lane; each round keeps BATCH x CPL loads in flight per lane.
template <int WARPS, int CPL, int BATCH>
__device__ __forceinline__ void merge_written_rounds(const float* lse_base, const float* o_base, int64_t lse_stride,
                                                     int64_t o_stride, int64_t n_parts, int chunks, int warp, int lane,
                                                     float& mw, float& sw, float4 (&acc)[2]) {
    for (int64_t q0 = warp; q0 < n_parts; q0 += (int64_t)WARPS * BATCH) {
        float l[BATCH];
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int64_t q = q0 + (int64_t)u * WARPS;
            l[u] = q < n_parts ? __ldg(lse_base + q * lse_stride) : -INFINITY;
        }
        float4 v[BATCH][CPL];
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int64_t q = q0 + (int64_t)u * WARPS;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const int ci = lane + 32 * c;
                v[u][c] = (q < n_parts && ci < chunks)
                              ? __ldg(reinterpret_cast<const float4*>(o_base + q * o_stride) + ci)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float bm = -INFINITY;
#pragma unroll
        for (int u = 0; u < BATCH; ++u) bm = fmaxf(bm, l[u]);
        const float nm = fmaxf(mw, bm);
        if (nm == -INFINITY) continue;
        const float keep = __expf(mw - nm);  // 0 when nothing was accumulated yet
        sw *= keep;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            acc[c].x *= keep;
            acc[c].y *= keep;
            acc[c].z *= keep;
            acc[c].w *= keep;
        }
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const float w = l[u] == -INFINITY ? 0.f : __expf(l[u] - nm);
            sw += w;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                acc[c].x = fmaf(w, v[u][c].x, acc[c].x);
                acc[c].y = fmaf(w, v[u][c].y, acc[c].y);
                acc[c].z = fmaf(w, v[u][c].z, acc[c].z);
                acc[c].w = fmaf(w, v[u][c].w, acc[c].w);
            }
        }
        mw = nm;
    }
}

template <int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 16 / WARPS) merge_kernel(const MergeParams p) {
    __shared__ float red[WARPS];
    __shared__ float wts[kWeightCache];
    extern __shared__ float4 acc_smem[];  // [warps][head_dim / 4]

    // let the next kernel start its prologue; it waits for this grid before reading
    pdl_launch_dependents();
    pdl_wait();
    const int row = blockIdx.x;  // s * n_rows + h
    const int s = row / p.n_rows;
    const int h = row - s * p.n_rows;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int chunks = p.head_dim / 4;

    int64_t n_parts = p.n_parts;
    if (p.seq_lens != nullptr) {
        int64_t L = p.seq_lens[s];
        L = L < 0 ? 0 : L;
        L = L < p.max_len ? L : p.max_len;
        L = L < p.len_cap ? L : p.len_cap;
        n_parts = (L + p.split - 1) / p.split;
    }
    const float* lse_base = p.part_lse + (int64_t)s * p.n_parts * p.n_rows + h;
    const float* o_base = p.part_o + ((int64_t)s * p.n_parts * p.n_rows + h) * p.head_dim;
    const int64_t lse_stride = p.n_rows;
    const int64_t o_stride = (int64_t)p.n_rows * p.head_dim;

    if (p.all_written) {
        float mw = -INFINITY, sw = 0.f;
        float4 acc[2];  // decode partials: head_dim <= 256, at most two float4 chunks per lane
        acc[0] = acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        // head_dim <= 128: one float4 per lane and part, eight parts a round; 256: two, four.
        // 128 registers, two CTAs per SM: the 192 rows of a four-sequence GQA-6 plan merge in
        // one wave (105.3 -> 103.4 us for the whole op), and a CTA launched early under
        // programmatic dependence leaves room for two decode CTAs of the next call beside it
        // while it waits (at 244 registers it left none: 14.7 -> 16.2 us per Qwen3-8B layer).
        if (chunks <= 32)
            merge_written_rounds<WARPS, 1, 8>(lse_base, o_base, lse_stride, o_stride, n_parts, chunks, warp, lane, mw, sw,
                                        acc);
        else
            merge_written_rounds<WARPS, 2, 4>(lse_base, o_base, lse_stride, o_stride, n_parts, chunks, warp, lane, mw, sw,
                                       acc);
        if (lane == 0) {
            red[warp] = mw;
            wts[warp] = sw;
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int ci = lane + 32 * c;
            if (ci < chunks) acc_smem[warp * chunks + ci] = acc[c];
        }
        __syncthreads();
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) M = fmaxf(M, red[w]);
        float W = 0.f;
        float scw[WARPS];
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            scw[w] = (M == -INFINITY || red[w] == -INFINITY) ? 0.f : __expf(red[w] - M);
            W = fmaf(scw[w], wts[w], W);
        }
        float4* out = reinterpret_cast<float4*>(p.out + (int64_t)row * p.head_dim);
        for (int ci = threadIdx.x; ci < chunks; ci += (WARPS * 32)) {
            float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
            if (W > 0.f) {
#pragma unroll
                for (int w = 0; w < WARPS; ++w) {
                    const float4 a = acc_smem[w * chunks + ci];
                    t.x = fmaf(scw[w], a.x, t.x);
                    t.y = fmaf(scw[w], a.y, t.y);
                    t.z = fmaf(scw[w], a.z, t.z);
                    t.w = fmaf(scw[w], a.w, t.w);
                }
                const float inv = 1.f / W;
                t.x *= inv;
                t.y *= inv;
                t.z *= inv;
                t.w *= inv;
            }
            out[ci] = t;
        }
        if (threadIdx.x == 0) p.lse[row] = (W > 0.f) ? M + __logf(W) : -INFINITY;
        return;
    }

    // pass 1: maximum LSE (all loads independent)
    float m = -INFINITY;
    for (int64_t q = threadIdx.x; q < n_parts; q += (WARPS * 32)) {
        const float l = __ldg(lse_base + q * lse_stride);
        if (q < kWeightCache) wts[q] = l;
        m = fmaxf(m, l);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    float M = red[0];
#pragma unroll
    for (int w = 1; w < WARPS; ++w) M = fmaxf(M, red[w]);
    __syncthreads();

    // pass 2: weights exp(LSE_p - M) (0 for empty parts) and their sum
    float wsum = 0.f;
    if (M != -INFINITY) {
        for (int64_t q = threadIdx.x; q < n_parts; q += (WARPS * 32)) {
            const float l = q < kWeightCache ? wts[q] : __ldg(lse_base + q * lse_stride);
            const float w = (l == -INFINITY) ? 0.f : __expf(l - M);
            if (q < kWeightCache) wts[q] = w;
            wsum += w;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    if (lane == 0) red[warp] = wsum;
    __syncthreads();
    float W = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) W += red[w];

    // pass 3: weighted sum of the O rows
    float4 acc[kMaxChunks];
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (W > 0.f) {
        constexpr int kUnroll = 4;
        for (int64_t q0 = warp; q0 < n_parts; q0 += WARPS * kUnroll) {
            float w[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t q = q0 + (int64_t)u * WARPS;
                float wq = 0.f;
                if (q < n_parts) {
                    if (q < kWeightCache) {
                        wq = wts[q];
                    } else {
                        const float l = __ldg(lse_base + q * lse_stride);
                        wq = (l == -INFINITY) ? 0.f : __expf(l - M);
                    }
                }
                w[u] = wq;
            }
#pragma unroll
            for (int c = 0; c < kMaxChunks; ++c) {
                const int ci = lane + 32 * c;
                if (ci < chunks) {
                    float4 v[kUnroll];
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u) {
                        const int64_t q = q0 + (int64_t)u * WARPS;
                        v[u] = w[u] != 0.f ? __ldg(reinterpret_cast<const float4*>(o_base + q * o_stride) + ci)
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u) {
                        acc[c].x = fmaf(w[u], v[u].x, acc[c].x);
                        acc[c].y = fmaf(w[u], v[u].y, acc[c].y);
                        acc[c].z = fmaf(w[u], v[u].z, acc[c].z);
                        acc[c].w = fmaf(w[u], v[u].w, acc[c].w);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) {
        const int ci = lane + 32 * c;
        if (ci < chunks) acc_smem[warp * chunks + ci] = acc[c];
    }
    __syncthreads();
    float4* out = reinterpret_cast<float4*>(p.out + (int64_t)row * p.head_dim);
    for (int ci = threadIdx.x; ci < chunks; ci += (WARPS * 32)) {
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
        if (W > 0.f) {
#pragma unroll
            for (int w = 0; w < WARPS; ++w) {
                const float4 v = acc_smem[w * chunks + ci];
                t.x += v.x;
                t.y += v.y;
                t.z += v.z;
                t.w += v.w;
            }
            const float inv = 1.f / W;
            t.x *= inv;
            t.y *= inv;
            t.z *= inv;
            t.w *= inv;
        }
        out[ci] = t;
    }
    if (threadIdx.x == 0) p.lse[row] = (W > 0.f) ? M + __logf(W) : -INFINITY;
}

// Decode partials of rows with many parts, one row spread over several CTAs: CTA (row,
// slice) merges float4 chunks [slice CW, slice CW + CW) of the row's O over all parts
// (CW = 8, 16 or 32; each
// CTA reads every LSE and computes the same weights).  Lanes form 32 / CW groups of CW
// lanes; group k of warp w reads parts w G + k, w G + k + WARPS G, ... (G groups a warp),
// BATCH parts per group and round, so one load instruction covers G parts.  The groups of a
// warp, then the warps, combine their (max, sum, O) with the usual rescaling.
template <int WARPS, int CW, int BATCH>
__global__ void __launch_bounds__(WARPS * 32) merge_slices_kernel(const MergeParams p) {
    constexpr int G = 32 / CW;
    __shared__ float red_m[WARPS], red_s[WARPS];
    __shared__ float4 acc_smem[WARPS][CW];
    pdl_launch_dependents();
    pdl_wait();
    const int row = blockIdx.x;  // s * n_rows + h
    const int s = row / p.n_rows;
    const int h = row - s * p.n_rows;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int grp = lane / CW;
    const int c = blockIdx.y * CW + (lane - grp * CW);  // this lane's float4 chunk of the row

    int64_t n_parts = p.n_parts;
    if (p.seq_lens != nullptr) {
        int64_t L = p.seq_lens[s];
        L = L < 0 ? 0 : L;
        L = L < p.max_len ? L : p.max_len;
        L = L < p.len_cap ? L : p.len_cap;
        n_parts = (L + p.split - 1) / p.split;
    }
    const float* lse_base = p.part_lse + (int64_t)s * p.n_parts * p.n_rows + h;
    const float4* o_base =
        reinterpret_cast<const float4*>(p.part_o + ((int64_t)s * p.n_parts * p.n_rows + h) * p.head_dim) + c;
    const int64_t lse_stride = p.n_rows;
    const int64_t o_stride = (int64_t)p.n_rows * p.head_dim / 4;  // in float4

    float mw = -INFINITY, sw = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t q0 = (int64_t)warp * G + grp; q0 < n_parts; q0 += (int64_t)WARPS * G * BATCH) {
        float l[BATCH];
        float4 v[BATCH];
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int64_t q = q0 + (int64_t)u * WARPS * G;
            l[u] = q < n_parts ? __ldg(lse_base + q * lse_stride) : -INFINITY;
            v[u] = q < n_parts ? __ldg(o_base + q * o_stride) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float bm = -INFINITY;
#pragma unroll
        for (int u = 0; u < BATCH; ++u) bm = fmaxf(bm, l[u]);
        const float nm = fmaxf(mw, bm);
        if (nm == -INFINITY) continue;
        const float keep = __expf(mw - nm);  // 0 when nothing was accumulated yet
        sw *= keep;
        acc.x *= keep;
        acc.y *= keep;
        acc.z *= keep;
        acc.w *= keep;
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const float w = l[u] == -INFINITY ? 0.f : __expf(l[u] - nm);
            sw += w;
            acc.x = fmaf(w, v[u].x, acc.x);
            acc.y = fmaf(w, v[u].y, acc.y);
            acc.z = fmaf(w, v[u].z, acc.z);
            acc.w = fmaf(w, v[u].w, acc.w);
        }
        mw = nm;
    }
    // the lane groups of the warp (lanes CW apart hold the same chunk)
#pragma unroll
    for (int o = 16; o >= CW; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, mw, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, sw, o);
        float4 a2;
        a2.x = __shfl_xor_sync(0xffffffffu, acc.x, o);
        a2.y = __shfl_xor_sync(0xffffffffu, acc.y, o);
        a2.z = __shfl_xor_sync(0xffffffffu, acc.z, o);
        a2.w = __shfl_xor_sync(0xffffffffu, acc.w, o);
        const float nm = fmaxf(mw, m2);
        const float f1 = mw == -INFINITY ? 0.f : __expf(mw - nm);
        const float f2 = m2 == -INFINITY ? 0.f : __expf(m2 - nm);
        sw = sw * f1 + s2 * f2;
        acc.x = acc.x * f1 + a2.x * f2;
        acc.y = acc.y * f1 + a2.y * f2;
        acc.z = acc.z * f1 + a2.z * f2;
        acc.w = acc.w * f1 + a2.w * f2;
        mw = nm;
    }
    if (lane == 0) {
        red_m[warp] = mw;
        red_s[warp] = sw;
    }
    if (lane < CW) acc_smem[warp][lane] = acc;
    __syncthreads();
    if (threadIdx.x < CW) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) M = fmaxf(M, red_m[w]);
        float W = 0.f;
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < WARPS; ++w) {
                const float f = red_m[w] == -INFINITY ? 0.f : __expf(red_m[w] - M);
                W = fmaf(f, red_s[w], W);
                const float4 a = acc_smem[w][threadIdx.x];
                t.x = fmaf(f, a.x, t.x);
                t.y = fmaf(f, a.y, t.y);
                t.z = fmaf(f, a.z, t.z);
                t.w = fmaf(f, a.w, t.w);
            }
        }
        const float inv = W > 0.f ? 1.f / W : 0.f;
        t.x *= inv;
        t.y *= inv;
        t.z *= inv;
        t.w *= inv;
        reinterpret_cast<float4*>(p.out + (int64_t)row * p.head_dim)[blockIdx.y * CW + threadIdx.x] = t;
        if (blockIdx.y == 0 && threadIdx.x == 0) p.lse[row] = (W > 0.f) ? M + __logf(W) : -INFINITY;
    }
}

}  // namespace

cudaError_t launch_merge(const MergeParams& params, cudaStream_t stream, bool pdl) {
    MergeParams p = params;
    if (p.head_dim > 256) p.all_written = 0;  // the one-round path holds two float4 per lane
    const int64_t rows = (int64_t)p.n_seq * p.n_rows;  // one CTA per row, numbered in 32 bits
    if (rows == 0) return cudaSuccess;
    if (rows > (int64_t)INT32_MAX) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.stream = stream;
    // Decode partials of head_dim-128 rows with more parts than one round of a CTA (64) and
    // too few rows to fill the SMs: each row's head_dim is split over several CTAs (slices of
    // 8 to 32 float4 chunks, at most one CTA per SM in all), so that more SMs read the parts
    // from L2 at once (Q8_0 over 131072 cells at split 512, 256 parts a row: 66.2 -> 64.9 us
    // per op).  At head_dim 256 the same split measured slower (114.7 -> 122.7 us), so those
    // rows keep one CTA each.
    const int chunks = p.head_dim / 4;
    if (p.all_written && p.allow_slices && p.head_dim == 128 && p.n_parts > 64) {
        int slices = chunks / 8;
        while (slices > 1 && rows * slices > p.wide_rows_max) slices >>= 1;
        const int cw = chunks / slices;  // float4 chunks per slice: 8, 16 or 32
        if (slices > 1 && chunks % slices == 0 && cw <= 32 && rows * (int64_t)slices <= (int64_t)INT32_MAX) {
            cfg.gridDim = dim3((unsigned)rows, (unsigned)slices, 1);
            cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
            cfg.dynamicSmemBytes = 0;
            if (cw == 8) return cudaLaunchKernelEx(&cfg, merge_slices_kernel<kMergeWarps, 8, 8>, p);
            if (cw == 16) return cudaLaunchKernelEx(&cfg, merge_slices_kernel<kMergeWarps, 16, 8>, p);
            return cudaLaunchKernelEx(&cfg, merge_slices_kernel<kMergeWarps, 32, 8>, p);
        }
    }
    cfg.gridDim = dim3((unsigned)rows, 1, 1);
    // Rows of decode partials with more than one round of parts for 8 warps (64 parts at
    // head_dim <= 128, 32 at 256) take 16 warps, half the dependent rounds of loads, when
    // the rows fit one CTA per SM (such a CTA holds a whole SM's registers, so it runs only
    // on SMs the decode has left; two waves of them would cost more than the rounds saved).
    const int64_t round8 = (int64_t)kMergeWarps * (p.head_dim <= 128 ? 8 : 4);
    const bool wide = p.all_written && p.n_parts > round8 && rows <= p.wide_rows_max;
    const int warps = wide ? 2 * kMergeWarps : kMergeWarps;
    cfg.blockDim = dim3(warps * 32, 1, 1);
    cfg.dynamicSmemBytes = warps * p.head_dim * sizeof(float);
    return wide ? cudaLaunchKernelEx(&cfg, merge_kernel<2 * kMergeWarps>, p)
                : cudaLaunchKernelEx(&cfg, merge_kernel<kMergeWarps>, p);
}

}  // namespace kvattn
