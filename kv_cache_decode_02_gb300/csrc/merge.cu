// LSE-weighted merge of partial attention results ("KVARN KV Performance optimizations",
// item 9: partial windows keep the online-softmax maximum, numerator and denominator and
// are merged afterwards; "Rolling-KV -- overflow throughput evaluations", section 3: the
// decode op's LSE channel).  For one output row:
//     M = max_p LSE_p,  w_p = exp(LSE_p - M),
//     O = sum_p w_p O_p / sum_p w_p,  LSE = M + ln sum_p w_p.
// Parts with LSE = -inf carry no cells; they are skipped and their O is never read.
//
// One CTA of 8 warps per row; warp w takes parts w, w+8, ...; each lane owns float4
// chunks of head_dim, so every part's O row is read with coalesced 16-byte loads.
#include <cmath>

#include "kvattn_internal.cuh"

namespace kvattn {

namespace {

constexpr int kMergeWarps = 8;
constexpr int kMaxChunks = 8;  // head_dim <= 1024

__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const MergeParams p) {
    __shared__ float red_m[kMergeWarps];
    __shared__ float red_w[kMergeWarps];
    extern __shared__ float4 acc_smem[];  // [warps][head_dim / 4]

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

    // pass 1: the row maximum over the parts
    float m = -INFINITY;
    for (int64_t q = warp * 32 + lane; q < n_parts; q += kMergeWarps * 32) m = fmaxf(m, lse_base[q * lse_stride]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red_m[warp] = m;
    __syncthreads();
    float M = red_m[0];
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w) M = fmaxf(M, red_m[w]);

    // pass 2: weighted sums
    float4 acc[kMaxChunks];
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (M != -INFINITY) {
        for (int64_t q = warp; q < n_parts; q += kMergeWarps) {
            const float l = lse_base[q * lse_stride];
            if (l == -INFINITY) continue;
            const float w = __expf(l - M);
            wsum += w;
            const float4* src = reinterpret_cast<const float4*>(o_base + q * o_stride);
#pragma unroll
            for (int c = 0; c < kMaxChunks; ++c) {
                const int ci = lane + 32 * c;
                if (ci < chunks) {
                    const float4 v = __ldg(src + ci);
                    acc[c].x = fmaf(w, v.x, acc[c].x);
                    acc[c].y = fmaf(w, v.y, acc[c].y);
                    acc[c].z = fmaf(w, v.z, acc[c].z);
                    acc[c].w = fmaf(w, v.w, acc[c].w);
                }
            }
        }
    }
    if (lane == 0) red_w[warp] = wsum;
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) {
        const int ci = lane + 32 * c;
        if (ci < chunks) acc_smem[warp * chunks + ci] = acc[c];
    }
    __syncthreads();
    float W = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) W += red_w[w];
    float4* out = reinterpret_cast<float4*>(p.out + (int64_t)row * p.head_dim);
    for (int ci = threadIdx.x; ci < chunks; ci += kMergeWarps * 32) {
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
        if (W > 0.f) {
#pragma unroll
            for (int w = 0; w < kMergeWarps; ++w) {
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
    pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream, bool pdl) {
    const int rows = p.n_seq * p.n_rows;
    if (rows == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rows, 1, 1);
    cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = kMergeWarps * p.head_dim * sizeof(float);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, merge_kernel, p);
}

}  // namespace kvattn
