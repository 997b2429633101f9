// Tail tile copy for the window + tail path ("Rolling-KV -- overflow throughput
// evaluations", sections 1 and 5c: the host-resident tail streams to the device tile by
// tile on a side stream, double-buffered).  On a host whose pinned memory the GPU reads
// coherently (Grace + GB300 over NVLink-C2C), a kernel of 16-byte loads moves a tile at the
// link's full rate, while each cudaMemcpyAsync carries a fixed cost of a few microseconds
// that 1 MiB tiles cannot hide.  One launch moves a tile's K and V rows.
#include "kvattn_internal.cuh"

namespace kvattn {

namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 8;  // 16-byte loads in flight per thread
constexpr int64_t kMaxCopyBlocks = 32;

__global__ void __launch_bounds__(kCopyThreads) tile_copy_kernel(const uint4* __restrict__ k_src,
                                                                 const uint4* __restrict__ v_src,
                                                                 uint4* __restrict__ k_dst, uint4* __restrict__ v_dst,
                                                                 int64_t n16) {
    const int64_t stride = (int64_t)gridDim.x * kCopyThreads;
    for (int64_t base = (int64_t)blockIdx.x * kCopyThreads + threadIdx.x; base < n16;
         base += stride * kCopyUnroll) {
        uint4 k[kCopyUnroll], v[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t i = base + (int64_t)u * stride;
            if (i < n16) {
                k[u] = __ldg(k_src + i);
                v[u] = __ldg(v_src + i);
            }
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t i = base + (int64_t)u * stride;
            if (i < n16) {
                k_dst[i] = k[u];
                v_dst[i] = v[u];
            }
        }
    }
}

}  // namespace

cudaError_t launch_tile_copy(const void* k_src, const void* v_src, void* k_dst, void* v_dst, size_t bytes,
                             cudaStream_t stream) {
    const int64_t n16 = (int64_t)(bytes / 16);
    if (n16 == 0) return cudaSuccess;
    // One CTA per 64 KiB of the tile pair, at most 32: 2 MiB in flight is ten link round
    // trips' worth, and a larger tile loops rather than holding more SM slots (the tile
    // decodes and the next window decode run beside the copy).  Measured on a 36-layer stack
    // with one 8.6 MB tile per layer: 0.91 of the link at 32 CTAs, 0.89 at 64, 0.85 at 269.
    int64_t blocks = (n16 + (int64_t)kCopyThreads * kCopyUnroll - 1) / ((int64_t)kCopyThreads * kCopyUnroll);
    blocks = blocks < 1 ? 1 : (blocks > kMaxCopyBlocks ? kMaxCopyBlocks : blocks);
    tile_copy_kernel<<<(unsigned)blocks, kCopyThreads, 0, stream>>>(
        static_cast<const uint4*>(k_src), static_cast<const uint4*>(v_src), static_cast<uint4*>(k_dst),
        static_cast<uint4*>(v_dst), n16);
    return cudaGetLastError();
}

}  // namespace kvattn
