// kvattn_decode_noalloc: kvattn_decode for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where they run
// decode attention: code that executes inside a memory pool's fixed budget, plugins
// handed only the input and output buffers by a host framework, or real-time paths that
// must not block on the driver's allocator.  This entry point serves them: it takes the
// same inputs and outputs as kvattn_decode, and keeps its scratch (the status word, the
// per-split descriptors and the partial results) in one array that lives in the
// library's own device memory for as long as the library is loaded.
//
// The array is a file-scope __device__ object.  Its name means nothing to host code (the
// host sees only a stand-in), so the host looks up the array's real device address with
// cudaGetSymbolAddress, once per device, on that device, the first time this entry point
// is called there, and passes that address on.  Nothing here allocates.
#include <mutex>

#include "kvattn_internal.cuh"

namespace {

// Scratch shared by every kvattn_decode_noalloc call on a device.  Zero at load time.
__device__ __align__(256) unsigned char g_decode_scratch[KVATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_decode_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** ptr) {
    static std::once_flag once[kMaxDevices];
    static void* addr[kMaxDevices];
    static cudaError_t err[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [dev] {
        void* p = nullptr;
        err[dev] = cudaGetSymbolAddress(&p, g_decode_scratch);
        addr[dev] = err[dev] == cudaSuccess ? p : nullptr;
    });
    *ptr = addr[dev];
    return err[dev];
}

}  // namespace

extern "C" int kvattn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                     const void* k_scales, const void* v_scales, int kv_type,
                                     int64_t n_cells, const int32_t* cell_plan, int64_t plan_stride,
                                     const int32_t* seq_lens, int n_seq, int64_t max_len, int n_head,
                                     int n_head_kv, int head_dim, int split, float scale, float* out,
                                     float* lse, void* stream) {
    if (split == 0) {  // the split kvattn_decode would select (a host-side query)
        split = kvattn_select_split(kv_type, n_seq, max_len, n_head_kv, head_dim);
        if (split < 0) return split;
    }
    // Refuse, before any work reaches the device, a call whose scratch would not fit.
    const size_t need = kvattn_decode_workspace_bytes(n_seq, n_head, head_dim, max_len, split);
    if (need == 0) return KVATTN_ERR_INVALID_ARG;
    if (need > (size_t)KVATTN_NOALLOC_SCRATCH_BYTES) return KVATTN_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess || scratch == nullptr) return KVATTN_ERR_CUDA;
    // The scratch keeps the previous call's contents; only the status word must start at
    // zero (descriptors and partials are fully rewritten by every call).
    if (cudaMemsetAsync(scratch, 0, kvattn::kStatusBytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KVATTN_ERR_CUDA;
    return kvattn_decode(q, k_cache, v_cache, k_scales, v_scales, kv_type, n_cells, cell_plan, plan_stride,
                         seq_lens, n_seq, max_len, n_head, n_head_kv, head_dim, split, scale, out, lse, scratch,
                         (size_t)KVATTN_NOALLOC_SCRATCH_BYTES, stream);
}
