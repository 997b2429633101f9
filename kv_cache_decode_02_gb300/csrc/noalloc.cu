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
    // Every argument and size check (a call whose scratch would not fit the array is
    // refused with KVATTN_ERR_WORKSPACE) runs before the array's address is looked up and
    // before anything is put on the stream; the status word is then cleared on the stream
    // (the array keeps the previous call's bytes; descriptors and partials are rewritten).
    const kvattn::LibraryScratch scratch{(size_t)KVATTN_NOALLOC_SCRATCH_BYTES, scratch_address};
    return kvattn::decode_with_library_scratch(q, k_cache, v_cache, k_scales, v_scales, kv_type, n_cells, cell_plan,
                                               plan_stride, seq_lens, n_seq, max_len, n_head, n_head_kv, head_dim,
                                               split, scale, out, lse, scratch, stream);
}
