// Causal multi-query decode on the fifth-generation tensor cores (decode_tc.cu).
#pragma once

#include "kvattn_internal.cuh"

namespace kvattn {

// f16 cache, head_dim 128, up to 128 query rows per KV head in one work unit.
constexpr int kTcMaxRows = 128;

// Launches the tcgen05 multi-query kernel over n_seq x unit_splits x n_head_kv units (the
// fields of p as for launch_split_decode; p.n_stages is ignored).
cudaError_t launch_split_decode_tc(const SplitDecodeParams& p, unsigned grid_ctas, cudaStream_t stream, bool pdl);
// Resident CTAs per SM of that kernel.
cudaError_t split_decode_tc_occupancy(int* blocks);

}  // namespace kvattn
