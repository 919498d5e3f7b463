// launch.h -- host-side launchers, one per kernel translation unit.
#pragma once
#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {

// Merge of split rows' fragments (one warp per worker record and head).
cudaError_t launch_combine(const MlaParams& p, cudaStream_t stream);
// Optional index validation (sets the status word; never traps).
cudaError_t launch_validate(const MlaParams& p, cudaStream_t stream);
// Block table + sequence lengths -> token-slot CSR (two kernels on `stream`).
cudaError_t launch_block_table_csr(const int32_t* block_table, const int32_t* seq_lens, int batch, int max_blocks,
                                   int page_size, int32_t* kv_indptr, int32_t* kv_indices, long long capacity,
                                   cudaStream_t stream);

}  // namespace mla
