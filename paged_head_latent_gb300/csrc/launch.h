// launch.h -- host-side launchers, one per kernel translation unit.
#pragma once
#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {

// CUDA-core attention kernel (16 heads per CTA), same partition and outputs as the
// tensor-core kernel: whole rows to out/lse, split rows' fragments to the workspace,
// and each worker's combine record.
cudaError_t launch_simt(const MlaParams& p, cudaStream_t stream);
// Merge of split rows' fragments (one CTA per worker and head).
cudaError_t launch_combine(const MlaParams& p, cudaStream_t stream);
// Optional index validation (sets the status word; never traps).
cudaError_t launch_validate(const MlaParams& p, cudaStream_t stream);

}  // namespace mla
