// launch.h -- host-side launchers, one per kernel translation unit.
#pragma once
#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {

// Merge of split rows' fragments (one warp per worker record and head).
cudaError_t launch_combine(const MlaParams& p, cudaStream_t stream);
// Optional index validation (sets the status word; never traps).
cudaError_t launch_validate(const MlaParams& p, cudaStream_t stream);

}  // namespace mla
