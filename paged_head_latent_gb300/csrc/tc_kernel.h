// tc_kernel.h -- TMA descriptors and launcher of the tensor-core attention kernel.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {

// 2-D bf16 tensor maps (box = columns x rows).
struct TmaMaps {
  CUtensorMap ckv;  // [slots, 512], box 64 x 64, 128-byte swizzle (a whole run of 64 slots)
  CUtensorMap kpe;  // [slots, 64],  box 32 x 64, 64-byte swizzle (half of the positional dims)
  // FP8 cache as [slots, 656] bytes: latent boxes 128 B x 64 tokens, scale boxes
  // 16 B x 32 tokens, rope boxes 64 B x 64 tokens (64-byte swizzle).
  CUtensorMap f8_lat;
  CUtensorMap f8_scl;
  CUtensorMap f8_rope;
};

// gather: the cache's page size is not a multiple of 64 (tiles are copied slot by slot).
cudaError_t launch_tc(const TmaMaps& maps, const MlaParams& p, bool gather, cudaStream_t stream);
uint32_t tc_smem_bytes();

}  // namespace mla
