// tc_kernel.h -- TMA descriptors and launcher of the tensor-core attention kernel.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {

// 2-D bf16 tensor maps, 128-byte swizzle, 64-column boxes.
struct TmaMaps {
  CUtensorMap q_nope;  // [rows*H, 512], box 64 x 128 (all heads of one query row)
  CUtensorMap q_pe;    // [rows*H, 64],  box 64 x 128
  CUtensorMap ckv;     // [slots, 512],  box 64 x 64 (a whole 64-slot page)
  CUtensorMap kpe;     // [slots, 64],   box 64 x 64
  CUtensorMap ckv_g;   // [slots, 512],  box 64 x 1 (tile::gather4 rows)
  CUtensorMap kpe_g;   // [slots, 64],   box 64 x 1
};

cudaError_t launch_tc(const TmaMaps& maps, const MlaParams& p, cudaStream_t stream);
uint32_t tc_smem_bytes();

}  // namespace mla
