// mla_combine.cu -- merge of split-KV fragments, and the optional index validation.
//
// Merge (Modular MAX "mla_decoding_single_batch": split-K partitions leave exp-sum
// and max statistics that a reduction merges): for a row split into fragments
// f = 1..F with base-2 lse_f and normalised outputs o_f,
//   lse = log2(sum_f 2^lse_f),   out = sum_f 2^(lse_f - lse) * o_f,
// summed in worker order, so the result does not depend on timing.
#include "common.cuh"
#include "launch.h"

namespace mla {

constexpr int kCombineThreads = 128;  // 128 threads x 4 dims = 512

__global__ void __launch_bounds__(kCombineThreads) mla_combine_kernel(MlaParams p) {
  const int w = blockIdx.x;
  const int h = blockIdx.y;
  const CombineRecord rec = p.records[w];
  if (rec.row < 0 || h >= p.heads) return;
  const long long T = rec.total_tiles;
  const int G = p.workers;
  float mx = -INFINITY;
  for (int f = rec.w_first; f <= w; ++f) {
    if (worker_start(f + 1, T, G) == worker_start(f, T, G)) continue;  // empty range
    const int slot = (f == rec.w_first) ? rec.slot_first : 0;
    mx = fmaxf(mx, p.part_lse[((size_t)f * 2 + slot) * p.heads + h]);
  }
  float sum = 0.f;
  for (int f = rec.w_first; f <= w; ++f) {
    if (worker_start(f + 1, T, G) == worker_start(f, T, G)) continue;
    const int slot = (f == rec.w_first) ? rec.slot_first : 0;
    sum += fast_exp2(p.part_lse[((size_t)f * 2 + slot) * p.heads + h] - mx);
  }
  const float lse2 = mx + fast_log2(sum);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int f = rec.w_first; f <= w; ++f) {
    if (worker_start(f + 1, T, G) == worker_start(f, T, G)) continue;
    const int slot = (f == rec.w_first) ? rec.slot_first : 0;
    const size_t frag = ((size_t)f * 2 + slot) * p.heads + h;
    const float wgt = fast_exp2(p.part_lse[frag] - lse2);
    const float4 v = reinterpret_cast<const float4*>(p.part_o + frag * kDimCkv)[threadIdx.x];
    acc.x = fmaf(wgt, v.x, acc.x);
    acc.y = fmaf(wgt, v.y, acc.y);
    acc.z = fmaf(wgt, v.z, acc.z);
    acc.w = fmaf(wgt, v.w, acc.w);
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&lo);
  packed.y = *reinterpret_cast<uint32_t*>(&hi);
  __nv_bfloat16* dst = p.out + ((size_t)rec.row * p.heads + h) * kDimCkv;
  reinterpret_cast<uint2*>(dst)[threadIdx.x] = packed;
  if (threadIdx.x == 0) p.lse[(size_t)rec.row * p.heads + h] = lse2 * 0.69314718055994531f;
}

// Index validation (flashinfer's "validate" switch on its planned wrapper inspired it):
// indptr starts at 0, is non-decreasing, ends at num_kv_indices (and total_q for
// qo_indptr), every request has kv_len >= q_len, every index is a slot of the cache.
// Sets kStatusBadIndex in the status word; never traps.
__global__ void mla_validate_kernel(MlaParams p) {
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  const int nthreads = gridDim.x * blockDim.x;
  bool bad = false;
  for (int b = tid; b <= p.batch; b += nthreads) {
    const int k = p.kv_indptr[b];
    if (b == 0 && k != 0) bad = true;
    if (b == p.batch && k != p.num_kv_indices) bad = true;
    if (b < p.batch) {
      const int k1 = p.kv_indptr[b + 1];
      if (k1 < k) bad = true;
      if (p.qo_indptr) {
        const int q0 = p.qo_indptr[b], q1 = p.qo_indptr[b + 1];
        if (q1 < q0 || (k1 - k) < (q1 - q0)) bad = true;
      }
    }
    if (p.qo_indptr) {
      const int q = p.qo_indptr[b];
      if (b == 0 && q != 0) bad = true;
      if (b == p.batch && q != p.rows) bad = true;
    }
  }
  for (int i = tid; i < p.num_kv_indices; i += nthreads) {
    const int s = p.kv_indices[i];
    if (s < 0 || s >= p.num_slots) bad = true;
  }
  if (bad) atomicOr(p.status, kStatusBadIndex);
}

cudaError_t launch_combine(const MlaParams& p, cudaStream_t stream) {
  mla_combine_kernel<<<dim3(p.workers, p.heads), kCombineThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_validate(const MlaParams& p, cudaStream_t stream) {
  mla_validate_kernel<<<64, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
