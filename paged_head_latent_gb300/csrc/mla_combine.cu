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

constexpr int kCombineWarps = 8;  // one warp per head, 8 heads per CTA
constexpr int kCombineThreads = 32 * kCombineWarps;

// Fragment f (0-based, worker w_first + f) of a record: its slot index in the workspace,
// or -1 if that worker has an empty range (possible only when tiles < workers).
__device__ __forceinline__ long long frag_index(const CombineRecord& rec, int f, int G) {
  const int wk = rec.w_first + f;
  const long long T = rec.total_tiles;
  // Every worker has at least one tile when T >= G, so the division is needed only below.
  if (T < G && worker_start(wk + 1, T, G) == worker_start(wk, T, G)) return -1;
  return (long long)wk * 2 + (f == 0 ? rec.slot_first : 0);
}

__global__ void __launch_bounds__(kCombineThreads) mla_combine_kernel(MlaParams p) {
  const int w = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * kCombineWarps + warp;
  const CombineRecord rec = p.records[w];
  if (rec.row < 0 || h >= p.heads) return;
  const int G = p.workers;
  const int F = w - rec.w_first + 1;
  // Pass 1: lse of every fragment (lanes in parallel), max and sum by warp shuffles.
  float mx = -INFINITY;
  for (int f = lane; f < F; f += 32) {
    const long long fi = frag_index(rec, f, G);
    if (fi >= 0) mx = fmaxf(mx, p.part_lse[fi * p.heads + h]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
  for (int f = lane; f < F; f += 32) {
    const long long fi = frag_index(rec, f, G);
    if (fi >= 0) sum += fast_exp2(p.part_lse[fi * p.heads + h] - mx);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float lse2 = mx + fast_log2(sum);
  // Pass 2: out = sum_f 2^(lse_f - lse) o_f, in fragment order; lane owns dims
  // 4*lane + 128*q (q = 0..3) so each load instruction of the warp is one 512-byte row.
  float4 acc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int f = 0; f < F; ++f) {
    const long long fi = frag_index(rec, f, G);
    if (fi < 0) continue;
    const size_t frag = (size_t)fi * p.heads + h;
    const float wgt = fast_exp2(p.part_lse[frag] - lse2);
    const float4* src = reinterpret_cast<const float4*>(p.part_o + frag * kDimCkv);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = src[lane + 32 * q];
      acc[q].x = fmaf(wgt, v.x, acc[q].x);
      acc[q].y = fmaf(wgt, v.y, acc[q].y);
      acc[q].z = fmaf(wgt, v.z, acc[q].z);
      acc[q].w = fmaf(wgt, v.w, acc[q].w);
    }
  }
  __nv_bfloat16* dst = p.out + ((size_t)rec.row * p.heads + h) * kDimCkv;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[q].x, acc[q].y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[q].z, acc[q].w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(dst)[lane + 32 * q] = packed;
  }
  if (lane == 0) p.lse[(size_t)rec.row * p.heads + h] = lse2 * 0.69314718055994531f;
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
  mla_combine_kernel<<<dim3(p.workers, (p.heads + kCombineWarps - 1) / kCombineWarps), kCombineThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_validate(const MlaParams& p, cudaStream_t stream) {
  mla_validate_kernel<<<64, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
