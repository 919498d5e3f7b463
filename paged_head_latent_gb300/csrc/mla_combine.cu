// mla_combine.cu -- merge of split-KV fragments, and the optional index validation.
//
// Merge (Modular MAX "mla_decoding_single_batch": split-K partitions leave exp-sum
// and max statistics that a reduction merges): for a row split into fragments
// f = 1..F with base-2 lse_f and normalised outputs o_f,
//   lse = log2(sum_f 2^lse_f),   out = sum_f 2^(lse_f - lse) * o_f.
// Every sum runs in a fixed order, so the result does not depend on timing.
//
// One CTA per (worker, group of 8 heads), one warp per head.  A row with at most
// kChunk fragments (or any row, when some workers have no tiles) is merged by its last
// worker's CTA.  A longer row (a request split over many workers, every worker holding
// a fragment) is merged in two levels so that many CTAs share it: the CTA of
// the last worker of each chunk of kChunk consecutive fragments merges that chunk into
// the chunk's first fragment slot, then counts itself in; the CTA that arrives last
// merges the chunk results, in chunk order, and resets the counter to zero for the next
// call (the workspace starts zero-filled).
#include "common.cuh"
#include "launch.h"

namespace mla {

constexpr int kCombineWarps = 8;  // one warp per head, 8 heads per CTA
constexpr int kCombineThreads = 32 * kCombineWarps;
constexpr int kChunk = 8;         // fragments merged by one CTA in the first level

// Fragment f (0-based, worker w_first + f) of a record: its slot index in the workspace,
// or -1 if that worker has no tiles.  Every worker has tiles when each one's share of
// the cost units exceeds a row's leading units (min_units > kRowCost).
__device__ __forceinline__ long long frag_index(const MlaParams& p, const CombineRecord& rec, int f) {
  const int wk = rec.w_first + f;
  if (rec.min_units <= kRowCost && !p.records[wk].live) return -1;
  return (long long)wk * 2 + (f == 0 ? rec.slot_first : 0);
}

// Merge fragments [f0, f1) of a record for head h (one warp).  Returns the base-2 lse
// and leaves the merged output in acc (lane owns dims 4*lane + 128*q, q = 0..3, so
// each load of the warp is one 512-byte row); -inf and zeros if no fragment exists.
__device__ __forceinline__ float merge_range(const MlaParams& p, const CombineRecord& rec, int f0, int f1,
                                             int h, int lane, float4 (&acc)[4]) {
  float mx = -INFINITY;
  for (int f = f0 + lane; f < f1; f += 32) {
    const long long fi = frag_index(p, rec, f);
    if (fi >= 0) mx = fmaxf(mx, p.part_lse[fi * p.heads + h]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
  for (int f = f0 + lane; f < f1; f += 32) {
    const long long fi = frag_index(p, rec, f);
    if (fi >= 0) sum += fast_exp2(p.part_lse[fi * p.heads + h] - mx);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (sum == 0.f) return -INFINITY;
  const float lse2 = mx + fast_log2(sum);
  for (int f = f0; f < f1; ++f) {
    const long long fi = frag_index(p, rec, f);
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
  return lse2;
}

// First existing fragment in [f0, f1), or -1.
__device__ __forceinline__ long long first_frag(const MlaParams& p, const CombineRecord& rec, int f0, int f1) {
  for (int f = f0; f < f1; ++f) {
    const long long fi = frag_index(p, rec, f);
    if (fi >= 0) return fi;
  }
  return -1;
}

__device__ __forceinline__ void write_final(const MlaParams& p, const CombineRecord& rec, int h, int lane,
                                            const float4 (&acc)[4], float lse2) {
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

__global__ void __launch_bounds__(kCombineThreads) mla_combine_kernel(MlaParams p) {
  // Launched as a programmatic dependent of the attention kernel: wait until that grid
  // has completed and its writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int w = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * kCombineWarps + warp;
  const CombineRecord rec = p.records[w];
  if (rec.row < 0) return;
  const int F = rec.w_last - rec.w_first + 1;
  const int fw = w - rec.w_first;
  float4 acc[4];
  // One level when the row has few fragments, or when some workers have no tiles (then
  // a chunk's last worker may have no record; the row has at most T < G fragments).
  if (F <= kChunk || rec.min_units <= kRowCost) {  // the row's last worker merges all fragments
    if (w != rec.w_last || h >= p.heads) return;
    const float lse2 = merge_range(p, rec, 0, F, h, lane, acc);
    write_final(p, rec, h, lane, acc, lse2);
    return;
  }
  const int chunk = fw / kChunk;
  const int f0 = chunk * kChunk, f1 = min(f0 + kChunk, F);
  if (fw != f1 - 1) return;  // not the last worker of its chunk
  // Level 1: merge this chunk into its first existing fragment's slot (normalised).
  const long long dst = first_frag(p, rec, f0, f1);
  if (h < p.heads && dst >= 0) {
    const float lse2 = merge_range(p, rec, f0, f1, h, lane, acc);
    const size_t frag = (size_t)dst * p.heads + h;
    float4* o = reinterpret_cast<float4*>(p.part_o + frag * kDimCkv);
#pragma unroll
    for (int q = 0; q < 4; ++q) o[lane + 32 * q] = acc[q];
    if (lane == 0) p.part_lse[frag] = lse2;
  }
  // Count this chunk in; the CTA that completes the count merges the chunk results.
  __shared__ int last;
  __threadfence();
  __syncthreads();
  const int nchunks = (F + kChunk - 1) / kChunk;
  if (threadIdx.x == 0) {
    int* cnt = p.merge_count + rec.w_last * ((p.heads + 7) / 8) + blockIdx.y;
    last = atomicAdd(cnt, 1) == nchunks - 1;
  }
  __syncthreads();
  if (!last) return;
  if (threadIdx.x == 0) p.merge_count[rec.w_last * ((p.heads + 7) / 8) + blockIdx.y] = 0;
  if (h >= p.heads) return;
  __threadfence();
  // Level 2: chunk k's result sits in its first existing fragment's slot.
  float mx = -INFINITY;
  for (int k = lane; k < nchunks; k += 32) {
    const long long fi = first_frag(p, rec, k * kChunk, min(k * kChunk + kChunk, F));
    if (fi >= 0) mx = fmaxf(mx, __ldcg(p.part_lse + fi * p.heads + h));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
  for (int k = lane; k < nchunks; k += 32) {
    const long long fi = first_frag(p, rec, k * kChunk, min(k * kChunk + kChunk, F));
    if (fi >= 0) sum += fast_exp2(__ldcg(p.part_lse + fi * p.heads + h) - mx);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float lse2 = mx + fast_log2(sum);
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < nchunks; ++k) {
    const long long fi = first_frag(p, rec, k * kChunk, min(k * kChunk + kChunk, F));
    if (fi < 0) continue;
    const size_t frag = (size_t)fi * p.heads + h;
    const float wgt = fast_exp2(__ldcg(p.part_lse + frag) - lse2);
    const float4* src = reinterpret_cast<const float4*>(p.part_o + frag * kDimCkv);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = __ldcg(src + lane + 32 * q);
      acc[q].x = fmaf(wgt, v.x, acc[q].x);
      acc[q].y = fmaf(wgt, v.y, acc[q].y);
      acc[q].z = fmaf(wgt, v.z, acc[q].z);
      acc[q].w = fmaf(wgt, v.w, acc[q].w);
    }
  }
  write_final(p, rec, h, lane, acc, lse2);
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
  // Programmatic stream serialisation: the launch overlaps the attention kernel's tail;
  // the kernel's griddepcontrol.wait keeps the data dependency.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.workers, (p.heads + kCombineWarps - 1) / kCombineWarps);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, mla_combine_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_validate(const MlaParams& p, cudaStream_t stream) {
  mla_validate_kernel<<<64, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
