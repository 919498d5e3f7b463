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
// merges the chunk results, in chunk order.  The attention kernel zeroes the counters at
// the start of every call.
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

template <bool kCg>
__device__ __forceinline__ float load_f(const float* ptr) {
  if constexpr (kCg) return __ldcg(ptr);
  else return *ptr;
}
template <bool kCg>
__device__ __forceinline__ float4 load_f4(const float4* ptr) {
  if constexpr (kCg) return __ldcg(ptr);
  else return *ptr;
}

// Two positions' rows: lanes k and k + 1 of fi name their slots (-1: none).
template <bool kCg>
__device__ __forceinline__ void load_rows(const MlaParams& p, long long fi, int k, int n, int h, int lane,
                                          float4 (&v)[2][4]) {
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const long long fu = __shfl_sync(0xffffffffu, fi, (k + u) & 31);
    const bool use = k + u < n && fu >= 0;
    const float4* src = reinterpret_cast<const float4*>(p.part_o + ((size_t)(use ? fu : 0) * p.heads + h) * kDimCkv);
#pragma unroll
    for (int q = 0; q < 4; ++q) v[u][q] = use ? load_f4<kCg>(src + lane + 32 * q) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}
__device__ __forceinline__ void add_rows(float wgt, int k, const float4 (&v)[2][4], float4 (&acc)[4]) {
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const float wg = __shfl_sync(0xffffffffu, wgt, (k + u) & 31);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc[q].x = fmaf(wg, v[u][q].x, acc[q].x);
      acc[q].y = fmaf(wg, v[u][q].y, acc[q].y);
      acc[q].z = fmaf(wg, v[u][q].z, acc[q].z);
      acc[q].w = fmaf(wg, v[u][q].w, acc[q].w);
    }
  }
}

// Merge the fragments at positions [f0, f1) for head h (one warp); slot(f) is the
// workspace slot of position f, or -1 if there is none.  Returns the base-2 lse and
// leaves the merged output in acc (lane owns dims 4*lane + 128*q, q = 0..3, so each load
// of the warp is one 512-byte row); -inf and zeros if no fragment exists.  The lanes
// gather the positions' slots and lse values (32 at a time); the first two rows are
// loaded while the statistics are reduced, and the rows are accumulated in position
// order, two loads in flight at a time.  kCg reads through L2 only (data written by
// other CTAs of this grid).
template <bool kCg, typename SlotFn>
__device__ __forceinline__ float merge_range(const MlaParams& p, int f0, int f1, int h, int lane,
                                             SlotFn slot, float4 (&acc)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  const int n0 = min(32, f1 - f0);
  const long long fi0 = lane < n0 ? slot(f0 + lane) : -1;
  const float ls0 = fi0 >= 0 ? load_f<kCg>(p.part_lse + fi0 * p.heads + h) : -INFINITY;
  float4 v[2][4];
  load_rows<kCg>(p, fi0, 0, n0, h, lane, v);
  // Running (max, sum of 2^(lse - max)) of this lane's positions.
  float mx = -INFINITY, sum = 0.f;
  for (int b0 = f0; b0 < f1; b0 += 32) {
    float ls = ls0;
    if (b0 != f0) {
      const long long fi = b0 + lane < f1 ? slot(b0 + lane) : -1;
      ls = fi >= 0 ? load_f<kCg>(p.part_lse + fi * p.heads + h) : -INFINITY;
    }
    if (ls > -INFINITY) {  // (a fragment with no weight adds nothing)
      const float m2 = fmaxf(mx, ls);
      sum = sum * fast_exp2(mx - m2) + fast_exp2(ls - m2);
      mx = m2;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, mx, o);
    const float so = __shfl_xor_sync(0xffffffffu, sum, o);
    const float m2 = fmaxf(mx, mo);
    sum = (sum == 0.f ? 0.f : sum * fast_exp2(mx - m2)) + (so == 0.f ? 0.f : so * fast_exp2(mo - m2));
    mx = m2;
  }
  if (sum == 0.f) return -INFINITY;
  const float lse2 = mx + fast_log2(sum);
  for (int b0 = f0; b0 < f1; b0 += 32) {
    const int n = min(32, f1 - b0);
    long long fi = fi0;
    float ls = ls0;
    if (b0 != f0) {
      fi = lane < n ? slot(b0 + lane) : -1;
      ls = fi >= 0 ? load_f<kCg>(p.part_lse + fi * p.heads + h) : -INFINITY;
    }
    const float wgt = ls > -INFINITY ? fast_exp2(ls - lse2) : 0.f;
    int k = 0;
    if (b0 == f0) {  // the two rows loaded above
      add_rows(wgt, 0, v, acc);
      k = 2;
    }
    for (; k < n; k += 2) {
      load_rows<kCg>(p, fi, k, n, h, lane, v);
      add_rows(wgt, k, v, acc);
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

// At most 48 registers: five CTAs per SM, so the whole grid (most of whose CTAs exit at
// once) is resident in one wave.
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
    const float lse2 = merge_range<false>(p, 0, F, h, lane, [&](int f) { return frag_index(p, rec, f); }, acc);
    write_final(p, rec, h, lane, acc, lse2);
    return;
  }
  const int chunk = fw / kChunk;
  const int f0 = chunk * kChunk, f1 = min(f0 + kChunk, F);
  if (fw != f1 - 1) return;  // not the last worker of its chunk
  // Level 1: merge this chunk into its first existing fragment's slot (normalised).
  const long long dst = first_frag(p, rec, f0, f1);
  if (h < p.heads && dst >= 0) {
    const float lse2 = merge_range<false>(p, f0, f1, h, lane, [&](int f) { return frag_index(p, rec, f); }, acc);
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
  if (h >= p.heads) return;
  __threadfence();
  // Level 2: chunk k's result sits in its first existing fragment's slot.
  const float lse2 = merge_range<true>(p, 0, nchunks, h, lane, [&](int k) {
    return first_frag(p, rec, k * kChunk, min(k * kChunk + kChunk, F));
  }, acc);
  write_final(p, rec, h, lane, acc, lse2);
}

// Index validation (flashinfer's "validate" switch on its planned wrapper inspired it):
// indptr starts at 0, is non-decreasing, ends at num_kv_indices (and total_q for
// qo_indptr), every request has kv_len >= q_len, every index is a slot of the cache.
// Sets kStatusBadIndex in the status word; never traps.
__global__ void mla_validate_kernel(MlaParams p) {
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  const int nthreads = gridDim.x * blockDim.x;
  // Sparse decode has no indptr, and any index may be padding: nothing to check.
  if (!p.kv_indptr) return;
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
      if (p.mtp_q > 0 && (k1 - k) < p.mtp_q) bad = true;  // packed tokens need kv_len >= q_len
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
