// common.cuh -- parameter block and workspace layout shared by the kernels and the launcher.
#pragma once
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "plan.cuh"

namespace mla {

constexpr int kDimCkv = 512;  // latent width (the V width too)
constexpr int kDimKpe = 64;   // positional-key width
constexpr int kMaxHeads = 128;

// Bits of the device status word (workspace offset 0).
constexpr uint32_t kStatusBadIndex = 1u;
constexpr uint32_t kStatusTimeout = 2u;
constexpr uint32_t kStatusInternal = 4u;  // an internal invariant failed (misaligned shared memory)

struct MlaParams {
  const __nv_bfloat16* q_nope;  // [rows, H, 512]
  const __nv_bfloat16* q_pe;    // [rows, H, 64]
  const __nv_bfloat16* ckv;     // [num_slots, 512]
  const __nv_bfloat16* kpe;     // [num_slots, 64]
  const int32_t* kv_indptr;     // [batch + 1], or nullptr (sparse decode: topk entries per row)
  const int32_t* qo_indptr;     // [batch + 1] or nullptr (decode)
  const int32_t* kv_indices;    // [num_kv_indices]
  __nv_bfloat16* out;           // [rows, H, 512]
  float* lse;                   // [rows, H]
  int batch;
  int heads;
  int rows;           // decode: batch; prefill: total_q
  int num_slots;      // num_pages * page_size
  int num_kv_indices;
  int workers;        // G
  float scale_log2;   // sm_scale * log2(e): scores are kept in base-2 units
  // workspace
  uint32_t* status;         // device status word
  CombineRecord* records;   // [G]
  int* merge_count;         // [G][ceil(H/8)] chunk-merge arrivals (zeroed by the attention kernel)
  float* part_lse;          // [G][2][H]  base-2 lse of partial fragments
  float* part_o;            // [G][2][H][512] normalised partial outputs
  // Packed multi-token decode (0 otherwise): each request has mtp_q query tokens of
  // mtp_h heads packed into heads = mtp_q * mtp_h rows; token i sees the first
  // kv_len - mtp_q + i + 1 keys (causal within the request).
  int mtp_q;
  int mtp_h;
  // Bounded waits give up after wait_ns nanoseconds.  fault_skip_tile >= 1 makes the
  // producer of worker 0, rank 0, skip that tile's loads and arrival (a test of the
  // give-up path; -1 in normal calls).
  unsigned long long wait_ns;
  int fault_skip_tile;
  int topk;  // sparse decode: entries per row (kv_indptr is nullptr); 0 otherwise
  // FP8 cache, or nullptr: [num_slots][656] bytes per token -- 512 E4M3 latent values,
  // 4 float32 scales (one per 128 values), 64 bf16 rope values.  ckv / kpe are unused.
  const uint8_t* kv_fp8;
};

constexpr int kFp8TokenBytes = 656;  // FP8 cache: 512 E4M3 + 4 float32 scales + 64 bf16 per token

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout: [status (256 B)] [records: G x 24 B] [merge counters] [part_lse] [part_o].
struct WorkspaceLayout {
  size_t records, merge_count, part_lse, part_o, total;
  __host__ __device__ WorkspaceLayout(int G, int H) {
    records = 256;
    merge_count = align_up(records + (size_t)G * sizeof(CombineRecord), 256);
    part_lse = align_up(merge_count + (size_t)G * ((H + 7) / 8) * sizeof(int), 256);
    part_o = align_up(part_lse + (size_t)G * 2 * H * sizeof(float), 256);
    total = align_up(part_o + (size_t)G * 2 * H * kDimCkv * sizeof(float), 256);
  }
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace mla

namespace mla {

// Rows that see no key (an empty decode request; a prefill row of a request with
// kv_len < q_len) get out = 0 and lse = -inf.  Run by one full warp of one CTA.
__device__ inline void warp_write_empty_rows(const MlaParams& p) {
  const int lane = threadIdx.x & 31;
  PlanArgs pa{p.kv_indptr, p.qo_indptr, p.batch, p.num_kv_indices, p.topk};
  for (int base = 0; base < p.batch; base += 32) {
    int b = base + lane;
    int n_empty = 0, row0 = 0;
    if (b < p.batch) {
      Req r = load_req(pa, b);
      n_empty = min(max(r.q_len - r.kv_len, 0), r.q_len);
      row0 = r.qo0;
    }
    unsigned todo = __ballot_sync(0xffffffffu, n_empty > 0);
    while (todo) {
      const int src = __ffs(todo) - 1;
      todo &= todo - 1;
      const int ne = __shfl_sync(0xffffffffu, n_empty, src);
      const int r0 = __shfl_sync(0xffffffffu, row0, src);
      for (int row = r0; row < r0 + ne; ++row) {
        if (row < 0 || row >= p.rows) continue;
        uint4* dst = reinterpret_cast<uint4*>(p.out + (size_t)row * p.heads * kDimCkv);
        for (int v = lane; v < p.heads * kDimCkv / 8; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
        for (int hh = lane; hh < p.heads; hh += 32) p.lse[(size_t)row * p.heads + hh] = -INFINITY;
      }
    }
  }
}

}  // namespace mla
