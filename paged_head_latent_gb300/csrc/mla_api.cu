// mla_api.cu -- the C ABI: argument checks, workspace layout, kernel launches.
//
// Every entry point only enqueues work on the caller's stream; nothing here
// synchronises or reads device memory except mla_read_device_status and
// mla_profile_read, which exist to do exactly that.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "mla_paged.h"
#include "common.cuh"
#include "launch.h"
#include "tc_kernel.h"

namespace {

using mla::MlaParams;

struct DeviceInfo {
  int sms = 0;
  int major = 0, minor = 0;
  bool ok = false;
};

std::mutex g_mu;
DeviceInfo g_dev[64];

// Test hook of the bounded waits (mla_debug_inject_timeout): the wait limit and the
// tile whose arrival worker 0's producer skips (-1: none).
std::atomic<unsigned long long> g_wait_ns{4000000000ull};
std::atomic<int> g_fault_skip_tile{-1};

int query_device(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ok) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    d.ok = true;
  }
  *out = d;
  return MLA_OK;
}

int check_dims(const mla_dims* d, bool prefill) {
  if (!d) return MLA_ERR_NULL;
  if (d->head_dim_ckv != mla::kDimCkv || d->head_dim_kpe != mla::kDimKpe) return MLA_ERR_DIMS;
  if (d->num_qo_heads < 1 || d->num_qo_heads > mla::kMaxHeads) return MLA_ERR_DIMS;
  if (d->batch < 0 || d->num_pages < 0 || d->page_size < 1 || d->num_kv_indices < 0) return MLA_ERR_DIMS;
  if (d->num_workers < 0) return MLA_ERR_DIMS;
  if ((long long)d->num_pages * d->page_size >= (1LL << 31)) return MLA_ERR_DIMS;
  if (prefill && d->total_q < 0) return MLA_ERR_DIMS;
  // Output row count times heads must index within int64 comfortably; rows*H < 2^31.
  long long rows = prefill ? d->total_q : d->batch;
  if (rows * d->num_qo_heads >= (1LL << 31)) return MLA_ERR_DIMS;
  return MLA_OK;
}

int resolve_workers(const mla_dims* d, int* G) {
  if (d->num_workers > 0) {
    *G = d->num_workers;
    return MLA_OK;
  }
  DeviceInfo info;
  int st = query_device(&info);
  if (st != MLA_OK) return st;
  *G = info.sms / 2 > 0 ? info.sms / 2 : 1;
  return MLA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- TMA descriptors
using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(f);
    cudaGetLastError();
  });
  return fn;
}

struct MapKey {
  const void* ptr;
  uint64_t rows, cols;
  uint32_t box_cols, box_rows;
  int swizzle, promo, bytes;  // bytes: element size (2: bf16, 1: uint8)
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && rows == o.rows && cols == o.cols && box_cols == o.box_cols && box_rows == o.box_rows &&
           swizzle == o.swizzle && promo == o.promo && bytes == o.bytes;
  }
};

struct MapCache {
  std::mutex mu;
  std::vector<std::pair<MapKey, CUtensorMap>> entries;  // most recent last
} g_maps;

// 2-D map over [rows, cols] of bf16 (bytes = 2) or uint8 (bytes = 1) elements (row
// stride = cols elements), box = box_cols x box_rows.
int get_map(CUtensorMap* out, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows,
            CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo, int bytes = 2) {
  if (rows == 0) {  // nothing can be loaded: the kernel is given no keys / rows for it
    std::memset(out, 0, sizeof(*out));
    return MLA_OK;
  }
  const MapKey key{ptr, rows, cols, box_cols, box_rows, (int)swizzle, (int)promo, bytes};
  std::lock_guard<std::mutex> lk(g_maps.mu);
  for (auto& e : g_maps.entries)
    if (e.first == key) {
      *out = e.second;
      return MLA_OK;
    }
  EncodeFn fn = encode_fn();
  if (!fn) return MLA_ERR_CUDA;
  alignas(64) CUtensorMap m;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (cuuint64_t)bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  const auto dt = bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = fn(&m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return MLA_ERR_CUDA;
  if (g_maps.entries.size() >= 96) g_maps.entries.erase(g_maps.entries.begin());
  g_maps.entries.emplace_back(key, m);
  *out = m;
  return MLA_OK;
}

// The attention kernel's tensor maps: 64-column ckv boxes in 128-byte swizzle (one
// 64-slot page, or one gathered row), 32-column kpe boxes in 64-byte swizzle (each CTA
// of a pair takes half of the 64 positional dims), and query rows (L2 prefetch only).
int build_maps(const MlaParams& p, mla::TmaMaps* m) {
  const uint64_t slots = (uint64_t)p.num_slots;
  const auto sw128 = CU_TENSOR_MAP_SWIZZLE_128B, sw64 = CU_TENSOR_MAP_SWIZZLE_64B;
  const auto l256 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B, l128 = CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
  int st;
  if ((st = get_map(&m->ckv, p.ckv, slots, 512, 64, 64, sw128, l256)) != MLA_OK) return st;
  if ((st = get_map(&m->kpe, p.kpe, slots, 64, 32, 64, sw64, l128)) != MLA_OK) return st;
  return MLA_OK;
}

// The FP8 cache's maps, over its tokens as [slots, 656] bytes (a whole run of 64 slots
// per tile): the latent half of a CTA in two boxes of 64 tokens x 128 bytes, the four scales
// in boxes of 32 tokens x 16 bytes, and the rope half in a box of 64 tokens x 64 bytes
// with the 64-byte swizzle the bf16 kpe tiles have.
int build_fp8_maps(const MlaParams& p, mla::TmaMaps* m) {
  const uint64_t slots = (uint64_t)p.num_slots;
  const auto none = CU_TENSOR_MAP_SWIZZLE_NONE, sw64 = CU_TENSOR_MAP_SWIZZLE_64B;
  const auto l256 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B, l128 = CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
  const uint64_t tok = mla::kFp8TokenBytes;
  int st;
  if ((st = get_map(&m->f8_lat, p.kv_fp8, slots, tok, 128, 64, none, l256, 1)) != MLA_OK) return st;
  if ((st = get_map(&m->f8_scl, p.kv_fp8, slots, tok, 16, 32, none, l128, 1)) != MLA_OK) return st;
  if ((st = get_map(&m->f8_rope, p.kv_fp8, slots, tok, 64, 64, sw64, l128, 1)) != MLA_OK) return st;
  return MLA_OK;
}

// ---------------------------------------------------------------- profiling
struct ProfileState {
  bool on = false;
  std::vector<cudaEvent_t> ev;  // 3 per call
  size_t used = 0;              // triples in use
};
ProfileState g_prof;
std::mutex g_prof_mu;

// Called with g_prof_mu held.
cudaEvent_t* profile_slot() {
  if (!g_prof.on) return nullptr;
  size_t need = (g_prof.used + 1) * 3;
  while (g_prof.ev.size() < need) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_prof.ev.push_back(e);
  }
  cudaEvent_t* slot = &g_prof.ev[g_prof.used * 3];
  ++g_prof.used;
  return slot;
}

// Rows (query heads) one work row of the kernel holds: H, or q_len * H for packed
// multi-token decode (q_len > 0).
int packed_heads(const mla_dims* d, int q_len) { return q_len > 0 ? q_len * d->num_qo_heads : d->num_qo_heads; }

// topk > 0: sparse decode (kv_indptr unused; row b owns kv_indices[b*topk .. +topk)).
int run(bool prefill, int q_len, const void* q_nope, const void* q_pe, const void* ckv_cache,
        const void* kpe_cache, const int32_t* qo_indptr, const int32_t* kv_indptr,
        const int32_t* kv_indices, float sm_scale, void* out, float* lse, const mla_dims* dims,
        void* workspace, size_t workspace_bytes, int flags, void* stream_ptr, int topk = 0,
        const void* kv_fp8 = nullptr) {
  int st = check_dims(dims, prefill);
  if (st != MLA_OK) return st;
  if (topk < 0) return MLA_ERR_DIMS;
  if (topk > 0 && (long long)dims->batch * topk != dims->num_kv_indices) return MLA_ERR_DIMS;
  if (q_len < 0 || packed_heads(dims, q_len) > mla::kMaxHeads) return MLA_ERR_DIMS;
  if ((long long)dims->batch * packed_heads(dims, q_len) >= (1LL << 31)) return MLA_ERR_DIMS;
  const long long rows = prefill ? dims->total_q : dims->batch;
  if (!q_nope || !q_pe || (!kv_indptr && topk == 0) || !out || !lse) return MLA_ERR_NULL;
  // The caches may be NULL only when they hold no slot at all.
  if ((kv_fp8 ? !kv_fp8 : (!ckv_cache || !kpe_cache)) && dims->num_pages > 0) return MLA_ERR_NULL;
  if (prefill && !qo_indptr) return MLA_ERR_NULL;
  if (dims->num_kv_indices > 0 && !kv_indices) return MLA_ERR_NULL;
  if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(ckv_cache) || !aligned16(kpe_cache) ||
      !aligned16(kv_fp8) || !aligned16(out))
    return MLA_ERR_ALIGN;
  if (!std::isfinite(sm_scale)) return MLA_ERR_DIMS;
  int G = 0;
  st = resolve_workers(dims, &G);
  if (st != MLA_OK) return st;
  const mla::WorkspaceLayout lay(G, packed_heads(dims, q_len));
  if (!workspace || workspace_bytes < lay.total) return MLA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MLA_ERR_ALIGN;
  if (rows == 0) return MLA_OK;
  DeviceInfo info;
  st = query_device(&info);
  if (st != MLA_OK) return st;
  if (info.major != 10 || info.minor != 3) return MLA_ERR_UNSUPPORTED;

  MlaParams p{};
  p.q_nope = static_cast<const __nv_bfloat16*>(q_nope);
  p.q_pe = static_cast<const __nv_bfloat16*>(q_pe);
  p.ckv = static_cast<const __nv_bfloat16*>(ckv_cache);
  p.kpe = static_cast<const __nv_bfloat16*>(kpe_cache);
  p.kv_fp8 = static_cast<const uint8_t*>(kv_fp8);
  p.kv_indptr = topk > 0 ? nullptr : kv_indptr;
  p.topk = topk;
  p.qo_indptr = prefill ? qo_indptr : nullptr;
  p.kv_indices = kv_indices;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.batch = dims->batch;
  p.heads = packed_heads(dims, q_len);
  p.mtp_q = q_len;
  p.mtp_h = dims->num_qo_heads;
  p.rows = (int)rows;
  p.num_slots = dims->num_pages * dims->page_size;
  // With an empty cache no key can be loaded: treat every request as empty.
  p.num_kv_indices = p.num_slots > 0 ? dims->num_kv_indices : 0;
  p.workers = G;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.wait_ns = g_wait_ns.load();
  p.fault_skip_tile = g_fault_skip_tile.load();
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.records = reinterpret_cast<mla::CombineRecord*>(ws + lay.records);
  p.merge_count = reinterpret_cast<int*>(ws + lay.merge_count);
  p.part_lse = reinterpret_cast<float*>(ws + lay.part_lse);
  p.part_o = reinterpret_cast<float*>(ws + lay.part_o);

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaGetLastError();  // clear stale errors so the checks below see only ours
  if (flags & MLA_VALIDATE) {
    if (mla::launch_validate(p, stream) != cudaSuccess) return MLA_ERR_LAUNCH;
  }
  // Benchmark timing (off unless mla_profile_enable): the lock keeps the event list
  // consistent when calls come from several host threads.
  std::unique_lock<std::mutex> prof_lk(g_prof_mu);
  cudaEvent_t* ev = profile_slot();
  if (!ev) prof_lk.unlock();
  if (ev) cudaEventRecord(ev[0], stream);
  {
    mla::TmaMaps maps{};
    st = kv_fp8 ? build_fp8_maps(p, &maps) : build_maps(p, &maps);
    if (st != MLA_OK) return st;
    // Small pages, or the scattered keys of sparse decode: the instance that copies
    // tiles slot by slot with two warps.
    const bool gather = dims->page_size % 64 != 0 || topk > 0;
    if (mla::launch_tc(maps, p, gather, stream) != cudaSuccess) return MLA_ERR_LAUNCH;
  }
  if (ev) cudaEventRecord(ev[1], stream);
  if (mla::launch_combine(p, stream) != cudaSuccess) return MLA_ERR_LAUNCH;
  if (ev) cudaEventRecord(ev[2], stream);
  return MLA_OK;
}

}  // namespace

extern "C" {

int mla_paged_decode(const void* q_nope, const void* q_pe, const void* ckv_cache,
                     const void* kpe_cache, const int32_t* kv_indptr, const int32_t* kv_indices,
                     float sm_scale, void* out, float* lse, const mla_dims* dims,
                     void* workspace, size_t workspace_bytes, int flags, void* stream) {
  return run(false, 0, q_nope, q_pe, ckv_cache, kpe_cache, nullptr, kv_indptr, kv_indices, sm_scale,
             out, lse, dims, workspace, workspace_bytes, flags, stream);
}

int mla_paged_decode_mtp(const void* q_nope, const void* q_pe, const void* ckv_cache,
                         const void* kpe_cache, const int32_t* kv_indptr, const int32_t* kv_indices,
                         float sm_scale, void* out, float* lse, const mla_dims* dims, int q_len,
                         void* workspace, size_t workspace_bytes, int flags, void* stream) {
  if (q_len < 1) return MLA_ERR_DIMS;
  return run(false, q_len, q_nope, q_pe, ckv_cache, kpe_cache, nullptr, kv_indptr, kv_indices, sm_scale,
             out, lse, dims, workspace, workspace_bytes, flags, stream);
}

int mla_paged_decode_sparse(const void* q_nope, const void* q_pe, const void* ckv_cache,
                            const void* kpe_cache, const int32_t* indices, int topk, float sm_scale,
                            void* out, float* lse, const mla_dims* dims, void* workspace,
                            size_t workspace_bytes, int flags, void* stream) {
  if (!dims) return MLA_ERR_NULL;
  if (topk < 1) return MLA_ERR_DIMS;
  if ((long long)dims->batch * topk >= (1LL << 31)) return MLA_ERR_DIMS;
  mla_dims d = *dims;
  d.num_kv_indices = dims->batch * topk;
  if (d.batch > 0 && !indices) return MLA_ERR_NULL;
  return run(false, 0, q_nope, q_pe, ckv_cache, kpe_cache, nullptr, nullptr, indices, sm_scale, out, lse, &d,
             workspace, workspace_bytes, flags, stream, topk);
}

int mla_paged_decode_fp8(const void* q_nope, const void* q_pe, const void* kv_fp8, const int32_t* kv_indptr,
                         const int32_t* kv_indices, float sm_scale, void* out, float* lse, const mla_dims* dims,
                         void* workspace, size_t workspace_bytes, int flags, void* stream) {
  return run(false, 0, q_nope, q_pe, nullptr, nullptr, nullptr, kv_indptr, kv_indices, sm_scale, out, lse, dims,
             workspace, workspace_bytes, flags, stream, 0, kv_fp8);
}

int mla_paged_decode_sparse_fp8(const void* q_nope, const void* q_pe, const void* kv_fp8, const int32_t* indices,
                                int topk, float sm_scale, void* out, float* lse, const mla_dims* dims,
                                void* workspace, size_t workspace_bytes, int flags, void* stream) {
  if (!dims) return MLA_ERR_NULL;
  if (topk < 1) return MLA_ERR_DIMS;
  if ((long long)dims->batch * topk >= (1LL << 31)) return MLA_ERR_DIMS;
  mla_dims d = *dims;
  d.num_kv_indices = dims->batch * topk;
  if (d.batch > 0 && !indices) return MLA_ERR_NULL;
  return run(false, 0, q_nope, q_pe, nullptr, nullptr, nullptr, nullptr, indices, sm_scale, out, lse, &d,
             workspace, workspace_bytes, flags, stream, topk, kv_fp8);
}

int mla_paged_prefill(const void* q_nope, const void* q_pe, const void* ckv_cache,
                      const void* kpe_cache, const int32_t* qo_indptr, const int32_t* kv_indptr,
                      const int32_t* kv_indices, float sm_scale, void* out, float* lse,
                      const mla_dims* dims, void* workspace, size_t workspace_bytes, int flags,
                      void* stream) {
  return run(true, 0, q_nope, q_pe, ckv_cache, kpe_cache, qo_indptr, kv_indptr, kv_indices, sm_scale,
             out, lse, dims, workspace, workspace_bytes, flags, stream);
}

int mla_block_table_to_csr(const int32_t* block_table, const int32_t* seq_lens, int batch, int max_blocks,
                           int page_size, int32_t* kv_indptr, int32_t* kv_indices, long long capacity,
                           void* stream) {
  if (batch < 0 || max_blocks < 0 || page_size < 1 || capacity < 0) return MLA_ERR_DIMS;
  if ((long long)max_blocks * page_size > 0x7fffffffLL || capacity > 0x7fffffffLL) return MLA_ERR_DIMS;
  if (!kv_indptr) return MLA_ERR_NULL;
  if (batch > 0 && (!seq_lens || (max_blocks > 0 && !block_table))) return MLA_ERR_NULL;
  if (capacity > 0 && !kv_indices) return MLA_ERR_NULL;
  if (mla::launch_block_table_csr(block_table, seq_lens, batch, max_blocks, page_size, kv_indptr, kv_indices,
                                  capacity, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_LAUNCH;
  return MLA_OK;
}

}  // extern "C"

namespace {
// Workspace of the block-table decode: the decode's own workspace, then the CSR the
// adapter writes (kv_indptr, then kv_indices with room for every block of every row).
struct BlockTableLayout {
  size_t decode, indptr, indices, total;
  long long capacity;
  BlockTableLayout(size_t decode_bytes, int batch, int max_blocks, int page_size) {
    capacity = (long long)batch * max_blocks * page_size;
    decode = mla::align_up(decode_bytes, 256);
    indptr = decode;
    indices = mla::align_up(indptr + ((size_t)batch + 1) * sizeof(int32_t), 256);
    total = mla::align_up(indices + (size_t)capacity * sizeof(int32_t), 256);
  }
};

// The decode dims with the capacity as num_kv_indices; false if it does not fit int32.
bool block_table_dims(const mla_dims* dims, int max_blocks, mla_dims* d) {
  if (!dims || max_blocks < 0) return false;
  const long long cap = (long long)dims->batch * max_blocks * dims->page_size;
  if (dims->batch < 0 || dims->page_size < 1 || cap > 0x7fffffffLL) return false;
  *d = *dims;
  d->num_kv_indices = (int)cap;
  return true;
}
}  // namespace

extern "C" {

size_t mla_workspace_bytes_block_table(const mla_dims* dims, int max_blocks) {
  mla_dims d;
  if (!block_table_dims(dims, max_blocks, &d)) return 0;
  const size_t base = mla_workspace_bytes(&d, 0);
  if (base == 0) return 0;
  return BlockTableLayout(base, d.batch, max_blocks, d.page_size).total;
}

int mla_paged_decode_block_table(const void* q_nope, const void* q_pe, const void* ckv_cache,
                                 const void* kpe_cache, const int32_t* block_table, const int32_t* seq_lens,
                                 int max_blocks, float sm_scale, void* out, float* lse, const mla_dims* dims,
                                 void* workspace, size_t workspace_bytes, int flags, void* stream) {
  if (!dims) return MLA_ERR_NULL;
  mla_dims d;
  if (flags != 0 || !block_table_dims(dims, max_blocks, &d)) return MLA_ERR_DIMS;
  const size_t base = mla_workspace_bytes(&d, 0);
  if (base == 0) return check_dims(&d, false) != MLA_OK ? check_dims(&d, false) : MLA_ERR_DIMS;
  const BlockTableLayout lay(base, d.batch, max_blocks, d.page_size);
  if (!workspace || workspace_bytes < lay.total) return MLA_ERR_WORKSPACE;
  auto* ws = static_cast<uint8_t*>(workspace);
  int32_t* indptr = reinterpret_cast<int32_t*>(ws + lay.indptr);
  int32_t* indices = reinterpret_cast<int32_t*>(ws + lay.indices);
  const int st = mla_block_table_to_csr(block_table, seq_lens, d.batch, max_blocks, d.page_size, indptr, indices,
                                        lay.capacity, stream);
  if (st != MLA_OK) return st;
  return run(false, 0, q_nope, q_pe, ckv_cache, kpe_cache, nullptr, indptr, indices, sm_scale, out, lse, &d,
             workspace, lay.decode, 0, stream);
}

size_t mla_workspace_bytes(const mla_dims* dims, int is_prefill) {
  if (check_dims(dims, is_prefill != 0) != MLA_OK) return 0;
  int G = 0;
  if (resolve_workers(dims, &G) != MLA_OK) return 0;
  return mla::WorkspaceLayout(G, dims->num_qo_heads).total;
}

size_t mla_workspace_bytes_mtp(const mla_dims* dims, int q_len) {
  if (check_dims(dims, false) != MLA_OK || q_len < 1 || packed_heads(dims, q_len) > mla::kMaxHeads) return 0;
  int G = 0;
  if (resolve_workers(dims, &G) != MLA_OK) return 0;
  return mla::WorkspaceLayout(G, packed_heads(dims, q_len)).total;
}

int mla_default_num_workers(void) {
  DeviceInfo info;
  int st = query_device(&info);
  if (st != MLA_OK) return st;
  return info.sms / 2 > 0 ? info.sms / 2 : 1;
}

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_NULL: return "MLA_ERR_NULL: a required pointer is NULL";
    case MLA_ERR_DIMS: return "MLA_ERR_DIMS: unsupported or inconsistent sizes";
    case MLA_ERR_ALIGN: return "MLA_ERR_ALIGN: a tensor pointer is not 16-byte aligned";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace missing or too small";
    case MLA_ERR_LAUNCH: return "MLA_ERR_LAUNCH: a kernel launch failed";
    case MLA_ERR_BAD_INDEX: return "MLA_ERR_BAD_INDEX: indptr/indices failed validation";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a bounded wait in a kernel gave up";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: a CUDA runtime call failed";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: current device is not sm_103";
    case MLA_ERR_INTERNAL: return "MLA_ERR_INTERNAL: a kernel found an internal invariant broken (shared memory misaligned)";
    default: return "unknown mla_status";
  }
}

int mla_read_device_status(void* workspace, void* stream_ptr) {
  if (!workspace) return MLA_ERR_NULL;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  if (word != 0) {
    if (cudaMemsetAsync(workspace, 0, sizeof(word), stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  if (word & mla::kStatusInternal) return MLA_ERR_INTERNAL;
  if (word & mla::kStatusTimeout) return MLA_ERR_TIMEOUT;
  if (word & mla::kStatusBadIndex) return MLA_ERR_BAD_INDEX;
  return MLA_OK;
}

int mla_debug_inject_timeout(int skip_tile, unsigned long long wait_ns) {
  if (skip_tile == 0 || skip_tile < -1) return MLA_ERR_DIMS;
  g_wait_ns.store(wait_ns ? wait_ns : 4000000000ull);
  g_fault_skip_tile.store(skip_tile);
  return MLA_OK;
}

int mla_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof.on = on != 0;
  g_prof.used = 0;
  return MLA_OK;
}

int mla_profile_read(double* main_ms, double* combine_ms, int* calls) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  double a = 0, b = 0;
  for (size_t i = 0; i < g_prof.used; ++i) {
    cudaEvent_t* e = &g_prof.ev[i * 3];
    if (cudaEventSynchronize(e[2]) != cudaSuccess) return MLA_ERR_CUDA;
    float x = 0, y = 0;
    if (cudaEventElapsedTime(&x, e[0], e[1]) != cudaSuccess ||
        cudaEventElapsedTime(&y, e[1], e[2]) != cudaSuccess)
      return MLA_ERR_CUDA;
    a += x;
    b += y;
  }
  if (main_ms) *main_ms = a;
  if (combine_ms) *combine_ms = b;
  if (calls) *calls = (int)g_prof.used;
  g_prof.used = 0;
  return MLA_OK;
}

}  // extern "C"
