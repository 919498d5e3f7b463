// mla_noalloc.cu -- paged MLA decode for callers that cannot allocate device memory.
//
// Some callers have no allocator to give us a workspace: code that runs inside
// another framework's memory pool, plugins that must not call cudaMalloc after
// start-up, or callers in a context where an allocation would synchronise the
// device.  For them this entry point keeps the split-KV scratch (status word,
// per-worker merge records, partial outputs and lse) in one file-scope device array
// of fixed size, so the call itself allocates nothing.
//
// Costs and rules of the static array:
//  - every GPU that loads this library holds kNoAllocScratchBytes of device memory
//    until the process exits;
//  - all calls share the one array, and it keeps the previous call's contents, so
//    calls that overlap on the GPU (different streams, or several host threads
//    without ordering) race and corrupt each other's partial results.  Nothing a call
//    relies on carries over from the call before: the status word is cleared here and
//    the attention kernel zeroes the merge counters, whatever sizes the previous call
//    had;
//  - the array's address is looked up once per device (cudaGetSymbolAddress) by the
//    first call made on that device, with that device current; make that first call
//    before any stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "mla_paged.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 32u << 20;  // 32 MiB

// Host code may not pass this name to a kernel: on the host it is only a stand-in
// for the symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_mla_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[64] = {};

int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_mla_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" int mla_paged_decode_noalloc(const void* q_nope, const void* q_pe, const void* ckv_cache,
                                        const void* kpe_cache, const int32_t* kv_indptr,
                                        const int32_t* kv_indices, float sm_scale, void* out, float* lse,
                                        const mla_dims* dims, int flags, void* stream) {
  if (!dims) return MLA_ERR_NULL;
  if (flags != 0) return MLA_ERR_DIMS;  // no MLA_VALIDATE: the status word is not readable here
  mla_dims d = *dims;
  if (mla_workspace_bytes(&d, 0) == 0) return MLA_ERR_DIMS;
  if (d.num_workers == 0) {
    // Default split: one worker per SM pair, fewer if the scratch cannot hold their
    // partial results for this head count.
    int g = mla_default_num_workers();
    if (g < 0) return g;
    d.num_workers = g;
    while (d.num_workers > 1 && mla_workspace_bytes(&d, 0) > kNoAllocScratchBytes) --d.num_workers;
  }
  const size_t need = mla_workspace_bytes(&d, 0);
  if (need == 0) return MLA_ERR_DIMS;
  if (need > kNoAllocScratchBytes) return MLA_ERR_WORKSPACE;  // more workers than the scratch holds
  void* scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != MLA_OK) return st;
  // The status word starts every call at zero (kernels only set bits in it), so after a
  // call mla_noalloc_read_status reports that call's device errors.
  if (cudaMemsetAsync(scratch, 0, 256, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_LAUNCH;
  }
  return mla_paged_decode(q_nope, q_pe, ckv_cache, kpe_cache, kv_indptr, kv_indices, sm_scale, out, lse, &d,
                          scratch, kNoAllocScratchBytes, 0, stream);
}

// The device status word of the most recent call on the current device (MLA_OK,
// MLA_ERR_TIMEOUT, MLA_ERR_INTERNAL), read and cleared after synchronising `stream`.
extern "C" int mla_noalloc_read_status(void* stream) {
  void* scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != MLA_OK) return st;
  return mla_read_device_status(scratch, stream);
}
