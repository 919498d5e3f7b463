// mla_adapter.cu -- block table + sequence lengths -> the token-slot CSR that the decode
// entry points take.
//
// The prims_ts wrapper ("batch_mla_decode_with_paged_kv_cache": block_tables
// [batch, max_num_blocks] and seq_lens) and FlashMLA's flash_mla_with_kvcache
// (block_table, cache_seqlens) describe a request's keys as the first seq_len slots of
// its pages, in block-table order.  With a slot being page * page_size + offset (the
// physical-index rule of the FlashMLA notes, "FP8 KV Cache Quantization and
// Dequantization"):
//   len_b = clamp(seq_lens[b], 0, max_blocks * page_size)
//   kv_indptr[b] = len_0 + ... + len_{b-1},   kv_indptr[batch] = the total
//   kv_indices[kv_indptr[b] + k] = block_table[b, k / page_size] * page_size + k % page_size
// A slot that is negative or does not fit in int32 is written as -1 (the decode skips
// any slot outside the cache).  Positions at or past `capacity` are not written.
#include "launch.h"

namespace mla {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kFillThreads = 256;

__device__ __forceinline__ long long clamped_len(const int32_t* seq_lens, int b, long long max_len) {
  const long long v = seq_lens[b];
  return v < 0 ? 0 : (v > max_len ? max_len : v);
}

// One CTA.  Thread t sums a contiguous run of requests; an inclusive scan of the run sums
// in shared memory gives each run its offset; the thread then writes its run's entries.
__global__ void __launch_bounds__(kScanThreads)
    csr_indptr_kernel(const int32_t* seq_lens, int batch, long long max_len, int32_t* kv_indptr) {
  __shared__ long long part[kScanThreads];
  const int t = threadIdx.x;
  const int per = (batch + kScanThreads - 1) / kScanThreads;
  const int b0 = min(t * per, batch), b1 = min(b0 + per, batch);
  long long sum = 0;
  for (int b = b0; b < b1; ++b) sum += clamped_len(seq_lens, b, max_len);
  part[t] = sum;
  __syncthreads();
  for (int o = 1; o < kScanThreads; o <<= 1) {
    const long long v = t >= o ? part[t - o] : 0;
    __syncthreads();
    part[t] += v;
    __syncthreads();
  }
  long long run = part[t] - sum;
  for (int b = b0; b < b1; ++b) {
    kv_indptr[b] = (int32_t)run;
    run += clamped_len(seq_lens, b, max_len);
  }
  if (t == kScanThreads - 1) kv_indptr[batch] = (int32_t)part[t];
}

// Requests strided over the CTAs, a request's keys over the threads.
__global__ void __launch_bounds__(kFillThreads)
    csr_indices_kernel(const int32_t* block_table, const int32_t* seq_lens, int batch, int max_blocks,
                       int page_size, const int32_t* kv_indptr, int32_t* kv_indices, long long capacity) {
  const long long max_len = (long long)max_blocks * page_size;
  for (int b = blockIdx.x; b < batch; b += gridDim.x) {
    const long long len = clamped_len(seq_lens, b, max_len);
    const long long base = kv_indptr[b];
    const int32_t* row = block_table + (size_t)b * max_blocks;
    for (long long k = threadIdx.x; k < len; k += kFillThreads) {
      const long long pos = base + k;
      if (pos >= capacity) break;
      const long long page = row[k / page_size];
      const long long slot = page * page_size + k % page_size;
      kv_indices[pos] = (slot < 0 || slot > 0x7fffffffLL) ? -1 : (int32_t)slot;
    }
  }
}

}  // namespace

cudaError_t launch_block_table_csr(const int32_t* block_table, const int32_t* seq_lens, int batch, int max_blocks,
                                   int page_size, int32_t* kv_indptr, int32_t* kv_indices, long long capacity,
                                   cudaStream_t stream) {
  csr_indptr_kernel<<<1, kScanThreads, 0, stream>>>(seq_lens, batch, (long long)max_blocks * page_size, kv_indptr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || batch == 0 || capacity == 0) return e;
  const int grid = batch < 4096 ? batch : 4096;
  csr_indices_kernel<<<grid, kFillThreads, 0, stream>>>(block_table, seq_lens, batch, max_blocks, page_size,
                                                        kv_indptr, kv_indices, capacity);
  return cudaGetLastError();
}

}  // namespace mla
