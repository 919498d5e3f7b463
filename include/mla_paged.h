/*
 * mla_paged.h -- C ABI of the GB300 (sm_103a) paged Multi-head Latent Attention library.
 *
 * What the calls compute (flashinfer-bench "MLA Paged", sections "decode" and
 * "prefill"): for every query row r and query head h,
 *
 *   s_t      = sm_scale * (q_nope[r,h,:] . ckv[t,:] + q_pe[r,h,:] . kpe[t,:])
 *   lse[r,h] = log(sum_t exp(s_t))                       (natural log)
 *   out[r,h] = sum_t exp(s_t - lse[r,h]) * ckv[t,:]      (V is the 512-wide latent itself,
 *                                                         Modular MAX "mla_decoding_single_batch")
 *
 * where t runs over the key slots kv_indices[kv_indptr[b] .. kv_indptr[b+1]) of the
 * row's request b (decode), or over the first kv_len_b - q_len_b + i + 1 of them for
 * query i of request b (prefill: causal, bottom-right aligned).  One KV head is shared
 * by all query heads.
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers to contiguous row-major arrays; the
 *    caller owns every buffer (inputs, outputs, workspace).  The library allocates
 *    nothing on the device and keeps only a host-side cache of TMA descriptors keyed
 *    by pointer and shape.
 *  - bf16 tensors (q_nope, q_pe, ckv_cache, kpe_cache, out) must start on a 16-byte
 *    boundary (TMA requirement) or the call returns MLA_ERR_ALIGN.
 *  - kv_indices holds token slots: slot = page * page_size + offset, an index into the
 *    caches viewed as [num_pages * page_size, 512] and [.., 64] (the physical-index
 *    mapping of FlashMLA's abs_indices2indices_in_kvcache).  kv_indptr counts keys, so
 *    a request's kv length is kv_indptr[b+1] - kv_indptr[b].
 *  - Calls only enqueue work on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  They never synchronise and never read device memory on the host, so
 *    they may be captured in a CUDA graph.  Launch errors are returned; faults
 *    inside a kernel surface at the caller's next synchronisation.
 *  - Slots outside kv_indices are never read into the result: NaN or Inf there does
 *    not change the output.  An index outside [0, num_pages*page_size) is skipped (it
 *    is not a key of the row) instead of faulting; MLA_VALIDATE reports it.
 *  - A request with no keys gets out = 0 and lse = -inf.
 */
#ifndef MLA_PAGED_H
#define MLA_PAGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes (0 = success, negative = error). */
enum mla_status {
  MLA_OK = 0,
  MLA_ERR_NULL = -1,       /* a required pointer is NULL                                  */
  MLA_ERR_DIMS = -2,       /* head dims != 512/64, heads not in 1..128, bad sizes          */
  MLA_ERR_ALIGN = -3,      /* a bf16 tensor pointer is not 16-byte aligned                 */
  MLA_ERR_WORKSPACE = -4,  /* workspace NULL or smaller than mla_workspace_bytes()         */
  MLA_ERR_LAUNCH = -5,     /* a kernel launch failed (cudaGetLastError after the launch)   */
  MLA_ERR_BAD_INDEX = -6,  /* (device status) MLA_VALIDATE found bad indptr/indices        */
  MLA_ERR_TIMEOUT = -7,    /* (device status) a bounded wait inside a kernel gave up       */
  MLA_ERR_CUDA = -8,       /* a CUDA runtime/driver call failed (device query, TMA encode) */
  MLA_ERR_UNSUPPORTED = -9, /* no sm_103a-class device is current                          */
  MLA_ERR_INTERNAL = -10   /* (device status) a kernel found an internal invariant broken  */
};

/* Flags (bitwise OR). */
enum mla_flags {
  MLA_VALIDATE = 1 /* run an index-validation kernel first; it records MLA_ERR_BAD_INDEX in
                      the workspace status word (read it with mla_read_device_status) */
};

/* Problem sizes.  All fields are host-side values. */
typedef struct mla_dims {
  int32_t batch;          /* decode: number of requests (= query rows); prefill: requests   */
  int32_t num_qo_heads;   /* query heads, 1..128 (one shared KV head)                       */
  int32_t head_dim_ckv;   /* must be 512                                                     */
  int32_t head_dim_kpe;   /* must be 64                                                      */
  int32_t num_pages;      /* pages in ckv_cache / kpe_cache                                  */
  int32_t page_size;      /* slots per page (>= 1); num_pages * page_size < 2^31             */
  int32_t total_q;        /* prefill: qo_indptr[batch] (query rows); decode: ignored         */
  int32_t num_kv_indices; /* kv_indptr[batch]: length of kv_indices                          */
  int32_t num_workers;    /* split-KV workers (CTA pairs); 0 = one per SM pair of the device */
} mla_dims;

/*
 * Paged MLA decode: flashinfer-bench "MLA Paged", section "decode".
 *   q_nope     [batch, H, 512] bf16      q_pe      [batch, H, 64] bf16
 *   ckv_cache  [num_pages, page_size, 512] bf16
 *   kpe_cache  [num_pages, page_size, 64]  bf16
 *   kv_indptr  [batch + 1] int32 (non-decreasing, kv_indptr[0] = 0)
 *   kv_indices [num_kv_indices] int32 token slots
 *   sm_scale   softmax scale multiplying the q.k dot product
 *   out        [batch, H, 512] bf16 (written)   lse [batch, H] fp32, natural log (written)
 *   workspace  device scratch of at least mla_workspace_bytes(dims, 0) bytes, caller-owned;
 *              it holds split-KV partial results, merge counters and the device status
 *              word.  Zero-fill it once before its first use (the status word, its first
 *              4 bytes, only accumulates error bits until mla_read_device_status clears
 *              it); everything else is rewritten by every call, so one workspace may serve
 *              calls with different sizes, worker counts or head counts.  Calls that share
 *              a workspace must not overlap on the GPU.
 *   flags      MLA_VALIDATE or 0;  stream: cudaStream_t
 * Returns MLA_OK or a negative mla_status; nothing is launched on an argument error.
 */
int mla_paged_decode(const void* q_nope, const void* q_pe, const void* ckv_cache,
                     const void* kpe_cache, const int32_t* kv_indptr, const int32_t* kv_indices,
                     float sm_scale, void* out, float* lse, const mla_dims* dims,
                     void* workspace, size_t workspace_bytes, int flags, void* stream);

/*
 * Paged MLA causal prefill: flashinfer-bench "MLA Paged", section "prefill"; the
 * causal mask is bottom-right aligned: query i of request b sees its first
 * kv_len_b - q_len_b + i + 1 keys (kv_len_b >= q_len_b is required; rows that
 * would see no key get out = 0, lse = -inf, and MLA_VALIDATE flags them).
 *   q_nope [total_q, H, 512], q_pe [total_q, H, 64], out [total_q, H, 512], lse [total_q, H]
 *   qo_indptr [batch + 1] int32 query offsets (qo_indptr[batch] = total_q)
 *   other arguments as for mla_paged_decode; workspace >= mla_workspace_bytes(dims, 1).
 */
int mla_paged_prefill(const void* q_nope, const void* q_pe, const void* ckv_cache,
                      const void* kpe_cache, const int32_t* qo_indptr, const int32_t* kv_indptr,
                      const int32_t* kv_indices, float sm_scale, void* out, float* lse,
                      const mla_dims* dims, void* workspace, size_t workspace_bytes, int flags,
                      void* stream);

/*
 * Packed multi-token decode (speculative / MTP decode): every request has the same
 * number q_len >= 1 of new query tokens, causal within the request: token i of request
 * b sees the first kv_len_b - q_len + i + 1 of its keys (kv_len_b >= q_len is required;
 * MLA_VALIDATE flags shorter requests).  This is the fixed-Q form of the packed-query
 * decode in flashinfer's prims_ts wrapper (batch_mla_decode_with_paged_kv_cache,
 * parameters qo_indptr / max_seq_len_q, mask_type "causal"), and FlashMLA's
 * flash_mla_with_kvcache with seq_len_q > 1: the q_len tokens of a request share each
 * KV tile, q_len * H rows per tile.
 *   q_nope [batch, q_len, H, 512], q_pe [batch, q_len, H, 64] bf16
 *   out    [batch, q_len, H, 512] bf16, lse [batch, q_len, H] fp32 (natural log)
 *   q_len * num_qo_heads must be <= 128 (else MLA_ERR_DIMS; use mla_paged_prefill with
 *   qo_indptr for more rows per request).
 *   workspace >= mla_workspace_bytes_mtp(dims, q_len); other arguments as for
 *   mla_paged_decode (dims->total_q is ignored).
 */
int mla_paged_decode_mtp(const void* q_nope, const void* q_pe, const void* ckv_cache,
                         const void* kpe_cache, const int32_t* kv_indptr, const int32_t* kv_indices,
                         float sm_scale, void* out, float* lse, const mla_dims* dims, int q_len,
                         void* workspace, size_t workspace_bytes, int flags, void* stream);

/*
 * Sparse (top-k) paged MLA decode: FlashMLA notes, "flash_mla_with_kvcache (Sparse
 * Attention with FP8 KV Cache)" and "Sparse Attention Decoding with KV Cache" (bf16
 * caches here).  Every query row attends only to the token slots listed for it, with no
 * causal mask.
 *   q_nope [rows, H, 512], q_pe [rows, H, 64] bf16: one row per (request, query token),
 *          e.g. [batch, s_q, H, 512] viewed as [batch * s_q, H, 512]
 *   indices [rows, topk] int32 token slots (slot = page * page_size + offset); an entry
 *          that is negative or >= num_pages * page_size is padding and is skipped; a
 *          row without a valid entry gets out = 0, lse = -inf
 *   out [rows, H, 512] bf16, lse [rows, H] fp32 (natural log)
 *   dims->batch = rows; dims->num_kv_indices is ignored (rows * topk); other fields as
 *   for mla_paged_decode; workspace >= mla_workspace_bytes(dims, 0).  MLA_VALIDATE
 *   checks nothing here (any index may be padding).
 */
int mla_paged_decode_sparse(const void* q_nope, const void* q_pe, const void* ckv_cache,
                            const void* kpe_cache, const int32_t* indices, int topk, float sm_scale,
                            void* out, float* lse, const mla_dims* dims, void* workspace,
                            size_t workspace_bytes, int flags, void* stream);

/*
 * Paged MLA decode over an FP8 KV cache (FlashMLA notes, "FP8 KV Cache Quantization
 * and Dequantization", layout V32_FP8Sparse; "flash_mla_with_kvcache" with
 * is_fp8_kvcache).  kv_fp8 [num_pages * page_size][656] bytes, 16-byte aligned: per
 * token, bytes 0-511 the 512 latent values as E4M3, bytes 512-527 four float32 scales
 * (one per 128 latent values), bytes 528-655 the 64 rope values as bf16.  Latent value
 * i of a token is read as bf16(float32(e4m3_i) * scale[i / 128]) (product in float32,
 * both roundings to nearest even), the BF16 that the page's dequantisation returns;
 * the attention is then exactly mla_paged_decode's over those values.  Other arguments
 * as for mla_paged_decode (same workspace size).  MLA_ERR_ALIGN if kv_fp8 is not
 * 16-byte aligned.  Codes 0x7F / 0xFF (E4M3 NaN) propagate as NaN.
 */
int mla_paged_decode_fp8(const void* q_nope, const void* q_pe, const void* kv_fp8, const int32_t* kv_indptr,
                         const int32_t* kv_indices, float sm_scale, void* out, float* lse, const mla_dims* dims,
                         void* workspace, size_t workspace_bytes, int flags, void* stream);

/*
 * Sparse (top-k) decode over an FP8 KV cache (FlashMLA notes, "flash_mla_with_kvcache
 * (Sparse Attention with FP8 KV Cache)"): mla_paged_decode_sparse's arguments with the
 * cache of mla_paged_decode_fp8.
 */
int mla_paged_decode_sparse_fp8(const void* q_nope, const void* q_pe, const void* kv_fp8, const int32_t* indices,
                                int topk, float sm_scale, void* out, float* lse, const mla_dims* dims,
                                void* workspace, size_t workspace_bytes, int flags, void* stream);

/*
 * Block-table adapter.  The prims_ts wrapper ("batch_mla_decode_with_paged_kv_cache":
 * block_tables [batch, max_num_blocks], seq_lens) and FlashMLA's flash_mla_with_kvcache
 * (block_table, cache_seqlens) name a request's keys as the first seq_len slots of its
 * pages, in block-table order.  This writes the token-slot CSR the decode calls take:
 *   len_b = clamp(seq_lens[b], 0, max_blocks * page_size)
 *   kv_indptr[b] = len_0 + ... + len_{b-1}  (kv_indptr[batch] = the total)
 *   kv_indices[kv_indptr[b] + k] = block_table[b * max_blocks + k / page_size] * page_size
 *                                  + k % page_size
 *   block_table [batch, max_blocks] int32 page ids (row-major; entries past a request's
 *               last needed block are not read), seq_lens [batch] int32
 *   kv_indptr [batch + 1] int32 (written), kv_indices [capacity] int32 (written)
 * A slot that is negative or does not fit in int32 is written as -1, and any slot
 * outside the cache is skipped by the decode (not a key).  Positions at or past
 * `capacity` are not written (kv_indptr still counts them; pass capacity as
 * num_kv_indices and the decode reads no further).  batch * max_blocks * page_size is
 * always enough.  Two kernel launches on `stream`, no synchronisation; graph-capturable.
 * Returns MLA_ERR_DIMS (negative sizes, page_size < 1, max_blocks * page_size or
 * capacity above INT32_MAX), MLA_ERR_NULL, MLA_ERR_LAUNCH, or MLA_OK.
 */
int mla_block_table_to_csr(const int32_t* block_table, const int32_t* seq_lens, int batch, int max_blocks,
                           int page_size, int32_t* kv_indptr, int32_t* kv_indices, long long capacity,
                           void* stream);

/*
 * Paged MLA decode from a block table: mla_block_table_to_csr into the workspace, then
 * mla_paged_decode on that CSR, on `stream`.  Arguments as for mla_paged_decode, with
 * block_table [batch, max_blocks] and seq_lens [batch] in place of kv_indptr and
 * kv_indices; dims->num_kv_indices is ignored (the CSR's capacity,
 * batch * max_blocks * page_size, is used and must fit int32, else MLA_ERR_DIMS).
 * workspace >= mla_workspace_bytes_block_table(dims, max_blocks) bytes, zero-filled
 * before first use like the decode's; flags must be 0 (MLA_ERR_DIMS otherwise: the
 * CSR ends short of its capacity, which MLA_VALIDATE would report).
 */
size_t mla_workspace_bytes_block_table(const mla_dims* dims, int max_blocks);
int mla_paged_decode_block_table(const void* q_nope, const void* q_pe, const void* ckv_cache,
                                 const void* kpe_cache, const int32_t* block_table, const int32_t* seq_lens,
                                 int max_blocks, float sm_scale, void* out, float* lse, const mla_dims* dims,
                                 void* workspace, size_t workspace_bytes, int flags, void* stream);

/*
 * Paged MLA decode for callers that cannot allocate device memory (a plugin that runs
 * inside another framework's memory pool, code that must not call cudaMalloc after
 * start-up, or a context where an allocation would synchronise the device).  This entry
 * point has no counterpart in the pages the library follows; it computes exactly what
 * mla_paged_decode computes, with the same arguments except the workspace.
 *
 * The split-KV scratch lives in one static device array of 32 MiB inside the library,
 * held by every GPU that loads the library until the process exits.  With
 * dims->num_workers == 0 the call uses one worker per SM pair, or fewer if their
 * partial results would not fit in the 32 MiB; an explicit num_workers whose scratch
 * needs more returns MLA_ERR_WORKSPACE.  flags must be 0 (the device status word is not
 * read through the status call below instead), else MLA_ERR_DIMS.  All calls share the
 * array and it keeps the last call's contents: calls that overlap on the GPU race.
 * Nothing else carries over between calls (each call clears the status word and zeroes
 * the merge counters it uses).  The first call on each device looks up the array's
 * address (with that device current); make it before any stream capture.  The call
 * itself allocates nothing.
 */
int mla_paged_decode_noalloc(const void* q_nope, const void* q_pe, const void* ckv_cache,
                             const void* kpe_cache, const int32_t* kv_indptr, const int32_t* kv_indices,
                             float sm_scale, void* out, float* lse, const mla_dims* dims, int flags,
                             void* stream);

/* Device status of the most recent mla_paged_decode_noalloc call on the current device:
 * synchronises `stream`, reads and clears the status word in the library's static
 * scratch and returns MLA_OK, MLA_ERR_TIMEOUT or MLA_ERR_INTERNAL (as
 * mla_read_device_status does for a caller's workspace).  No counterpart on the pages. */
int mla_noalloc_read_status(void* stream);

/* Workspace bytes a call with these dims needs (0 on invalid dims).  With
 * dims->num_workers == 0 it queries the current device's SM count. */
size_t mla_workspace_bytes(const mla_dims* dims, int is_prefill);

/* Workspace bytes of mla_paged_decode_mtp with q_len tokens per request (0 on invalid
 * dims or q_len * num_qo_heads > 128). */
size_t mla_workspace_bytes_mtp(const mla_dims* dims, int q_len);

/* Number of split-KV workers (CTA pairs) used when dims->num_workers == 0, for the
 * current device; negative mla_status on failure. */
int mla_default_num_workers(void);

/* Human-readable name of a status code (static string). */
const char* mla_status_string(int status);

/* Synchronises `stream`, reads the device status word kept in `workspace` (MLA_OK,
 * MLA_ERR_BAD_INDEX, MLA_ERR_TIMEOUT or MLA_ERR_INTERNAL), clears it, and returns it.
 * Returns MLA_ERR_CUDA if the synchronisation itself reports an error. */
int mla_read_device_status(void* workspace, void* stream);

/* Test hook of the kernels' bounded waits (off by default; not for production use).
 * With skip_tile >= 1, the attention kernel's producer for split-KV worker 0 (first CTA
 * of the pair) skips the loads and the arrival of that tile of its range in every call
 * that follows, so the waits on it run out; wait_ns sets the limit of every bounded wait
 * (0 = the default of 4 s).  The kernel then gives up, unwinds (drains its copies and
 * matrix operations, frees tensor memory) and records MLA_ERR_TIMEOUT in the status
 * word, where mla_read_device_status finds it; outputs of that call are undefined.
 * skip_tile = -1 restores normal calls.  Returns MLA_ERR_DIMS for skip_tile 0 or < -1.
 * Not thread-safe with respect to calls in flight on other threads. */
int mla_debug_inject_timeout(int skip_tile, unsigned long long wait_ns);

/* Kernel timing for benchmarks.  When enabled, every call records CUDA events on its
 * stream around its main attention kernel and its combine kernel;
 * mla_profile_read synchronises on the last events, returns the summed milliseconds
 * and the number of timed calls since the last read, and resets the sums. */
int mla_profile_enable(int on);
int mla_profile_read(double* main_ms, double* combine_ms, int* calls);

#ifdef __cplusplus
}
#endif

#endif /* MLA_PAGED_H */
