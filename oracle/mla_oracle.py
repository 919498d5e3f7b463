"""Float64 CPU oracle for paged Multi-head Latent Attention (decode and causal prefill).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code with
the CUDA path: it never imports the ``paged_head_latent_gb300`` package and the
package never imports it.

What is computed (the plain definition, evaluated in float64):

* Operator inputs and outputs: flashinfer-bench "MLA Paged", sections "decode"
  and "prefill" (axes, input list, outputs ``output`` [.., 512] and ``lse``).
* Score of query head h against key slot t:
  ``s = sm_scale * (q_nope[h] . ckv[t] + q_pe[h] . kpe[t])`` -- the query and the
  key are split into a 512-wide latent part and a 64-wide positional part, one
  shared KV head for all query heads (FlashMLA "flash_mla_with_kvcache (Dense
  Attention)": num_heads_kv = 1, head_dim 576 = 512 + 64).
* Values are the latent rows themselves: V = K[:, :512] (Modular MAX
  "mla_decoding_single_batch": "V is derived as K[:, :depth_v]").
* ``lse = log(sum_t exp(s_t))`` in the natural log; ``output = sum_t exp(s_t - lse) * ckv[t]``
  (the materialised-softmax form of FlashMLA's "Sparse MLA Prefill Kernel"
  reference listing, with natural instead of base-2 logarithms).
* ``kv_indices`` hold token slots ``page * page_size + offset`` (FlashMLA
  "FP8 KV Cache Quantization and Dequantization": physical index =
  block_index * block_size + offset); ``kv_indptr`` counts keys.
* Prefill is causal and bottom-right aligned: query i of a request with q_len
  queries and kv_len keys sees its first ``kv_len - q_len + i + 1`` keys.

Readings taken where the pages are silent or garbled:

* an empty request (kv_len = 0) gives output 0 and lse = -inf;
* prefill with kv_len < q_len is rejected (ValueError);
* the scale multiplies the dot product (the "MLA Paged" page calls sm_scale the
  softmax scale; the seesaw page's "/ qk_scale" is read as a different
  convention);
* the online-softmax rescale factor on the old accumulator is
  ``exp(m_old - m_new)`` (the seesaw page prints the reciprocal).

Pins (see tests/test_oracle.py): brute force on tiny inputs, single key,
zero query, two-key closed form, torch scaled_dot_product_attention in float64
(with an independent lse probe), page-permutation, poisoning, head/request
permutation, lse bounds, convexity, split-count invariance, and last-prefill-row
equals decode.
"""

from __future__ import annotations

import numpy as np

HEAD_DIM_CKV = 512
HEAD_DIM_KPE = 64


def _as_f64(x):
    return np.asarray(x, dtype=np.float64)


def _flat_caches(ckv_cache, kpe_cache):
    """View the paged caches as [num_slots, 512] and [num_slots, 64] (slot = page*page_size+offset)."""
    ckv = np.asarray(ckv_cache).reshape(-1, HEAD_DIM_CKV)
    kpe = np.asarray(kpe_cache).reshape(-1, HEAD_DIM_KPE)
    return ckv, kpe


def scores(q_nope_row, q_pe_row, ckv_rows, kpe_rows, sm_scale):
    """s[h, t] = sm_scale * (q_nope[h] . ckv[t] + q_pe[h] . kpe[t]) for one query row.

    q_nope_row [H, 512], q_pe_row [H, 64], ckv_rows [n, 512], kpe_rows [n, 64].
    ("MLA Paged": q_nope/q_pe split of the query; ckv/kpe split of the key.)
    """
    return float(sm_scale) * (_as_f64(q_nope_row) @ _as_f64(ckv_rows).T
                              + _as_f64(q_pe_row) @ _as_f64(kpe_rows).T)


def attend(q_nope_row, q_pe_row, ckv_rows, kpe_rows, sm_scale):
    """Attention of one query row (all heads) over the given key rows.

    Returns (out [H, 512], lse [H]).  lse = m + log(sum exp(s - m)) with m the
    row maximum (the shift only avoids overflow; it cancels exactly in the
    definition).  out = sum_t exp(s_t - lse) * ckv[t].
    """
    h = np.asarray(q_nope_row).shape[0]
    n = np.asarray(ckv_rows).shape[0]
    if n == 0:
        return np.zeros((h, HEAD_DIM_CKV)), np.full(h, -np.inf)
    s = scores(q_nope_row, q_pe_row, ckv_rows, kpe_rows, sm_scale)
    m = s.max(axis=1, keepdims=True)
    lse = m + np.log(np.exp(s - m).sum(axis=1, keepdims=True))
    weights = np.exp(s - lse)
    out = weights @ _as_f64(ckv_rows)
    return out, lse[:, 0]


def mla_decode(q_nope, q_pe, ckv_cache, kpe_cache, kv_indptr, kv_indices, sm_scale):
    """Paged MLA decode ("MLA Paged", section "decode").

    q_nope [B, H, 512], q_pe [B, H, 64], ckv_cache [P, ps, 512], kpe_cache [P, ps, 64],
    kv_indptr [B+1] (key counts), kv_indices [kv_indptr[B]] (token slots).
    Returns output [B, H, 512] float64 and lse [B, H] float64 (natural log).
    """
    ckv, kpe = _flat_caches(ckv_cache, kpe_cache)
    indptr = np.asarray(kv_indptr, dtype=np.int64)
    idx = np.asarray(kv_indices, dtype=np.int64)
    q_nope = np.asarray(q_nope)
    q_pe = np.asarray(q_pe)
    b, h = q_nope.shape[0], q_nope.shape[1]
    out = np.zeros((b, h, HEAD_DIM_CKV))
    lse = np.zeros((b, h))
    for r in range(b):
        slots = idx[indptr[r]:indptr[r + 1]]
        out[r], lse[r] = attend(q_nope[r], q_pe[r], ckv[slots], kpe[slots], sm_scale)
    return out, lse


def block_table_to_csr(block_table, seq_lens, page_size):
    """Token-slot CSR of a block table.

    The prims_ts wrapper ("batch_mla_decode_with_paged_kv_cache": block_tables
    [batch, max_num_blocks], seq_lens) and FlashMLA's ``flash_mla_with_kvcache``
    (block_table, cache_seqlens) name a request's keys as the first seq_len slots of its
    pages, taken in table order; a slot is page * page_size + offset (FlashMLA notes, "FP8
    KV Cache Quantization and Dequantization", physical index).  A length is clamped to
    [0, max_blocks * page_size]; a slot that is negative or above the int32 range is
    written as -1 (not a key).  Returns (kv_indptr [batch + 1], kv_indices), int64 numpy.
    """
    table = np.asarray(block_table, dtype=np.int64)
    lens = np.asarray(seq_lens, dtype=np.int64)
    indptr = [0]
    indices = []
    for b in range(table.shape[0]):
        n = min(max(int(lens[b]), 0), table.shape[1] * page_size)
        for k in range(n):
            slot = int(table[b, k // page_size]) * page_size + k % page_size
            indices.append(slot if 0 <= slot <= 2 ** 31 - 1 else -1)
        indptr.append(len(indices))
    return np.asarray(indptr, dtype=np.int64), np.asarray(indices, dtype=np.int64)


def mla_decode_block_table(q_nope, q_pe, ckv_cache, kpe_cache, block_table, seq_lens, sm_scale):
    """Decode whose keys come from a block table (``block_table_to_csr``).  A slot outside
    the cache is not a key of the row (the reading the sparse page's -1 padding implies),
    so such entries are dropped before ``mla_decode``."""
    page_size = np.asarray(ckv_cache).shape[1]
    num_slots = np.asarray(ckv_cache).shape[0] * page_size
    indptr, indices = block_table_to_csr(block_table, seq_lens, page_size)
    kept_ptr = [0]
    kept = []
    for b in range(len(indptr) - 1):
        row = [int(t) for t in indices[indptr[b]:indptr[b + 1]] if 0 <= t < num_slots]
        kept.extend(row)
        kept_ptr.append(len(kept))
    return mla_decode(q_nope, q_pe, ckv_cache, kpe_cache, np.asarray(kept_ptr), np.asarray(kept, dtype=np.int64),
                      sm_scale)


FP8_TOKEN_BYTES = 656  # 512 e4m3 + 4 fp32 scales + 64 bf16 (FlashMLA notes, V32_FP8Sparse)


def e4m3_to_float(codes):
    """Value of FP8 E4M3 codes (uint8), from the format's definition: 1 sign bit, 4
    exponent bits with bias 7, 3 mantissa bits; exponent 0 is subnormal
    (mantissa / 8 * 2^-6); no infinities; S.1111.111 is NaN.  Returns float64."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    v = sign * np.where(e == 0, sub, normal)
    return np.where((e == 0xF) & (m == 0x7), np.nan, v)


def _round_bf16(x32):
    """float32 -> nearest bfloat16 (ties to even), returned as float64."""
    import torch  # a library primitive for the rounding step only
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def dequantize_fp8_cache(kv_fp8):
    """The 656-byte-per-token cache (FlashMLA notes, "FP8 KV Cache Quantization and
    Dequantization", V32_FP8Sparse: bytes 0-511 the 512-wide latent as E4M3, bytes
    512-527 four float32 scales, one per 128-element tile, bytes 528-655 the 64-wide
    rope part in bfloat16, unquantised) back to BF16, as the page's dequantize
    returns: latent element i of a token = bf16(float32(e4m3_i) * scale_{i // 128}),
    the product in float32.  kv_fp8 [P, ps, 656] uint8.  Returns (ckv [P, ps, 512],
    kpe [P, ps, 64]) float64 holding bf16 values."""
    raw = np.asarray(kv_fp8, dtype=np.uint8)
    assert raw.shape[-1] == FP8_TOKEN_BYTES
    lead = raw.shape[:-1]
    vals = e4m3_to_float(raw[..., :512]).astype(np.float32)  # exact: E4M3 fits in float32
    scales = np.ascontiguousarray(raw[..., 512:528]).view(np.float32).reshape(*lead, 4)
    prod = (vals.reshape(*lead, 4, 128) * scales[..., None]).astype(np.float32).reshape(*lead, 512)
    ckv = _round_bf16(prod)
    rope = np.ascontiguousarray(raw[..., 528:656]).view(np.uint16).reshape(*lead, 64).astype(np.uint32) << 16
    kpe = rope.view(np.float32).astype(np.float64)
    return ckv, kpe


def mla_decode_fp8(q_nope, q_pe, kv_fp8, kv_indptr, kv_indices, sm_scale):
    """Decode over an FP8 cache: the dense decode of the dequantised cache."""
    ckv, kpe = dequantize_fp8_cache(kv_fp8)
    return mla_decode(q_nope, q_pe, ckv, kpe, kv_indptr, kv_indices, sm_scale)


def mla_sparse_decode_fp8(q_nope, q_pe, kv_fp8, indices, sm_scale):
    """Sparse decode over an FP8 cache (FlashMLA notes, "flash_mla_with_kvcache (Sparse
    Attention with FP8 KV Cache)"): the sparse decode of the dequantised cache."""
    ckv, kpe = dequantize_fp8_cache(kv_fp8)
    return mla_sparse_decode(q_nope, q_pe, ckv, kpe, indices, sm_scale)


def visible_len(kv_len, q_len, i):
    """Keys visible to query i of a request (causal, bottom-right aligned)."""
    return kv_len - q_len + i + 1


def mla_prefill(q_nope, q_pe, ckv_cache, kpe_cache, qo_indptr, kv_indptr, kv_indices, sm_scale,
                rows=None):
    """Paged MLA causal prefill ("MLA Paged", section "prefill"; bottom-right causal mask).

    q_nope [total_q, H, 512], q_pe [total_q, H, 64]; qo_indptr [B+1] query offsets,
    kv_indptr [B+1] key offsets.  Returns output [total_q, H, 512], lse [total_q, H].
    With ``rows`` (an iterable of global query indices) only those rows are
    computed; the others stay 0 / NaN.
    """
    ckv, kpe = _flat_caches(ckv_cache, kpe_cache)
    qo = np.asarray(qo_indptr, dtype=np.int64)
    kvp = np.asarray(kv_indptr, dtype=np.int64)
    idx = np.asarray(kv_indices, dtype=np.int64)
    q_nope = np.asarray(q_nope)
    q_pe = np.asarray(q_pe)
    total_q, h = q_nope.shape[0], q_nope.shape[1]
    if qo[-1] != total_q:
        raise ValueError("total_q != qo_indptr[-1]")
    out = np.zeros((total_q, h, HEAD_DIM_CKV))
    lse = np.full((total_q, h), np.nan)
    wanted = None if rows is None else set(int(r) for r in rows)
    for b in range(len(qo) - 1):
        q_len = qo[b + 1] - qo[b]
        kv_len = kvp[b + 1] - kvp[b]
        if kv_len < q_len:
            raise ValueError(f"request {b}: kv_len {kv_len} < q_len {q_len}")
        slots = idx[kvp[b]:kvp[b + 1]]
        for i in range(q_len):
            r = qo[b] + i
            if wanted is not None and r not in wanted:
                continue
            vis = slots[:visible_len(kv_len, q_len, i)]
            out[r], lse[r] = attend(q_nope[r], q_pe[r], ckv[vis], kpe[vis], sm_scale)
    return out, lse


def mla_sparse_decode(q_nope, q_pe, ckv_cache, kpe_cache, indices, sm_scale):
    """Sparse (top-k) MLA decode (FlashMLA notes, "flash_mla_with_kvcache (Sparse
    Attention with FP8 KV Cache)" and "Sparse Attention Decoding with KV Cache": each
    query attends only to the token slots listed for it; "Sparse MLA Prefill Kernel":
    invalid entries are -1 or any value >= the number of tokens).

    q_nope [R, H, 512], q_pe [R, H, 64] -- one row per (request, query token); indices
    [R, topk] token slots into the caches viewed as [num_slots, 512] / [.., 64].  Entries
    outside [0, num_slots) are padding and skipped; a slot listed twice counts twice.
    No causal mask.  Returns output [R, H, 512] and lse [R, H] (natural log); a row
    without a valid entry gets 0 and -inf.
    """
    ckv, kpe = _flat_caches(ckv_cache, kpe_cache)
    n = ckv.shape[0]
    idx = np.asarray(indices, dtype=np.int64)
    q_nope = np.asarray(q_nope)
    q_pe = np.asarray(q_pe)
    r_count, h = q_nope.shape[0], q_nope.shape[1]
    out = np.zeros((r_count, h, HEAD_DIM_CKV))
    lse = np.zeros((r_count, h))
    for r in range(r_count):
        sel = idx[r]
        sel = sel[(sel >= 0) & (sel < n)]
        out[r], lse[r] = attend(q_nope[r], q_pe[r], ckv[sel], kpe[sel], sm_scale)
    return out, lse


# ---------------------------------------------------------------------------
# Split-KV form: blocked online softmax per split, then the partial combine.
# ---------------------------------------------------------------------------

def online_softmax_partial(q_nope_row, q_pe_row, ckv_rows, kpe_rows, sm_scale, block):
    """Flash-attention-2 style pass over key blocks (Modular MAX
    "mla_decoding_single_batch": "Flash attention v2 algorithm"; FlashMLA deep
    dive "Seesaw Scheduling" steps 3-5 and 8, with the rescale factor read as
    exp(m_old - m_new)).

    Keeps a running max m, running sum l and unnormalised accumulator o.  Returns
    the normalised partial output o / l and its lse = m + log(l).
    """
    h = np.asarray(q_nope_row).shape[0]
    n = np.asarray(ckv_rows).shape[0]
    m = np.full(h, -np.inf)
    l = np.zeros(h)
    o = np.zeros((h, HEAD_DIM_CKV))
    for start in range(0, n, block):
        kn = ckv_rows[start:start + block]
        kp = kpe_rows[start:start + block]
        s = scores(q_nope_row, q_pe_row, kn, kp, sm_scale)  # step 1/2: p = q K^T * scale
        m_new = np.maximum(m, s.max(axis=1))                 # step 3: running max
        scale = np.exp(m - m_new)                            # exp(m_old - m_new) <= 1
        p = np.exp(s - m_new[:, None])                       # step 4: p <- exp(p - m_new)
        l = l * scale + p.sum(axis=1)
        o = o * scale[:, None] + p @ _as_f64(kn)             # step 5: o <- o*scale + p V
        m = m_new
    if n == 0:
        return np.zeros((h, HEAD_DIM_CKV)), np.full(h, -np.inf)
    return o / l[:, None], m + np.log(l)


def combine_partials(outs, lses):
    """Merge split-KV fragments (Modular MAX "mla_decoding_single_batch": split-K
    partitions with exp-sum/max statistics; FlashMLA ``num_splits``).

    outs: list of normalised partial outputs [H, 512]; lses: list of [H] lse
    values.  lse = log sum_i exp(lse_i);  out = sum_i exp(lse_i - lse) * out_i,
    summed in list order.
    """
    lses = np.stack([_as_f64(x) for x in lses])       # [F, H]
    outs = np.stack([_as_f64(x) for x in outs])       # [F, H, 512]
    m = lses.max(axis=0)
    safe_m = np.where(np.isfinite(m), m, 0.0)
    total = safe_m + np.log(np.exp(lses - safe_m).sum(axis=0))
    w = np.exp(lses - total)                          # [F, H]; 0 for empty fragments
    w = np.where(np.isfinite(lses), w, 0.0)
    out = (w[:, :, None] * outs).sum(axis=0)
    return out, total


def mla_decode_split(q_nope, q_pe, ckv_cache, kpe_cache, kv_indptr, kv_indices, sm_scale,
                     num_splits, block=64):
    """Decode computed as ``num_splits`` contiguous key splits per request, each by the
    blocked online softmax, then merged by ``combine_partials``."""
    ckv, kpe = _flat_caches(ckv_cache, kpe_cache)
    indptr = np.asarray(kv_indptr, dtype=np.int64)
    idx = np.asarray(kv_indices, dtype=np.int64)
    q_nope = np.asarray(q_nope)
    q_pe = np.asarray(q_pe)
    b, h = q_nope.shape[0], q_nope.shape[1]
    out = np.zeros((b, h, HEAD_DIM_CKV))
    lse = np.zeros((b, h))
    for r in range(b):
        slots = idx[indptr[r]:indptr[r + 1]]
        n = len(slots)
        if n == 0:
            out[r], lse[r] = 0.0, -np.inf
            continue
        bounds = [n * k // num_splits for k in range(num_splits + 1)]
        outs, lses = [], []
        for k in range(num_splits):
            part = slots[bounds[k]:bounds[k + 1]]
            o, ls = online_softmax_partial(q_nope[r], q_pe[r], ckv[part], kpe[part], sm_scale, block)
            outs.append(o)
            lses.append(ls)
        out[r], lse[r] = combine_partials(outs, lses)
    return out, lse
