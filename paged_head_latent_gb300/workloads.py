"""Seeded synthetic inputs for paged MLA decode and prefill.

This module only draws inputs: lengths, page tables, and N(0,1) bf16 tensors.
It holds none of the attention arithmetic, so both the CUDA path and the
float64 oracle can take their inputs from here without sharing any math.

The tensors follow the operator definition on the flashinfer-bench page
"MLA Paged" (sections "prefill" and "decode"):

* ``q_nope``  [rows, num_qo_heads, 512]  bf16
* ``q_pe``    [rows, num_qo_heads, 64]   bf16
* ``ckv_cache`` [num_pages, page_size, 512] bf16
* ``kpe_cache`` [num_pages, page_size, 64]  bf16
* ``kv_indptr`` [batch + 1] int32, ``kv_indices`` [kv_indptr[-1]] int32
* ``qo_indptr`` [batch + 1] int32 (prefill only)

``kv_indices`` are token slots: ``slot = page * page_size + offset`` (the
physical-index mapping shown in FlashMLA's ``abs_indices2indices_in_kvcache``
example), so ``kv_indptr`` counts keys and a request's kv length is the
difference of two consecutive ``kv_indptr`` entries.

Draw order per workload (one CPU ``torch.Generator``): kv lengths, page
permutation, q_nope, q_pe, ckv_cache, kpe_cache.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import torch

HEAD_DIM_CKV = 512
HEAD_DIM_KPE = 64
DEFAULT_SM_SCALE = 192.0 ** -0.5


@dataclasses.dataclass
class Workload:
    """One seeded input set. All tensors live on the CPU until ``to`` is called."""

    name: str
    kind: str  # "decode" or "prefill"
    num_qo_heads: int
    page_size: int
    num_pages: int
    sm_scale: float
    q_nope: torch.Tensor
    q_pe: torch.Tensor
    ckv_cache: torch.Tensor
    kpe_cache: torch.Tensor
    kv_indptr: torch.Tensor
    kv_indices: torch.Tensor
    qo_indptr: Optional[torch.Tensor] = None
    # Sparse (top-k) decode: [rows, topk] token slots per query row; entries outside the
    # cache are padding.  kv_indptr / kv_indices then hold the same lists as a CSR view
    # (row r owns entries r*topk .. r*topk + topk - 1).
    indices: Optional[torch.Tensor] = None
    # FP8 cache (kinds "decode_fp8" / "sparse_fp8"): [num_pages, page_size, 656] uint8 per
    # token -- 512 E4M3 latent values, 4 float32 scales (one per 128 values), 64 bf16
    # rope values (FlashMLA's V32_FP8Sparse layout).  ckv_cache / kpe_cache then hold the
    # bf16 values it was quantised from.
    kv_fp8: Optional[torch.Tensor] = None

    @property
    def batch(self) -> int:
        return self.kv_indptr.numel() - 1

    @property
    def rows(self) -> int:
        """Query rows: batch for decode, total_q for prefill."""
        return self.q_nope.shape[0]

    @property
    def mtp_q_len(self) -> int:
        """Tokens per request of a packed multi-token decode workload."""
        return self.rows // self.batch if self.batch else 0

    @property
    def num_kv_indices(self) -> int:
        return self.kv_indices.numel()

    @property
    def topk(self) -> int:
        return self.indices.shape[1] if self.indices is not None else 0

    def valid_per_row(self) -> List[int]:
        """Sparse decode: entries of each row that name a slot of the cache."""
        n = self.num_pages * self.page_size
        return ((self.indices >= 0) & (self.indices < n)).sum(dim=1).tolist()

    def kv_lens(self) -> List[int]:
        p = self.kv_indptr.tolist()
        return [p[i + 1] - p[i] for i in range(len(p) - 1)]

    def q_lens(self) -> List[int]:
        if self.qo_indptr is None:
            return [1] * self.batch
        p = self.qo_indptr.tolist()
        return [p[i + 1] - p[i] for i in range(len(p) - 1)]

    def visible_keys(self) -> int:
        """Number of (query row, key) pairs the operator scores, per head."""
        if self.kind in ("decode", "decode_fp8"):
            return sum(self.kv_lens())
        if self.kind in ("sparse", "sparse_fp8"):
            return sum(self.valid_per_row())
        total = 0
        for ql, kl in zip(self.q_lens(), self.kv_lens()):
            prefix = kl - ql
            total += ql * prefix + ql * (ql + 1) // 2
        return total

    def tensors(self) -> Dict[str, torch.Tensor]:
        d = dict(q_nope=self.q_nope, q_pe=self.q_pe, ckv_cache=self.ckv_cache,
                 kpe_cache=self.kpe_cache, kv_indptr=self.kv_indptr,
                 kv_indices=self.kv_indices)
        if self.qo_indptr is not None:
            d["qo_indptr"] = self.qo_indptr
        if self.indices is not None:
            d["indices"] = self.indices
        if self.kv_fp8 is not None:
            d["kv_fp8"] = self.kv_fp8
        return d

    def to(self, device) -> "Workload":
        moved = {k: v.to(device) for k, v in self.tensors().items()}
        return dataclasses.replace(self, **moved)


def _randn_bf16(shape: Sequence[int], gen: torch.Generator, chunk: int = 1 << 24) -> torch.Tensor:
    """N(0,1) drawn in float32 and rounded to bf16, in chunks to bound memory."""
    out = torch.empty(int(math.prod(shape)), dtype=torch.bfloat16)
    n = out.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = torch.randn(e - s, generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return out.view(*shape)


def _page_table(kv_lens: Sequence[int], page_size: int, pool_pages: Optional[int],
                gen: torch.Generator, token_shuffle: bool):
    """Assign pages of a permuted pool to requests in order; expand to token slots.

    Returns (kv_indptr, kv_indices, num_pages).  With ``token_shuffle`` the slots
    of the whole pool are permuted token by token instead (no page alignment),
    which is the layout a page_size-1 cache has.
    """
    need = [-(-l // page_size) for l in kv_lens]
    total_pages = sum(need)
    num_pages = total_pages if pool_pages is None else pool_pages
    if num_pages < total_pages:
        raise ValueError("page pool smaller than the pages the requests need")
    indptr = [0]
    for l in kv_lens:
        indptr.append(indptr[-1] + l)
    if token_shuffle:
        slots = torch.randperm(num_pages * page_size, generator=gen, dtype=torch.int64)
        indices = slots[: indptr[-1]].to(torch.int32)
    else:
        perm = torch.randperm(num_pages, generator=gen, dtype=torch.int64)[:total_pages]
        parts = []
        p0 = 0
        for l, n in zip(kv_lens, need):
            pages = perm[p0:p0 + n]
            p0 += n
            slots = (pages[:, None] * page_size + torch.arange(page_size)[None, :]).reshape(-1)
            parts.append(slots[:l])
        indices = torch.cat(parts).to(torch.int32) if parts else torch.zeros(0, dtype=torch.int32)
    return torch.tensor(indptr, dtype=torch.int32), indices.contiguous(), num_pages


def make_decode(kv_lens: Sequence[int], num_qo_heads: int, page_size: int, seed: int,
                pool_pages: Optional[int] = None, token_shuffle: bool = False,
                sm_scale: float = DEFAULT_SM_SCALE, name: str = "decode",
                kv_lens_fn=None) -> Workload:
    """Decode workload: one query per request.

    ``kv_lens_fn(gen)`` may draw the lengths from the workload's generator (it
    is called first, so the draw order stays fixed); otherwise ``kv_lens``
    is used as given.
    """
    gen = torch.Generator().manual_seed(seed)
    if kv_lens_fn is not None:
        kv_lens = kv_lens_fn(gen)
    kv_lens = [int(x) for x in kv_lens]
    indptr, indices, num_pages = _page_table(kv_lens, page_size, pool_pages, gen, token_shuffle)
    b = len(kv_lens)
    q_nope = _randn_bf16((b, num_qo_heads, HEAD_DIM_CKV), gen)
    q_pe = _randn_bf16((b, num_qo_heads, HEAD_DIM_KPE), gen)
    ckv = _randn_bf16((num_pages, page_size, HEAD_DIM_CKV), gen)
    kpe = _randn_bf16((num_pages, page_size, HEAD_DIM_KPE), gen)
    return Workload(name=name, kind="decode", num_qo_heads=num_qo_heads, page_size=page_size,
                    num_pages=num_pages, sm_scale=sm_scale, q_nope=q_nope, q_pe=q_pe,
                    ckv_cache=ckv, kpe_cache=kpe, kv_indptr=indptr, kv_indices=indices)


@dataclasses.dataclass
class BlockTableInputs:
    """Decode inputs in block-table form (the prims_ts wrapper's block_tables
    [batch, max_num_blocks] and seq_lens; FlashMLA's block_table and cache_seqlens)."""

    num_qo_heads: int
    page_size: int
    num_pages: int
    sm_scale: float
    q_nope: torch.Tensor
    q_pe: torch.Tensor
    ckv_cache: torch.Tensor
    kpe_cache: torch.Tensor
    block_table: torch.Tensor  # [batch, max_blocks] int32 page ids
    seq_lens: torch.Tensor     # [batch] int32

    def to(self, device) -> "BlockTableInputs":
        return dataclasses.replace(self, **{f.name: getattr(self, f.name).to(device)
                                            for f in dataclasses.fields(self)
                                            if isinstance(getattr(self, f.name), torch.Tensor)})


def make_block_table_decode(seq_lens: Sequence[int], num_qo_heads: int, page_size: int, max_blocks: int,
                            seed: int, junk: str = "random", sm_scale: float = DEFAULT_SM_SCALE) -> BlockTableInputs:
    """Block-table decode inputs: request b's ceil(len_b / page_size) pages (len_b its
    sequence length, clamped to the table's width) are drawn from a permuted pool and
    fill the front of row b; the rest of the row holds ``junk``: random page ids of the
    pool ("random") or -1 ("minus1"), which a correct reader never uses.  A sequence
    length may be negative or exceed max_blocks * page_size (the reader clamps it).
    Draw order: page permutation, junk, q_nope, q_pe, ckv_cache, kpe_cache."""
    gen = torch.Generator().manual_seed(seed)
    lens = [min(max(int(x), 0), max_blocks * page_size) for x in seq_lens]
    need = [-(-l // page_size) for l in lens]
    num_pages = max(sum(need), 1)
    perm = torch.randperm(num_pages, generator=gen, dtype=torch.int64)
    b = len(lens)
    if junk == "random":
        table = torch.randint(0, num_pages, (b, max_blocks), generator=gen, dtype=torch.int64)
    else:
        table = torch.full((b, max_blocks), -1, dtype=torch.int64)
    p0 = 0
    for r, n in enumerate(need):
        table[r, :n] = perm[p0:p0 + n]
        p0 += n
    q_nope = _randn_bf16((b, num_qo_heads, HEAD_DIM_CKV), gen)
    q_pe = _randn_bf16((b, num_qo_heads, HEAD_DIM_KPE), gen)
    ckv = _randn_bf16((num_pages, page_size, HEAD_DIM_CKV), gen)
    kpe = _randn_bf16((num_pages, page_size, HEAD_DIM_KPE), gen)
    return BlockTableInputs(num_qo_heads=num_qo_heads, page_size=page_size, num_pages=num_pages,
                            sm_scale=sm_scale, q_nope=q_nope, q_pe=q_pe, ckv_cache=ckv, kpe_cache=kpe,
                            block_table=table.to(torch.int32).contiguous(),
                            seq_lens=torch.tensor([int(x) for x in seq_lens], dtype=torch.int32))


def make_prefill(q_lens: Sequence[int], prefixes: Sequence[int], num_qo_heads: int,
                 page_size: int, seed: int, pool_pages: Optional[int] = None,
                 token_shuffle: bool = False, sm_scale: float = DEFAULT_SM_SCALE,
                 name: str = "prefill") -> Workload:
    """Prefill workload: request b has q_lens[b] new queries after prefixes[b] cached keys.

    kv_len = q_len + prefix; the causal mask is bottom-right aligned (query i of
    a request sees its first prefix + i + 1 keys).
    """
    gen = torch.Generator().manual_seed(seed)
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(q) + int(p) for q, p in zip(q_lens, prefixes)]
    indptr, indices, num_pages = _page_table(kv_lens, page_size, pool_pages, gen, token_shuffle)
    qo = [0]
    for q in q_lens:
        qo.append(qo[-1] + q)
    total_q = qo[-1]
    q_nope = _randn_bf16((total_q, num_qo_heads, HEAD_DIM_CKV), gen)
    q_pe = _randn_bf16((total_q, num_qo_heads, HEAD_DIM_KPE), gen)
    ckv = _randn_bf16((num_pages, page_size, HEAD_DIM_CKV), gen)
    kpe = _randn_bf16((num_pages, page_size, HEAD_DIM_KPE), gen)
    return Workload(name=name, kind="prefill", num_qo_heads=num_qo_heads, page_size=page_size,
                    num_pages=num_pages, sm_scale=sm_scale, q_nope=q_nope, q_pe=q_pe,
                    ckv_cache=ckv, kpe_cache=kpe, kv_indptr=indptr, kv_indices=indices,
                    qo_indptr=torch.tensor(qo, dtype=torch.int32))


def make_mtp(kv_lens: Optional[Sequence[int]], q_len: int, num_qo_heads: int, page_size: int, seed: int,
             kv_lens_fn=None, name: str = "mtp") -> Workload:
    """Packed multi-token decode: every request has q_len new tokens at the end of its
    kv_len keys (a prefill with q_lens = q_len and prefixes = kv_len - q_len, kind "mtp")."""
    if kv_lens is None:
        kv_lens = kv_lens_fn(torch.Generator().manual_seed(seed))
    w = make_prefill([q_len] * len(kv_lens), [k - q_len for k in kv_lens], num_qo_heads=num_qo_heads,
                     page_size=page_size, seed=seed, name=name)
    return dataclasses.replace(w, kind="mtp")


def make_sparse_decode(kv_lens: Optional[Sequence[int]], topk: int, num_qo_heads: int, page_size: int,
                       seed: int, s_q: int = 1, kv_lens_fn=None, name: str = "sparse") -> Workload:
    """Sparse (top-k) decode: each of a request's s_q query tokens attends to its own
    list of topk token slots of that request (FlashMLA's sparse decoding, where an
    indexer picks the keys).  Slots are drawn without replacement from the request's
    slots in random order; a request with fewer than topk keys lists all of them and
    pads with -1.  Draw order: kv lengths, page permutation, index draws (row by row),
    q_nope, q_pe, ckv_cache, kpe_cache."""
    gen = torch.Generator().manual_seed(seed)
    if kv_lens_fn is not None:
        kv_lens = kv_lens_fn(gen)
    kv_lens = [int(x) for x in kv_lens]
    indptr, slots, num_pages = _page_table(kv_lens, page_size, None, gen, False)
    ip = indptr.tolist()
    rows = []
    for b, l in enumerate(kv_lens):
        own = slots[ip[b]:ip[b + 1]]
        for _ in range(s_q):
            take = min(topk, l)
            pick = own[torch.randperm(l, generator=gen)[:take]] if take else own[:0]
            rows.append(torch.cat([pick, torch.full((topk - take,), -1, dtype=torch.int32)]))
    indices = torch.stack(rows).to(torch.int32).contiguous()
    r = len(rows)
    q_nope = _randn_bf16((r, num_qo_heads, HEAD_DIM_CKV), gen)
    q_pe = _randn_bf16((r, num_qo_heads, HEAD_DIM_KPE), gen)
    ckv = _randn_bf16((num_pages, page_size, HEAD_DIM_CKV), gen)
    kpe = _randn_bf16((num_pages, page_size, HEAD_DIM_KPE), gen)
    csr_indptr = torch.arange(r + 1, dtype=torch.int32) * topk
    return Workload(name=name, kind="sparse", num_qo_heads=num_qo_heads, page_size=page_size,
                    num_pages=num_pages, sm_scale=DEFAULT_SM_SCALE, q_nope=q_nope, q_pe=q_pe,
                    ckv_cache=ckv, kpe_cache=kpe, kv_indptr=csr_indptr, kv_indices=indices.reshape(-1).clone(),
                    indices=indices)


def poison_unreferenced(w: Workload, value: float = float("nan")) -> Workload:
    """Return a copy whose cache slots not named in kv_indices hold ``value``."""
    ckv = w.ckv_cache.clone()
    kpe = w.kpe_cache.clone()
    used = torch.zeros(w.num_pages * w.page_size, dtype=torch.bool)
    idx = w.kv_indices.long()
    used[idx[(idx >= 0) & (idx < used.numel())]] = True
    ckv.view(-1, HEAD_DIM_CKV)[~used] = value
    kpe.view(-1, HEAD_DIM_KPE)[~used] = value
    return dataclasses.replace(w, ckv_cache=ckv, kpe_cache=kpe)


# --------------------------------------------------------------------------
# The five named workloads.  Seeds are 1000 + the workload's number.
# --------------------------------------------------------------------------

def decode_b4_h16_ps64() -> Workload:
    """Small decode: batch 4, 16 heads, page 64, kv lens {1, 63, 64, 200}, 16-page pool."""
    return make_decode([1, 63, 64, 200], num_qo_heads=16, page_size=64, seed=1001,
                       pool_pages=16, name="decode_b4_h16_ps64")


def decode_b64_h128_ps64() -> Workload:
    """Decode: batch 64, 128 heads, page 64, kv lens uniform in [1024, 8192]."""
    def lens(gen):
        return torch.randint(1024, 8193, (64,), generator=gen).tolist()
    return make_decode(None, num_qo_heads=128, page_size=64, seed=1002, kv_lens_fn=lens,
                       name="decode_b64_h128_ps64")


def decode_b128_h128_ps1() -> Workload:
    """Decode with token-granular paging: batch 128, 128 heads, page 1, kv 4096 each."""
    return make_decode([4096] * 128, num_qo_heads=128, page_size=1, seed=1003,
                       name="decode_b128_h128_ps1")


def decode_b32_h128_skew() -> Workload:
    """Skewed decode: one request of 131072 keys and 31 of 512; 128 heads, page 64."""
    return make_decode([131072] + [512] * 31, num_qo_heads=128, page_size=64, seed=1004,
                       name="decode_b32_h128_skew")


def prefill_causal_h128() -> Workload:
    """Causal prefill: q lens {1024..4096}, prefixes {0, 1024, 2048, 4096}, 128 heads, page 64."""
    return make_prefill([1024, 2048, 3072, 4096], [0, 1024, 2048, 4096], num_qo_heads=128,
                        page_size=64, seed=1005, name="prefill_causal_h128")


def prefill_causal_h128_r1() -> Workload:
    """One request of the causal prefill batch, reduced for single-launch profiling: q_len
    2048 after a prefix of 1024, 128 heads, page 64."""
    return make_prefill([2048], [1024], num_qo_heads=128, page_size=64, seed=1015, name="prefill_causal_h128_r1")


def mtp_b64_h16_q4_ps64() -> Workload:
    """Packed multi-token decode: batch 64, 16 heads, 4 tokens per request (64 rows per
    tile), page 64, kv lens uniform in [1024, 8192]."""
    def lens(gen):
        return torch.randint(1024, 8193, (64,), generator=gen).tolist()
    return make_mtp(None, 4, num_qo_heads=16, page_size=64, seed=1006, kv_lens_fn=lens,
                    name="mtp_b64_h16_q4_ps64")


def sparse_b64_h128_topk2048() -> Workload:
    """Sparse decode: 64 requests of 128 heads, page 64; 60 requests of 4096..16384 keys
    and 4 of 512..2047 keys (shorter than topk, so padded with -1); each query attends to
    2048 of its request's keys."""
    def lens(gen):
        long = torch.randint(4096, 16385, (60,), generator=gen).tolist()
        short = torch.randint(512, 2048, (4,), generator=gen).tolist()
        return long[:15] + short[:1] + long[15:30] + short[1:2] + long[30:45] + short[2:3] + long[45:] + short[3:]
    return make_sparse_decode(None, 2048, num_qo_heads=128, page_size=64, seed=1007, kv_lens_fn=lens,
                              name="sparse_b64_h128_topk2048")


FP8_TOKEN_BYTES = 656


def quantize_fp8(w: Workload, name: Optional[str] = None) -> Workload:
    """The workload with its cache in the 656-byte FP8 layout.  Each token's 512 latent
    values are quantised in tiles of 128: scale = max|x| / 448 (1 for an all-zero tile),
    code = E4M3 nearest to x / scale (clamped to +-448); the rope part stays bf16.  This
    only prepares inputs; how the cache is read back is the reader's business."""
    ckv = w.ckv_cache.float()
    lead = ckv.shape[:-1]
    tiles = ckv.reshape(*lead, 4, 128)
    amax = tiles.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).to(torch.float32)
    codes = (tiles / scale[..., None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    buf = torch.empty(*lead, FP8_TOKEN_BYTES, dtype=torch.uint8)
    buf[..., :512] = codes.reshape(*lead, 512).view(torch.uint8)
    buf[..., 512:528] = scale.contiguous().view(torch.uint8).reshape(*lead, 16)
    buf[..., 528:] = w.kpe_cache.contiguous().view(torch.uint8).reshape(*lead, 128)
    kind = {"decode": "decode_fp8", "sparse": "sparse_fp8"}[w.kind]
    return dataclasses.replace(w, kind=kind, kv_fp8=buf, name=name or (w.name + "_fp8"))


def fp8_b64_h128_ps64() -> Workload:
    """The 64-request, 128-head, page-64 decode batch with its cache in FP8."""
    return quantize_fp8(decode_b64_h128_ps64(), name="fp8_b64_h128_ps64")


NAMED = {
    "decode_b4_h16_ps64": decode_b4_h16_ps64,
    "decode_b64_h128_ps64": decode_b64_h128_ps64,
    "decode_b128_h128_ps1": decode_b128_h128_ps1,
    "decode_b32_h128_skew": decode_b32_h128_skew,
    "prefill_causal_h128": prefill_causal_h128,
    "prefill_causal_h128_r1": prefill_causal_h128_r1,
    "mtp_b64_h16_q4_ps64": mtp_b64_h16_q4_ps64,
    "sparse_b64_h128_topk2048": sparse_b64_h128_topk2048,
    "fp8_b64_h128_ps64": fp8_b64_h128_ps64,
}


def by_name(name: str) -> Workload:
    return NAMED[name]()
