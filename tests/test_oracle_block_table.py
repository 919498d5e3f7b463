"""Pins of the oracle's block-table conversion (CPU only).

The prims_ts wrapper ("batch_mla_decode_with_paged_kv_cache": block_tables
[batch, max_num_blocks], seq_lens) and FlashMLA's flash_mla_with_kvcache (block_table,
cache_seqlens) name a request's keys as the first seq_len slots of its pages in table
order, slot = page * page_size + offset (FlashMLA notes, "FP8 KV Cache Quantization and
Dequantization", physical index).  The expected values below are worked out by hand
from that rule.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_head_latent_gb300 import workloads as wl


def test_hand_example():
    # page_size 4.  Request 0: 9 keys on pages 7, 2, 9 -> slots 28..31, 8..11, 36.
    # Request 1: 3 keys on page 5 -> slots 20, 21, 22 (its other entries are unused).
    indptr, indices = oracle.block_table_to_csr([[7, 2, 9], [5, 0, 0]], [9, 3], 4)
    assert indptr.tolist() == [0, 9, 12]
    assert indices.tolist() == [28, 29, 30, 31, 8, 9, 10, 11, 36, 20, 21, 22]


def test_lengths_are_clamped_and_bad_pages_marked():
    # Request 0: length 0.  Request 1: length 11 > 2 blocks * 4 -> 8 keys.  Request 2:
    # negative length -> 0.  Request 3: a negative page id gives -1 for its slots.
    # Request 4: a page id whose slots pass the int32 range gives -1.
    big = 2 ** 30
    indptr, indices = oracle.block_table_to_csr([[3, 1], [6, 4], [2, 2], [-1, 0], [big, 0]], [0, 11, -5, 2, 1], 4)
    assert indptr.tolist() == [0, 0, 8, 8, 10, 11]
    assert indices.tolist() == [24, 25, 26, 27, 16, 17, 18, 19, -1, -1, -1]


def test_page_size_one_is_the_table_itself():
    t = [[9, 4, 7, 1], [3, 3, 0, 5]]
    indptr, indices = oracle.block_table_to_csr(t, [4, 2], 1)
    assert indptr.tolist() == [0, 4, 6] and indices.tolist() == [9, 4, 7, 1, 3, 3]


def test_decode_equals_decode_on_the_listed_slots():
    """The block-table decode is the dense decode over the same keys; a slot outside the
    cache is dropped (not a key)."""
    x = wl.make_block_table_decode([70, 0, 130, 5], num_qo_heads=4, page_size=16, max_blocks=10, seed=5100)
    t = x.block_table.clone()
    t[2, 3] = x.num_pages + 7  # request 2's keys 48..63 lie outside the cache
    qn, qp, ckv, kpe = (a.float().numpy() for a in (x.q_nope, x.q_pe, x.ckv_cache, x.kpe_cache))
    out, lse = oracle.mla_decode_block_table(qn, qp, ckv, kpe, t.numpy(), x.seq_lens.numpy(), x.sm_scale)
    ps = 16
    rows = []
    for b, n in enumerate([70, 0, 130, 5]):
        rows.append([int(t[b, k // ps]) * ps + k % ps for k in range(n)
                     if int(t[b, k // ps]) < x.num_pages])
    indptr = np.cumsum([0] + [len(r) for r in rows])
    ref_out, ref_lse = oracle.mla_decode(qn, qp, ckv, kpe, indptr,
                                         np.asarray(sum(rows, []), dtype=np.int64), x.sm_scale)
    assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse)
    assert len(rows[2]) == 130 - 16
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))


def _transposed(block_table, seq_lens, page_size):
    t = np.asarray(block_table)
    return oracle.mla_oracle.__dict__["_orig_bt"](t.T.copy() if t.shape[0] == t.shape[1] else t[:, ::-1].copy(),
                                                  seq_lens, page_size)


def _offset_off_by_one(block_table, seq_lens, page_size):
    indptr, indices = oracle.mla_oracle.__dict__["_orig_bt"](block_table, seq_lens, page_size)
    return indptr, np.where(indices >= 0, indices + 1, indices)


@pytest.mark.parametrize("mutant", [_transposed, _offset_off_by_one])
def test_hand_pin_catches_mutants(mutant, monkeypatch):
    monkeypatch.setitem(oracle.mla_oracle.__dict__, "_orig_bt", oracle.mla_oracle.block_table_to_csr)
    monkeypatch.setattr(oracle.mla_oracle, "block_table_to_csr", mutant)
    monkeypatch.setattr(oracle, "block_table_to_csr", mutant)
    with pytest.raises(AssertionError):
        test_hand_example()
