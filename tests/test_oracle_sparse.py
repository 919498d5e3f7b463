"""Pins of the oracle's sparse (top-k) decode, independent of the CUDA path.

FlashMLA notes, "Sparse Attention Decoding with KV Cache" and "Sparse MLA Prefill
Kernel": each query attends to the token slots listed for it; -1, or any value at or
beyond the number of tokens, marks an invalid entry.  The pins below fix that reading
against the plain decode definition, brute force, and invariances.
"""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from oracle import mla_oracle
from paged_head_latent_gb300 import workloads as wl
from tests.oracle_io import np_inputs, oracle_run, to_lists


def _csr_rows(w):
    """Each decode request's slot list (the CSR form), as numpy arrays."""
    ip = w.kv_indptr.tolist()
    return [w.kv_indices[ip[b]:ip[b + 1]].numpy().astype(np.int64) for b in range(w.batch)]


def test_equals_decode_when_indices_list_the_requests_keys():
    w = wl.make_decode([5, 70, 33], num_qo_heads=4, page_size=16, seed=4100)
    topk = 80
    rows = [np.concatenate([r, -np.ones(topk - len(r), np.int64)]) for r in _csr_rows(w)]
    a = np_inputs(w)
    o1, l1 = oracle.mla_sparse_decode(a["q_nope"], a["q_pe"], a["ckv_cache"], a["kpe_cache"], np.stack(rows),
                                      a["sm_scale"])
    o2, l2 = oracle_run(w)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_matches_brute_force():
    w = wl.make_sparse_decode([9, 40, 3], topk=12, num_qo_heads=3, page_size=4, seed=4101, s_q=2)
    a = np_inputs(w)
    out, lse = oracle_run(w)
    n = w.num_pages * w.page_size
    indptr, flat = [0], []
    for r in a["indices"]:
        v = [int(x) for x in r if 0 <= x < n]
        flat += v
        indptr.append(len(flat))
    bo, bl = oracle.brute_decode(to_lists(a["q_nope"]), to_lists(a["q_pe"]), to_lists(a["ckv_cache"]),
                                 to_lists(a["kpe_cache"]), indptr, flat, a["sm_scale"])
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-12)


def test_invariant_under_permutation_of_indices():
    w = wl.make_sparse_decode([300, 120], topk=100, num_qo_heads=8, page_size=64, seed=4102)
    a = np_inputs(w)
    o1, l1 = oracle_run(w)
    rng = np.random.default_rng(5)
    perm = np.stack([r[rng.permutation(len(r))] for r in a["indices"]])
    o2, l2 = oracle.mla_sparse_decode(a["q_nope"], a["q_pe"], a["ckv_cache"], a["kpe_cache"], perm, a["sm_scale"])
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def test_out_of_range_entries_change_nothing():
    w = wl.make_sparse_decode([64, 200], topk=50, num_qo_heads=4, page_size=16, seed=4103)
    a = np_inputs(w)
    o1, l1 = oracle_run(w)
    n = w.num_pages * w.page_size
    bad = np.array([-1, n, n + 7, -1000], np.int64)
    mixed = np.stack([np.insert(r, [0, 10, 20, len(r)], bad) for r in a["indices"]])
    o2, l2 = oracle.mla_sparse_decode(a["q_nope"], a["q_pe"], a["ckv_cache"], a["kpe_cache"], mixed, a["sm_scale"])
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_row_without_valid_entry_is_zero_and_minus_inf():
    w = wl.make_sparse_decode([10], topk=4, num_qo_heads=2, page_size=4, seed=4104)
    a = np_inputs(w)
    out, lse = oracle.mla_sparse_decode(a["q_nope"], a["q_pe"], a["ckv_cache"], a["kpe_cache"],
                                        -np.ones((1, 4), np.int64), a["sm_scale"])
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_duplicate_slot_counts_twice():
    """A slot listed twice is two keys (as in the CSR decode): the same as decode over the
    list with the duplicate."""
    w = wl.make_decode([6], num_qo_heads=2, page_size=8, seed=4105)
    a = np_inputs(w)
    lst = np.array([a["kv_indices"][0], a["kv_indices"][3], a["kv_indices"][3]], np.int64)
    o1, l1 = oracle.mla_sparse_decode(a["q_nope"], a["q_pe"], a["ckv_cache"], a["kpe_cache"], lst[None],
                                      a["sm_scale"])
    o2, l2 = oracle.mla_decode(a["q_nope"], a["q_pe"], a["ckv_cache"], a["kpe_cache"], np.array([0, 3]), lst,
                               a["sm_scale"])
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_named_sparse_workload_shape():
    w = wl.sparse_b64_h128_topk2048()
    assert w.indices.shape == (64, 2048) and w.q_nope.shape == (64, 128, 512)
    valid = w.valid_per_row()
    assert max(valid) == 2048 and min(valid) < 2048  # some short requests are padded
    n = w.num_pages * w.page_size
    ip = None
    for r, row in enumerate(w.indices.tolist()):
        good = [x for x in row if x >= 0]
        assert len(set(good)) == len(good) and all(x < n for x in good)
        assert row[len(good):] == [-1] * (len(row) - len(good))


# ------------------------------------------------- mutation: pins catch slips

def _mutant_python_negative_index(q_nope, q_pe, ckv_cache, kpe_cache, indices, sm_scale):
    """A slip: -1 taken as Python's 'last slot' instead of padding."""
    ckv, kpe = mla_oracle._flat_caches(ckv_cache, kpe_cache)
    idx = np.asarray(indices, dtype=np.int64)
    h = np.asarray(q_nope).shape[1]
    out = np.zeros((idx.shape[0], h, 512))
    lse = np.zeros((idx.shape[0], h))
    for r in range(idx.shape[0]):
        sel = idx[r][idx[r] < ckv.shape[0]]
        out[r], lse[r] = mla_oracle.attend(q_nope[r], q_pe[r], ckv[sel], kpe[sel], sm_scale)
    return out, lse


def _mutant_clamp(q_nope, q_pe, ckv_cache, kpe_cache, indices, sm_scale):
    """A slip: out-of-range entries clamped into the cache instead of skipped."""
    ckv, _ = mla_oracle._flat_caches(ckv_cache, kpe_cache)
    idx = np.clip(np.asarray(indices, dtype=np.int64), 0, ckv.shape[0] - 1)
    return REAL(q_nope, q_pe, ckv_cache, kpe_cache, idx, sm_scale)


REAL = oracle.mla_sparse_decode


@pytest.mark.parametrize("mutant", [_mutant_python_negative_index, _mutant_clamp])
def test_pins_catch_padding_mutants(mutant, monkeypatch):
    monkeypatch.setattr(oracle, "mla_sparse_decode", mutant)
    failed = 0
    for pin in (test_equals_decode_when_indices_list_the_requests_keys, test_out_of_range_entries_change_nothing,
                test_row_without_valid_entry_is_zero_and_minus_inf):
        try:
            pin()
        except (AssertionError, IndexError):
            failed += 1
    assert failed >= 1
