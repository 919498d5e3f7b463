"""Pins for the float64 oracle, each independent of the oracle's own code path.

Nothing here needs a GPU.  Every pin is chosen so that a plausible slip in the
oracle (a dropped kpe term, V taken as the 576-wide key, a log2 lse, an
off-by-one causal bound, a transposed operand) fails at least one of them; the
mutation tests at the bottom plant such slips in a copy of the oracle and check
that the pins catch them.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import mla_oracle
from paged_head_latent_gb300 import workloads as wl
from tests.oracle_io import np_inputs, oracle_run, to_lists


def _tiny_decode(seed, kv_lens, heads=3, page_size=4, shuffle=False, pool=None):
    return wl.make_decode(kv_lens, num_qo_heads=heads, page_size=page_size, seed=seed,
                          token_shuffle=shuffle, pool_pages=pool)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("kv_lens,page_size,shuffle", [
    ([1, 5, 9], 4, False),
    ([70, 3], 64, False),
    ([17, 33, 2], 1, False),
    ([12, 7], 4, True),
])
def test_brute_force_decode(kv_lens, page_size, shuffle):
    w = _tiny_decode(11 + len(kv_lens) + page_size, kv_lens, page_size=page_size, shuffle=shuffle)
    a = np_inputs(w)
    out, lse = oracle_run(w)
    bo, bl = oracle.brute_decode(to_lists(a["q_nope"]), to_lists(a["q_pe"]), to_lists(a["ckv_cache"]),
                                 to_lists(a["kpe_cache"]), to_lists(a["kv_indptr"]),
                                 to_lists(a["kv_indices"]), a["sm_scale"])
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-12)


def test_brute_force_prefill():
    w = wl.make_prefill([3, 5], [2, 0], num_qo_heads=2, page_size=4, seed=21)
    a = np_inputs(w)
    out, lse = oracle_run(w)
    bo, bl = oracle.brute_prefill(to_lists(a["q_nope"]), to_lists(a["q_pe"]), to_lists(a["ckv_cache"]),
                                  to_lists(a["kpe_cache"]), to_lists(a["qo_indptr"]),
                                  to_lists(a["kv_indptr"]), to_lists(a["kv_indices"]), a["sm_scale"])
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- closed forms

def test_single_key_exact():
    """One key: output is that ckv row exactly and lse is its score."""
    w = _tiny_decode(31, [1, 1], heads=4, page_size=8)
    a = np_inputs(w)
    # Put a known score in: q_nope = a*e_3, q_pe = b*e_5; score = sm_scale*(a*ckv[t,3] + b*kpe[t,5]).
    qn = np.zeros_like(a["q_nope"]); qn[:, :, 3] = 2.0
    qp = np.zeros_like(a["q_pe"]); qp[:, :, 5] = -0.5
    out, lse = oracle.mla_decode(qn, qp, a["ckv_cache"], a["kpe_cache"], a["kv_indptr"],
                                 a["kv_indices"], a["sm_scale"])
    ckv = a["ckv_cache"].reshape(-1, 512)
    kpe = a["kpe_cache"].reshape(-1, 64)
    for b in range(2):
        t = a["kv_indices"][b]
        assert np.array_equal(out[b], np.broadcast_to(ckv[t].astype(np.float64), out[b].shape))
        want = a["sm_scale"] * (2.0 * float(ckv[t, 3]) + (-0.5) * float(kpe[t, 5]))
        np.testing.assert_allclose(lse[b], want, rtol=0, atol=1e-14)


def test_zero_query_is_mean_and_log_n():
    """q = 0 gives equal weights: output = mean of referenced rows, lse = ln N."""
    w = _tiny_decode(41, [5, 64, 1], heads=2, page_size=4)
    a = np_inputs(w)
    out, lse = oracle.mla_decode(np.zeros_like(a["q_nope"]), np.zeros_like(a["q_pe"]), a["ckv_cache"],
                                 a["kpe_cache"], a["kv_indptr"], a["kv_indices"], a["sm_scale"])
    ckv = a["ckv_cache"].reshape(-1, 512).astype(np.float64)
    ip = a["kv_indptr"]
    for b in range(3):
        slots = a["kv_indices"][ip[b]:ip[b + 1]]
        np.testing.assert_allclose(out[b], np.broadcast_to(ckv[slots].mean(axis=0), out[b].shape),
                                   rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[b], math.log(len(slots)), rtol=0, atol=1e-13)


def test_sm_scale_zero_is_mean():
    w = _tiny_decode(43, [9], heads=2, page_size=4)
    a = np_inputs(w)
    out, lse = oracle.mla_decode(a["q_nope"], a["q_pe"], a["ckv_cache"], a["kpe_cache"],
                                 a["kv_indptr"], a["kv_indices"], 0.0)
    ckv = a["ckv_cache"].reshape(-1, 512).astype(np.float64)
    np.testing.assert_allclose(out[0], np.broadcast_to(ckv[a["kv_indices"]].mean(axis=0), out[0].shape),
                               rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0], math.log(9), atol=1e-13)


def test_two_keys_sigmoid_form():
    """Two keys: out = sigma(s1-s2) v1 + sigma(s2-s1) v2, lse = s2 + log1p(exp(s1-s2))."""
    w = _tiny_decode(51, [2], heads=3, page_size=2)
    a = np_inputs(w)
    out, lse = oracle_run(w)
    ckv = a["ckv_cache"].reshape(-1, 512).astype(np.float64)
    kpe = a["kpe_cache"].reshape(-1, 64).astype(np.float64)
    t1, t2 = a["kv_indices"]
    for h in range(3):
        qn = a["q_nope"][0, h].astype(np.float64)
        qp = a["q_pe"][0, h].astype(np.float64)
        s1 = a["sm_scale"] * (math.fsum(qn * ckv[t1]) + math.fsum(qp * kpe[t1]))
        s2 = a["sm_scale"] * (math.fsum(qn * ckv[t2]) + math.fsum(qp * kpe[t2]))
        sig = 1.0 / (1.0 + math.exp(-(s1 - s2)))
        np.testing.assert_allclose(out[0, h], sig * ckv[t1] + (1 - sig) * ckv[t2], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[0, h], s2 + math.log1p(math.exp(s1 - s2)), atol=1e-12)


# ------------------------------------------------------ library reduction (SDPA)

def _sdpa_row(qn, qp, kn, kp, sm_scale, mask=None):
    """torch SDPA in float64 with K = [ckv | kpe], V = ckv, one KV head broadcast to all heads.

    lse comes from a second SDPA call with one extra probe key of score 0 whose
    value is 1 in an extra column: that column returns 1 / (1 + Z), Z = sum exp(s).
    """
    q = torch.from_numpy(np.concatenate([qn, qp], axis=-1)).double()       # [R, H, 576]
    k = torch.from_numpy(np.concatenate([kn, kp], axis=-1)).double()       # [n, 576]
    v = torch.from_numpy(np.asarray(kn)).double()                          # [n, 512]
    R, H, _ = q.shape
    n = k.shape[0]
    qh = q.permute(1, 0, 2)                                                # [H, R, 576]
    kh = k.expand(H, n, 576)
    vh = v.expand(H, n, 512)
    attn_mask = None if mask is None else torch.from_numpy(mask)           # [R, n] bool
    o = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=attn_mask, scale=sm_scale)
    kz = torch.cat([kh, torch.zeros(H, 1, 576, dtype=torch.float64)], dim=1)
    vz = torch.cat([torch.cat([vh, torch.zeros(H, n, 1, dtype=torch.float64)], dim=2),
                    torch.cat([torch.zeros(H, 1, 512, dtype=torch.float64),
                               torch.ones(H, 1, 1, dtype=torch.float64)], dim=2)], dim=1)
    mz = None
    if mask is not None:
        mz = torch.cat([attn_mask, torch.ones(R, 1, dtype=torch.bool)], dim=1)
    oz = torch.nn.functional.scaled_dot_product_attention(qh, kz, vz, attn_mask=mz, scale=sm_scale)
    probe = oz[..., 512]                                                   # 1 / (1 + Z)
    lse = torch.log(1.0 / probe - 1.0)
    return o.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


@pytest.mark.parametrize("seed,kv_lens,heads,ps", [(61, [1, 63, 64, 200], 16, 64),
                                                    (62, [130, 7], 5, 1),
                                                    (63, [300], 128, 16)])
def test_decode_matches_sdpa(seed, kv_lens, heads, ps):
    w = _tiny_decode(seed, kv_lens, heads=heads, page_size=ps)
    a = np_inputs(w)
    out, lse = oracle_run(w)
    ckv = a["ckv_cache"].reshape(-1, 512)
    kpe = a["kpe_cache"].reshape(-1, 64)
    ip = a["kv_indptr"]
    for b in range(len(kv_lens)):
        s = a["kv_indices"][ip[b]:ip[b + 1]]
        o, l = _sdpa_row(a["q_nope"][b:b + 1], a["q_pe"][b:b + 1], ckv[s], kpe[s], a["sm_scale"])
        np.testing.assert_allclose(out[b], o[0], rtol=0, atol=1e-11)
        np.testing.assert_allclose(lse[b], l[0], rtol=0, atol=1e-9)


@pytest.mark.parametrize("q_lens,prefixes", [([5, 9], [0, 4]), ([70], [60])])
def test_prefill_matches_sdpa_bottom_right_mask(q_lens, prefixes):
    w = wl.make_prefill(q_lens, prefixes, num_qo_heads=4, page_size=8, seed=71)
    a = np_inputs(w)
    out, lse = oracle_run(w)
    ckv = a["ckv_cache"].reshape(-1, 512)
    kpe = a["kpe_cache"].reshape(-1, 64)
    qo, kp = a["qo_indptr"], a["kv_indptr"]
    for b in range(len(q_lens)):
        s = a["kv_indices"][kp[b]:kp[b + 1]]
        ql, kl = q_lens[b], kp[b + 1] - kp[b]
        # bottom-right causal: query i sees key j iff j <= i + (kl - ql)
        mask = np.arange(kl)[None, :] <= (np.arange(ql)[:, None] + (kl - ql))
        o, l = _sdpa_row(a["q_nope"][qo[b]:qo[b + 1]], a["q_pe"][qo[b]:qo[b + 1]], ckv[s], kpe[s],
                         a["sm_scale"], mask=mask)
        np.testing.assert_allclose(out[qo[b]:qo[b + 1]], o, rtol=0, atol=1e-11)
        np.testing.assert_allclose(lse[qo[b]:qo[b + 1]], l, rtol=0, atol=1e-9)


def test_prefill_without_prefix_matches_sdpa_is_causal():
    """With prefix 0 bottom-right and top-left alignment coincide: SDPA is_causal applies."""
    w = wl.make_prefill([33], [0], num_qo_heads=3, page_size=4, seed=73)
    a = np_inputs(w)
    out, _ = oracle_run(w)
    ckv = a["ckv_cache"].reshape(-1, 512)
    kpe = a["kpe_cache"].reshape(-1, 64)
    s = a["kv_indices"]
    q = torch.from_numpy(np.concatenate([a["q_nope"], a["q_pe"]], -1)).double().permute(1, 0, 2)
    k = torch.from_numpy(np.concatenate([ckv[s], kpe[s]], -1)).double().expand(3, 33, 576)
    v = torch.from_numpy(ckv[s]).double().expand(3, 33, 512)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=a["sm_scale"])
    np.testing.assert_allclose(out, o.permute(1, 0, 2).numpy(), rtol=0, atol=1e-11)


# ---------------------------------------------------------------- invariants

def test_page_permutation_bit_identical():
    w = _tiny_decode(81, [40, 9, 17], heads=4, page_size=4, pool=20)
    a = np_inputs(w)
    out, lse = oracle_run(w)
    perm = np.random.default_rng(5).permutation(w.num_pages)       # new page p' holds old page perm[p']
    inv = np.argsort(perm)
    ckv2 = a["ckv_cache"][perm]
    kpe2 = a["kpe_cache"][perm]
    idx = a["kv_indices"]
    idx2 = inv[idx // 4] * 4 + idx % 4
    out2, lse2 = oracle.mla_decode(a["q_nope"], a["q_pe"], ckv2, kpe2, a["kv_indptr"], idx2, a["sm_scale"])
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_unreferenced_slots_poisoned_with_nan_change_nothing():
    w = _tiny_decode(82, [5, 63, 3], heads=3, page_size=64, pool=6)
    out, lse = oracle_run(w)
    out2, lse2 = oracle_run(wl.poison_unreferenced(w))
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_head_and_request_permutation_equivariance():
    w = _tiny_decode(83, [11, 30, 2, 64], heads=5, page_size=8)
    a = np_inputs(w)
    out, lse = oracle_run(w)
    hp = np.array([3, 0, 4, 1, 2])
    out_h, lse_h = oracle.mla_decode(a["q_nope"][:, hp], a["q_pe"][:, hp], a["ckv_cache"], a["kpe_cache"],
                                     a["kv_indptr"], a["kv_indices"], a["sm_scale"])
    assert np.array_equal(out_h, out[:, hp]) and np.array_equal(lse_h, lse[:, hp])
    rp = [2, 0, 3, 1]
    ip = a["kv_indptr"]
    segs = [a["kv_indices"][ip[r]:ip[r + 1]] for r in rp]
    ip2 = np.concatenate([[0], np.cumsum([len(s) for s in segs])])
    out_r, lse_r = oracle.mla_decode(a["q_nope"][rp], a["q_pe"][rp], a["ckv_cache"], a["kpe_cache"],
                                     ip2, np.concatenate(segs), a["sm_scale"])
    assert np.array_equal(out_r, out[rp]) and np.array_equal(lse_r, lse[rp])


def test_lse_bounds_and_convexity():
    w = _tiny_decode(84, [1, 2, 77, 130], heads=6, page_size=16)
    a = np_inputs(w)
    out, lse = oracle_run(w)
    ckv = a["ckv_cache"].reshape(-1, 512).astype(np.float64)
    kpe = a["kpe_cache"].reshape(-1, 64).astype(np.float64)
    ip = a["kv_indptr"]
    for b in range(4):
        s_idx = a["kv_indices"][ip[b]:ip[b + 1]]
        n = len(s_idx)
        for h in range(6):
            # scores via a plain loop over keys (not the oracle's matmul)
            sc = [a["sm_scale"] * (math.fsum(a["q_nope"][b, h].astype(np.float64) * ckv[t])
                                   + math.fsum(a["q_pe"][b, h].astype(np.float64) * kpe[t])) for t in s_idx]
            mx = max(sc)
            assert mx - 1e-12 <= lse[b, h] <= mx + math.log(n) + 1e-12
            # lse = log sum exp(s), via math.fsum over exact-shifted terms
            np.testing.assert_allclose(lse[b, h], mx + math.log(math.fsum(math.exp(x - mx) for x in sc)),
                                       atol=1e-12)
        lo = ckv[s_idx].min(axis=0)
        hi = ckv[s_idx].max(axis=0)
        assert np.all(out[b] >= lo - 1e-12) and np.all(out[b] <= hi + 1e-12)


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("block", [64, 7])
def test_split_count_invariance(splits, block):
    """Blocked online softmax per split + combine == direct definition (to 1e-12)."""
    w = _tiny_decode(85, [1, 64, 200, 129], heads=4, page_size=16)
    a = np_inputs(w)
    out, lse = oracle_run(w)
    o2, l2 = oracle.mla_decode_split(a["q_nope"], a["q_pe"], a["ckv_cache"], a["kpe_cache"],
                                     a["kv_indptr"], a["kv_indices"], a["sm_scale"], splits, block)
    np.testing.assert_allclose(o2, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, lse, rtol=0, atol=1e-12)


def test_combine_of_disjoint_fragments_is_full_softmax():
    """Merging two fragments of disjoint key sets equals attention over their union."""
    w = _tiny_decode(86, [50], heads=3, page_size=1)
    a = np_inputs(w)
    ckv = a["ckv_cache"].reshape(-1, 512)
    kpe = a["kpe_cache"].reshape(-1, 64)
    s = a["kv_indices"]
    full = oracle.attend(a["q_nope"][0], a["q_pe"][0], ckv[s], kpe[s], a["sm_scale"])
    f1 = oracle.attend(a["q_nope"][0], a["q_pe"][0], ckv[s[:13]], kpe[s[:13]], a["sm_scale"])
    f2 = oracle.attend(a["q_nope"][0], a["q_pe"][0], ckv[s[13:]], kpe[s[13:]], a["sm_scale"])
    empty = (np.zeros((3, 512)), np.full(3, -np.inf))
    o, l = oracle.combine_partials([f1[0], empty[0], f2[0]], [f1[1], empty[1], f2[1]])
    np.testing.assert_allclose(o, full[0], atol=1e-12)
    np.testing.assert_allclose(l, full[1], atol=1e-12)


def test_last_prefill_row_equals_decode():
    w = wl.make_prefill([6, 3], [10, 0], num_qo_heads=3, page_size=4, seed=87)
    a = np_inputs(w)
    out, lse = oracle_run(w)
    last = a["qo_indptr"][1:] - 1
    od, ld = oracle.mla_decode(a["q_nope"][last], a["q_pe"][last], a["ckv_cache"], a["kpe_cache"],
                               a["kv_indptr"], a["kv_indices"], a["sm_scale"])
    assert np.array_equal(out[last], od) and np.array_equal(lse[last], ld)


def test_empty_request_and_short_kv_rejected():
    w = _tiny_decode(88, [0, 3], heads=2, page_size=4)
    out, lse = oracle_run(w)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    w2 = wl.make_prefill([3], [0], num_qo_heads=2, page_size=4, seed=89)
    a = np_inputs(w2)
    with pytest.raises(ValueError):
        oracle.mla_prefill(a["q_nope"], a["q_pe"], a["ckv_cache"], a["kpe_cache"], a["qo_indptr"],
                           np.array([0, 2]), a["kv_indices"][:2], a["sm_scale"])


def test_named_workload_shapes():
    """The generator reproduces the stated structure of the small named workload."""
    w = wl.decode_b4_h16_ps64()
    assert w.kv_lens() == [1, 63, 64, 200] and w.num_pages == 16 and w.page_size == 64
    assert w.q_nope.shape == (4, 16, 512) and w.kpe_cache.shape == (16, 64, 64)
    pages = set((w.kv_indices // 64).tolist())
    assert len(pages) == 7
    p = wl.make_prefill([1024, 2048, 3072, 4096], [0, 1024, 2048, 4096], 1, 64, 1)
    assert p.kv_indptr.tolist() == [0, 1024, 4096, 9216, 17408]
    assert p.qo_indptr.tolist() == [0, 1024, 3072, 6144, 10240]
    assert p.num_pages == 272 and p.visible_keys() == 40899584


# ------------------------------------------------- mutation: pins catch slips

def _mutants():
    def drop_kpe(qn, qp, kn, kp, sc):
        return float(sc) * (np.asarray(qn, np.float64) @ np.asarray(kn, np.float64).T)

    def wrong_sign_pe(qn, qp, kn, kp, sc):
        return float(sc) * (np.asarray(qn, np.float64) @ np.asarray(kn, np.float64).T
                            - np.asarray(qp, np.float64) @ np.asarray(kp, np.float64).T)

    def divide_scale(qn, qp, kn, kp, sc):
        return (np.asarray(qn, np.float64) @ np.asarray(kn, np.float64).T
                + np.asarray(qp, np.float64) @ np.asarray(kp, np.float64).T) / float(sc)
    return {"drop_kpe": drop_kpe, "wrong_sign_pe": wrong_sign_pe, "divide_scale": divide_scale}


@pytest.mark.parametrize("name", ["drop_kpe", "wrong_sign_pe", "divide_scale"])
def test_pins_catch_score_mutants(name, monkeypatch):
    monkeypatch.setattr(mla_oracle, "scores", _mutants()[name])
    with pytest.raises(AssertionError):
        test_decode_matches_sdpa(61, [1, 63, 64, 200], 16, 64)


def test_pins_catch_log2_lse(monkeypatch):
    real_attend = mla_oracle.attend

    def log2_attend(*args):
        o, l = real_attend(*args)
        return o, l / math.log(2)
    monkeypatch.setattr(mla_oracle, "attend", log2_attend)
    with pytest.raises(AssertionError):
        test_single_key_exact()


def test_pins_catch_causal_off_by_one(monkeypatch):
    monkeypatch.setattr(mla_oracle, "visible_len", lambda kv, q, i: kv - q + i)
    with pytest.raises((AssertionError, ValueError, IndexError)):
        test_prefill_matches_sdpa_bottom_right_mask([5, 9], [0, 4])
