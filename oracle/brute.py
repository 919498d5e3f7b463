"""Scalar pure-Python brute force for tiny paged-MLA cases.

TEST INFRASTRUCTURE ONLY (see mla_oracle.py).  Written independently of
mla_oracle.py -- no shared helpers -- so that the two can pin each other.  It
uses nothing but Python floats (IEEE double) and ``math``; every sum is an
explicit loop.  Meant for B <= 3, H <= 4, kv <= ~70.

Definition followed: flashinfer-bench "MLA Paged" (decode / prefill inputs and
outputs), V = the ckv latent (Modular MAX "mla_decoding_single_batch"), natural-log
lse, bottom-right causal prefill.
"""

from __future__ import annotations

import math


def _row(cache, slot, width):
    """Row ``slot`` of a paged cache given as nested lists [pages][page_size][width]."""
    page_size = len(cache[0])
    page, off = divmod(slot, page_size)
    r = cache[page][off]
    assert len(r) == width
    return r


def _one_query(qn, qp, ckv, kpe, slots, sm_scale):
    """All heads of one query over the listed slots -> (out [H][512], lse [H])."""
    heads = len(qn)
    out, lse = [], []
    for h in range(heads):
        if not slots:
            out.append([0.0] * 512)
            lse.append(-math.inf)
            continue
        s = []
        for t in slots:
            kn = _row(ckv, t, 512)
            kp = _row(kpe, t, 64)
            dot = 0.0
            for d in range(512):
                dot += qn[h][d] * kn[d]
            for d in range(64):
                dot += qp[h][d] * kp[d]
            s.append(sm_scale * dot)
        big = max(s)
        z = 0.0
        for x in s:
            z += math.exp(x - big)
        l = big + math.log(z)
        o = [0.0] * 512
        for x, t in zip(s, slots):
            w = math.exp(x - l)
            kn = _row(ckv, t, 512)
            for d in range(512):
                o[d] += w * kn[d]
        out.append(o)
        lse.append(l)
    return out, lse


def brute_decode(q_nope, q_pe, ckv_cache, kpe_cache, kv_indptr, kv_indices, sm_scale):
    """Arguments as nested Python lists / ints; returns (out, lse) as nested lists."""
    outs, lses = [], []
    for b in range(len(kv_indptr) - 1):
        slots = list(kv_indices[kv_indptr[b]:kv_indptr[b + 1]])
        o, l = _one_query(q_nope[b], q_pe[b], ckv_cache, kpe_cache, slots, sm_scale)
        outs.append(o)
        lses.append(l)
    return outs, lses


def brute_prefill(q_nope, q_pe, ckv_cache, kpe_cache, qo_indptr, kv_indptr, kv_indices, sm_scale):
    outs, lses = [], []
    for b in range(len(qo_indptr) - 1):
        q_len = qo_indptr[b + 1] - qo_indptr[b]
        kv_len = kv_indptr[b + 1] - kv_indptr[b]
        slots = list(kv_indices[kv_indptr[b]:kv_indptr[b + 1]])
        for i in range(q_len):
            r = qo_indptr[b] + i
            n = kv_len - q_len + i + 1
            o, l = _one_query(q_nope[r], q_pe[r], ckv_cache, kpe_cache, slots[:n], sm_scale)
            outs.append(o)
            lses.append(l)
    return outs, lses
