"""Marshalling between seeded workloads (bf16 torch tensors) and the oracle (numpy).

bf16 -> float32 is exact, so the oracle sees exactly the values the GPU sees.
No attention arithmetic here.
"""

import numpy as np
import torch


def np_inputs(w):
    d = dict(
        q_nope=w.q_nope.float().numpy(),
        q_pe=w.q_pe.float().numpy(),
        ckv_cache=w.ckv_cache.float().numpy(),
        kpe_cache=w.kpe_cache.float().numpy(),
        kv_indptr=w.kv_indptr.numpy().astype(np.int64),
        kv_indices=w.kv_indices.numpy().astype(np.int64),
        sm_scale=w.sm_scale,
    )
    if w.qo_indptr is not None:
        d["qo_indptr"] = w.qo_indptr.numpy().astype(np.int64)
    if w.indices is not None:
        d["indices"] = w.indices.numpy().astype(np.int64)
    return d


def oracle_run(w, rows=None):
    import oracle
    a = np_inputs(w)
    if w.kind == "decode_fp8":
        return oracle.mla_decode_fp8(a["q_nope"], a["q_pe"], w.kv_fp8.numpy(), a["kv_indptr"], a["kv_indices"],
                                     a["sm_scale"])
    if w.kind == "sparse_fp8":
        return oracle.mla_sparse_decode_fp8(a["q_nope"], a["q_pe"], w.kv_fp8.numpy(), a["indices"], a["sm_scale"])
    if w.kind == "sparse":
        return oracle.mla_sparse_decode(a["q_nope"], a["q_pe"], a["ckv_cache"], a["kpe_cache"], a["indices"],
                                        a["sm_scale"])
    if w.kind == "decode":
        out, lse = oracle.mla_decode(a["q_nope"], a["q_pe"], a["ckv_cache"], a["kpe_cache"],
                                     a["kv_indptr"], a["kv_indices"], a["sm_scale"])
        return out, lse
    return oracle.mla_prefill(a["q_nope"], a["q_pe"], a["ckv_cache"], a["kpe_cache"],
                              a["qo_indptr"], a["kv_indptr"], a["kv_indices"], a["sm_scale"],
                              rows=rows)


def oracle_rows_decode(w, rows):
    """Oracle output for selected decode requests only (for full-size sampling)."""
    import oracle
    ckv = w.ckv_cache.view(-1, 512)
    kpe = w.kpe_cache.view(-1, 64)
    ip = w.kv_indptr.tolist()
    res = {}
    for r in rows:
        slots = w.kv_indices[ip[r]:ip[r + 1]].long()
        o, l = oracle.attend(w.q_nope[r].float().numpy(), w.q_pe[r].float().numpy(),
                             ckv[slots].float().numpy(), kpe[slots].float().numpy(), w.sm_scale)
        res[r] = (o, l)
    return res


def oracle_rows_prefill(w, rows):
    """Oracle output for selected prefill query rows only."""
    import oracle
    ckv = w.ckv_cache.view(-1, 512)
    kpe = w.kpe_cache.view(-1, 64)
    qo = w.qo_indptr.tolist()
    kp = w.kv_indptr.tolist()
    res = {}
    for r in rows:
        b = max(i for i in range(len(qo) - 1) if qo[i] <= r)
        i = r - qo[b]
        n = oracle.visible_len(kp[b + 1] - kp[b], qo[b + 1] - qo[b], i)
        slots = w.kv_indices[kp[b]:kp[b] + n].long()
        o, l = oracle.attend(w.q_nope[r].float().numpy(), w.q_pe[r].float().numpy(),
                             ckv[slots].float().numpy(), kpe[slots].float().numpy(), w.sm_scale)
        res[r] = (o, l)
    return res


def to_lists(a):
    return np.asarray(a).tolist()
