"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerances (max-abs): 2e-2 on the bf16 output, 1e-3 on the fp32 natural-log lse.
Small cases and the full-size decode workloads compare every element; the full-size
causal prefill compares a dense set of query rows (see below).
"""

import dataclasses

import numpy as np
import pytest
import torch

from paged_head_latent_gb300 import workloads as wl
from tests.conftest import require_gpu
from tests.oracle_io import oracle_run

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2
LSE_TOL = 1e-3


def run_gpu(lib, w, **kw):
    require_gpu()
    wd = w.to("cuda")
    ws = torch.zeros(lib.workload_workspace_bytes(w, kw.get("num_workers", 0)), dtype=torch.uint8, device="cuda")
    out, lse = lib.run_workload(wd, workspace=ws, **kw)
    assert lib.read_device_status(ws) == 0, "device status word reports an error (bounded wait gave up?)"
    return out.float().cpu().numpy(), lse.cpu().numpy()


def assert_close(out, lse, ref_out, ref_lse, what=""):
    assert out.shape == ref_out.shape and lse.shape == ref_lse.shape
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: lse finiteness differs"
    assert np.all(np.isneginf(lse[~fin])), f"{what}: empty rows must have lse = -inf"
    eo = np.max(np.abs(out - ref_out)) if out.size else 0.0
    el = np.max(np.abs(lse[fin] - ref_lse[fin])) if fin.any() else 0.0
    assert eo <= OUT_TOL, f"{what}: max |out - oracle| = {eo}"
    assert el <= LSE_TOL, f"{what}: max |lse - oracle| = {el}"


def check_full(lib, w, **kw):
    out, lse = run_gpu(lib, w, **kw)
    ref_out, ref_lse = oracle_run(w)
    assert_close(out, lse, ref_out, ref_lse, w.name)
    return out, lse


# --------------------------------------------------------------- small decode

def test_decode_small_named(lib):
    check_full(lib, wl.decode_b4_h16_ps64())


@pytest.mark.parametrize("heads", [1, 16, 64, 100, 128])
def test_decode_head_counts(lib, heads):
    w = wl.make_decode([1, 63, 64, 65, 127, 128, 200], num_qo_heads=heads, page_size=64, seed=2000 + heads)
    check_full(lib, w)


@pytest.mark.parametrize("page_size,shuffle", [(1, False), (16, False), (64, True), (32, True)])
def test_decode_page_layouts(lib, page_size, shuffle):
    w = wl.make_decode([3, 64, 129, 700, 31], num_qo_heads=128, page_size=page_size, seed=2100 + page_size,
                       token_shuffle=shuffle)
    check_full(lib, w)


@pytest.mark.parametrize("layout", ["sequential", "mixed"])
def test_decode_small_pages_with_runs(lib, layout):
    """Page size 1 (the small-page kernel instance, two copy warps) whose slots form runs
    of 64: such tiles come in as TMA boxes, the others are copied.  "sequential" makes
    every full tile a run; "mixed" reverses every other tile's slots so runs and copies
    alternate within each request."""
    w = wl.make_decode([700, 129, 64, 300, 5], num_qo_heads=128, page_size=1, seed=2110)
    n = w.num_kv_indices
    idx = torch.arange(n, dtype=torch.int32)
    if layout == "mixed":
        for t0 in range(64, n, 128):  # reverse the slots of every other 64-entry block
            idx[t0:t0 + 64] = idx[t0:t0 + 64].flip(0)
    w = dataclasses.replace(w, kv_indices=idx)
    check_full(lib, w)


# ------------------------------------------------- packed multi-token decode

@pytest.mark.parametrize("q_len,heads,ps,lens", [
    (2, 16, 64, [2, 63, 64, 65, 700, 129]),   # 32 rows per tile
    (4, 32, 64, [4, 5, 200, 1000, 64]),       # 128 rows per tile
    (3, 16, 1, [3, 90, 300]),                 # small pages (copied tiles)
    (1, 128, 64, [1, 100, 640]),              # one token: plain decode through the packed path
])
def test_mtp_small(lib, q_len, heads, ps, lens):
    w = wl.make_mtp(lens, q_len, num_qo_heads=heads, page_size=ps, seed=2800 + q_len * heads + ps)
    check_full(lib, w)


@pytest.mark.parametrize("workers", [1, 3, 40])
def test_mtp_split_rows(lib, workers):
    """Requests split across workers so that some tokens see no key of a segment
    (the first token's horizon ends one key before the last token's)."""
    w = wl.make_mtp([4 * 64 + 1, 130, 2000, 67], 4, num_qo_heads=32, page_size=64, seed=2810)
    check_full(lib, w, num_workers=workers)


def test_mtp_rejects_too_many_rows(lib):
    require_gpu()
    w = wl.make_mtp([10, 20], 2, num_qo_heads=128, page_size=64, seed=2811).to("cuda")
    with pytest.raises(lib.MlaError):
        lib.run_workload(w)


def test_decode_empty_request(lib):
    w = wl.make_decode([0, 5, 0, 130], num_qo_heads=32, page_size=16, seed=2201)
    check_full(lib, w)


def test_decode_all_empty(lib):
    w = wl.make_decode([0, 0], num_qo_heads=8, page_size=16, seed=2202)
    check_full(lib, w)


@pytest.mark.parametrize("batch,ps,workers", [(3000, 16, 0), (5000, 1, 7), (1500, 64, 150)])
def test_decode_many_requests(lib, batch, ps, workers):
    """Thousands of short requests (many rows per worker, most of them whole, some empty):
    the on-device plan walks every request's length and every worker's range."""
    gen = torch.Generator().manual_seed(2210 + batch)
    lens = torch.randint(0, 150, (batch,), generator=gen).tolist()
    w = wl.make_decode(lens, num_qo_heads=16, page_size=ps, seed=2210 + batch)
    check_full(lib, w, num_workers=workers)


@pytest.mark.parametrize("ps", [64, 1])
def test_decode_duplicate_slots(lib, ps):
    """A slot listed twice in a request is two keys (the CSR reading): a duplicate inside a
    64-slot run turns a whole-page tile into a copied one, and one request lists the same
    slot many times."""
    w = wl.make_decode([200, 130, 70], num_qo_heads=64, page_size=ps, seed=2220 + ps)
    idx = w.kv_indices.clone()
    ip = w.kv_indptr.tolist()
    idx[ip[0] + 5] = idx[ip[0] + 3]
    idx[ip[0] + 100] = idx[ip[0] + 150]
    idx[ip[2]:ip[2] + 40] = idx[ip[2]]
    check_full(lib, dataclasses.replace(w, kv_indices=idx))


def test_decode_nan_in_unreferenced_slots(lib):
    w = wl.make_decode([1, 63, 65, 200, 5], num_qo_heads=128, page_size=64, seed=2203, pool_pages=12)
    ref_out, ref_lse = oracle_run(w)
    out, lse = run_gpu(lib, wl.poison_unreferenced(w))
    assert np.all(np.isfinite(out))
    assert_close(out, lse, ref_out, ref_lse, "poisoned")


@pytest.mark.parametrize("workers", [1, 2, 3, 7, 40, 200])
def test_decode_split_count(lib, workers):
    """Any number of split-KV workers gives the oracle's answer (within tolerance)."""
    w = wl.make_decode([1000, 64, 1, 333, 2049], num_qo_heads=128, page_size=64, seed=2300)
    check_full(lib, w, num_workers=workers)


def test_decode_deterministic(lib):
    w = wl.make_decode([1000, 64, 1, 333, 2049], num_qo_heads=128, page_size=64, seed=2301)
    a = run_gpu(lib, w, num_workers=11)
    b = run_gpu(lib, w, num_workers=11)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_decode_long_request_last(lib):
    """Skewed batch with the long request last (the named skew workload has it first)."""
    w = wl.make_decode([512] * 7 + [20000], num_qo_heads=128, page_size=64, seed=2302)
    check_full(lib, w)


@pytest.mark.parametrize("sm_scale", [0.0, -0.05, 0.5])
def test_decode_unusual_scales(lib, sm_scale):
    """Zero scale (uniform weights), a negative scale and a large one (peaked rows), with
    tails that leave tiles partly empty."""
    w = dataclasses.replace(wl.make_decode([1, 63, 65, 200, 777], num_qo_heads=128, page_size=64, seed=2304),
                            sm_scale=sm_scale)
    check_full(lib, w)


def test_decode_dominant_key(lib):
    """One key per request lines up with head 0's query, so that head's softmax puts all
    its weight on that key (its score is ~20 above the rest): lse must track that
    single score to the tolerance."""
    w = wl.make_decode([300, 64, 1000], num_qo_heads=128, page_size=64, seed=2305)
    ckv = w.ckv_cache.clone().view(-1, 512)
    kpe = w.kpe_cache.clone().view(-1, 64)
    for b in range(w.batch):
        slot = int(w.kv_indices[int(w.kv_indptr[b]) + 17 % max(1, int(w.kv_indptr[b + 1] - w.kv_indptr[b]))])
        ckv[slot] = (w.q_nope[b, 0].float() * 0.5).to(torch.bfloat16)
        kpe[slot] = (w.q_pe[b, 0].float() * 0.5).to(torch.bfloat16)
    w = dataclasses.replace(w, ckv_cache=ckv.view_as(w.ckv_cache), kpe_cache=kpe.view_as(w.kpe_cache))
    check_full(lib, w)


def test_bound_call_repeats_the_call(lib):
    """bind_workload's prepared call gives the same bits as the checked call, twice."""
    require_gpu()
    w = wl.make_decode([300, 64, 1000], num_qo_heads=128, page_size=64, seed=2306).to("cuda")
    dims = lib.make_dims(w.batch, w.num_qo_heads, w.num_pages, w.page_size, w.num_kv_indices)
    ws = torch.zeros(lib.workspace_bytes(dims, False), dtype=torch.uint8, device="cuda")
    ref_out, ref_lse = lib.run_workload(w, workspace=ws)
    ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
    out = torch.empty_like(ref_out)
    lse = torch.empty_like(ref_lse)
    stream = torch.cuda.current_stream()
    call = lib.bind_workload(w, out, lse, ws, stream)
    for _ in range(2):
        out.zero_()
        call()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


# ------------------------------------------------------ sparse (top-k) decode

@pytest.mark.parametrize("kv_lens,topk,heads,s_q,ps", [
    ([5, 130, 700], 64, 128, 1, 64),    # short requests padded with -1
    ([300, 1000], 200, 16, 2, 16),      # two query tokens per request, ragged last tile
    ([2049, 90], 128, 128, 1, 1),       # page size 1
    ([64], 64, 1, 1, 64),               # one head, exactly one tile
])
def test_sparse_small(lib, kv_lens, topk, heads, s_q, ps):
    w = wl.make_sparse_decode(kv_lens, topk, num_qo_heads=heads, page_size=ps, seed=4200 + topk + heads, s_q=s_q)
    check_full(lib, w)


def test_sparse_out_of_range_and_duplicate_entries(lib):
    """-1, large and negative entries anywhere in a row are skipped; a duplicate counts twice."""
    w = wl.make_sparse_decode([400, 250], 96, num_qo_heads=64, page_size=64, seed=4210)
    idx = w.indices.clone()
    n = w.num_pages * w.page_size
    idx[0, 3] = -1
    idx[0, 40] = n
    idx[1, 0] = -77
    idx[1, 90] = n + 1000
    idx[1, 91] = idx[1, 5]
    w = dataclasses.replace(w, indices=idx, kv_indices=idx.reshape(-1).clone())
    check_full(lib, w)


@pytest.mark.parametrize("workers", [1, 3, 40])
def test_sparse_split_count(lib, workers):
    w = wl.make_sparse_decode([3000, 100, 1500, 20], 700, num_qo_heads=128, page_size=64, seed=4220)
    check_full(lib, w, num_workers=workers)


def test_sparse_row_of_padding_only(lib):
    w = wl.make_sparse_decode([300, 300, 300], 128, num_qo_heads=32, page_size=64, seed=4230)
    idx = w.indices.clone()
    idx[1, :] = -1
    w = dataclasses.replace(w, indices=idx, kv_indices=idx.reshape(-1).clone())
    for workers in (0, 5):
        out, lse = check_full(lib, w, num_workers=workers)
        assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))


def test_sparse_nan_in_unreferenced_slots(lib):
    w = wl.make_sparse_decode([500, 129], 100, num_qo_heads=128, page_size=64, seed=4240)
    ref_out, ref_lse = oracle_run(w)
    out, lse = run_gpu(lib, wl.poison_unreferenced(w))
    assert np.all(np.isfinite(out))
    assert_close(out, lse, ref_out, ref_lse, "sparse poisoned")


def test_decode_skips_out_of_range_slot(lib):
    """A CSR index outside the cache is not a key of the row (the same rule as sparse
    padding): the result is the oracle's over the remaining keys."""
    w = wl.make_decode([70, 200], num_qo_heads=16, page_size=64, seed=4250)
    bad = w.kv_indices.clone()
    bad[10] = w.num_pages * w.page_size + 3
    w_bad = dataclasses.replace(w, kv_indices=bad)
    keep = torch.ones(bad.numel(), dtype=torch.bool)
    keep[10] = False
    ip = w.kv_indptr.clone()
    ip[1:] -= 1
    w_ref = dataclasses.replace(w, kv_indices=bad[keep].clone(), kv_indptr=ip)
    ref_out, ref_lse = oracle_run(w_ref)
    out, lse = run_gpu(lib, w_bad)
    assert_close(out, lse, ref_out, ref_lse, "out-of-range slot")


# -------------------------------------------------------------- small prefill

@pytest.mark.parametrize("q_lens,prefixes,heads,ps", [
    ([5, 3], [2, 64], 2, 64),
    ([64, 65, 1], [0, 63, 200], 16, 64),
    ([130, 17], [70, 0], 128, 1),
    ([100], [0], 128, 16),
])
def test_prefill_small(lib, q_lens, prefixes, heads, ps):
    w = wl.make_prefill(q_lens, prefixes, num_qo_heads=heads, page_size=ps, seed=2400 + sum(q_lens))
    check_full(lib, w)


@pytest.mark.parametrize("workers", [1, 5, 76])
def test_prefill_split_count(lib, workers):
    w = wl.make_prefill([40, 90], [30, 100], num_qo_heads=64, page_size=64, seed=2500)
    check_full(lib, w, num_workers=workers)


# ----------------------------------------------------------- robustness / API

def test_validate_flag(lib):
    require_gpu()
    w = wl.make_decode([5, 70], num_qo_heads=16, page_size=64, seed=2600).to("cuda")
    ws = torch.zeros(lib.workspace_bytes(lib.make_dims(2, 16, w.num_pages, 64, w.num_kv_indices), False),
                     dtype=torch.uint8, device="cuda")
    lib.run_workload(w, workspace=ws, flags=lib.MLA_VALIDATE)
    assert lib.read_device_status(ws) == 0
    bad = w.kv_indices.clone()
    bad[3] = w.num_pages * w.page_size + 5  # out of range: reads zeros, flagged
    w2 = dataclasses.replace(w, kv_indices=bad)
    lib.run_workload(w2, workspace=ws, flags=lib.MLA_VALIDATE)
    assert lib.read_device_status(ws) == -6
    assert lib.read_device_status(ws) == 0  # the word was cleared


def test_cuda_graph_capture(lib):
    require_gpu()
    w = wl.make_decode([100, 2000, 7], num_qo_heads=128, page_size=64, seed=2700).to("cuda")
    out = torch.empty(3, 128, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(3, 128, dtype=torch.float32, device="cuda")
    ws = torch.zeros(lib.workspace_bytes(lib.make_dims(3, 128, w.num_pages, 64, w.num_kv_indices), False),
                     dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        lib.run_workload(w, out=out, lse=lse, workspace=ws, stream=s)  # warm-up (tensor maps cached)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref = (out.clone(), lse.clone())
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lib.run_workload(w, out=out, lse=lse, workspace=ws, stream=torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])


# ------------------------------------------------------- full-size workloads
#
# The named full-size workloads run in the launch configuration the benchmark times
# (default worker count, one call) and are compared with the oracle element by element:
# every output and lse value of the three decode workloads and of the packed
# multi-token workload; for the causal prefill (about 11 TFLOP in float64) every eighth
# query row plus every row whose visible length sits at a 64-key tile boundary, the first
# and last row of every request, and every row where a split-KV worker's range starts or
# ends.

FULL_DECODE = ["decode_b64_h128_ps64", "decode_b128_h128_ps1", "decode_b32_h128_skew", "sparse_b64_h128_topk2048"]


@pytest.mark.parametrize("name", FULL_DECODE)
def test_full_size_decode_every_element(lib, name):
    w = wl.by_name(name)
    out, lse = run_gpu(lib, w)
    ref_out, ref_lse = oracle_run(w)
    assert_close(out, lse, ref_out, ref_lse, name)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


def test_full_size_mtp_every_element(lib):
    w = wl.by_name("mtp_b64_h16_q4_ps64")
    out, lse = run_gpu(lib, w)
    ref_out, ref_lse = oracle_run(w)
    assert_close(out, lse, ref_out, ref_lse, "mtp_b64_h16_q4_ps64")


def worker_boundary_rows(w, workers, row_cost=5, tile=64):
    """Query rows in which a split-KV worker's range starts or ends, for a partition of
    the cost sequence (a row start counts row_cost units, a 64-key tile one unit) into
    ``workers`` even parts.  Used only to choose which rows to check."""
    qo = w.qo_indptr.tolist()
    kp = w.kv_indptr.tolist()
    spans = []  # (first cost unit, last cost unit, row)
    c = 0
    for b in range(w.batch):
        ql, kl = qo[b + 1] - qo[b], kp[b + 1] - kp[b]
        for i in range(ql):
            vis = kl - ql + i + 1
            if vis <= 0:
                continue
            n = row_cost + -(-vis // tile)
            spans.append((c, c + n - 1, qo[b] + i))
            c += n
    bounds = sorted({k * c // workers for k in range(1, workers)})
    rows, j = set(), 0
    for x in bounds:
        while spans[j][1] < x:
            j += 1
        rows.add(spans[j][2])
        if j > 0:
            rows.add(spans[j - 1][2])
    return rows


def test_full_size_prefill_dense_rows(lib):
    w = wl.prefill_causal_h128()
    out, lse = run_gpu(lib, w)
    qo, kp = w.qo_indptr.tolist(), w.kv_indptr.tolist()
    rows = set(range(0, w.rows, 8))
    for b in range(w.batch):
        ql, kl = qo[b + 1] - qo[b], kp[b + 1] - kp[b]
        rows.update((qo[b], qo[b + 1] - 1))
        for i in range(ql):
            if (kl - ql + i + 1) % 64 in (0, 1):
                rows.add(qo[b] + i)
    rows |= worker_boundary_rows(w, lib.default_num_workers())
    rows = sorted(rows)
    ref_out, ref_lse = oracle_run(w, rows=rows)
    assert_close(out[rows], lse[rows], ref_out[rows], ref_lse[rows], f"prefill_causal_h128 ({len(rows)} rows)")
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
