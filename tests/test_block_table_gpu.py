"""The block-table adapter on the GPU.

The conversion (block table + sequence lengths -> token-slot CSR) is integer work, so
it must equal the oracle's conversion bit for bit; the block-table decode must match
the float64 oracle within the parity tolerances, and equal bit for bit the CSR decode
run on the adapter's CSR (the same kernel on the same keys).  Inputs follow the prims_ts
wrapper's block_tables [batch, max_num_blocks] and seq_lens, with junk (random page ids
or -1) in every table entry a request does not use.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_head_latent_gb300 import workloads as wl
from tests.conftest import require_gpu

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2
LSE_TOL = 1e-3

CASES = [
    (1, [1, 0, 37, 500, 4096, 3]),
    (16, [0, 15, 16, 17, 900, 2048]),
    (64, [1, 63, 64, 65, 5000, 0, 777]),
]


def _f64(*ts):
    return [t.float().numpy() for t in ts]


@pytest.mark.parametrize("page_size,lens", CASES)
@pytest.mark.parametrize("junk", ["random", "minus1"])
def test_conversion_matches_oracle(lib, page_size, lens, junk):
    """Lengths of 0, partial and full pages, one negative length and one longer than the
    table (clamped), and one page id of -2 inside a request's blocks."""
    require_gpu()
    max_blocks = max(-(-l // page_size) for l in lens) + 2
    x = wl.make_block_table_decode(lens + [-3, max_blocks * page_size + 50], 1, page_size, max_blocks,
                                   seed=5200 + page_size, junk=junk)
    t = x.block_table.clone()
    t[2, 0] = -2
    ref_ptr, ref_idx = oracle.block_table_to_csr(t.numpy(), x.seq_lens.numpy(), page_size)
    ptr, idx = lib.block_table_to_csr(t.cuda(), x.seq_lens.cuda(), page_size)
    torch.cuda.synchronize()
    assert ptr.cpu().tolist() == ref_ptr.tolist()
    assert idx[:int(ref_ptr[-1])].cpu().tolist() == ref_idx.tolist()
    assert (ref_idx == -1).sum() == min(lens[2], page_size)


def test_conversion_stops_at_capacity(lib):
    """Positions at or past the capacity are never written; kv_indptr still counts them."""
    require_gpu()
    x = wl.make_block_table_decode([100, 300, 50], 1, 16, 20, seed=5250)
    ref_ptr, ref_idx = oracle.block_table_to_csr(x.block_table.numpy(), x.seq_lens.numpy(), 16)
    cap = 250
    bt, sl = x.block_table.cuda(), x.seq_lens.cuda()
    ptr = torch.full((4,), -7, dtype=torch.int32, device="cuda")
    idx = torch.full((cap + 64,), -7, dtype=torch.int32, device="cuda")
    v = ctypes.c_void_p
    st = lib.lib().mla_block_table_to_csr(v(bt.data_ptr()), v(sl.data_ptr()), 3, 20, 16, v(ptr.data_ptr()),
                                          v(idx.data_ptr()), cap, v(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert ptr.cpu().tolist() == ref_ptr.tolist()
    assert idx[:cap].cpu().tolist() == ref_idx[:cap].tolist()
    assert (idx[cap:] == -7).all()


def test_conversion_rejects_bad_arguments(lib):
    require_gpu()
    v = ctypes.c_void_p
    buf = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = v(buf.data_ptr())
    f = lib.lib().mla_block_table_to_csr
    assert f(p, p, 1, 1, 0, p, p, 4, None) == -2        # page_size < 1
    assert f(p, p, -1, 1, 1, p, p, 4, None) == -2       # negative batch
    assert f(p, p, 1, 1 << 20, 1 << 12, p, p, 4, None) == -2  # table wider than int32 slots
    assert f(p, p, 1, 1, 1, None, p, 4, None) == -1     # no kv_indptr
    assert f(p, None, 1, 1, 1, p, p, 4, None) == -1     # no seq_lens


@pytest.mark.parametrize("page_size", [1, 16, 64])
def test_block_table_decode(lib, page_size):
    """128 heads, split and whole rows, an empty request, and a page id outside the cache
    inside one request's blocks (its slots are not keys)."""
    require_gpu()
    lens = [1, 0, 63, 64, 65, 1500, 3000, 200, 4096]
    max_blocks = -(-4096 // page_size) + 3
    x = wl.make_block_table_decode(lens, 128, page_size, max_blocks, seed=5300 + page_size)
    t = x.block_table.clone()
    t[5, 1] = x.num_pages + 11
    ref_out, ref_lse = oracle.mla_decode_block_table(*_f64(x.q_nope, x.q_pe, x.ckv_cache, x.kpe_cache),
                                                     t.numpy(), x.seq_lens.numpy(), x.sm_scale)
    xd, td = x.to("cuda"), t.cuda()
    out, lse = lib.mla_paged_decode_block_table(xd.q_nope, xd.q_pe, xd.ckv_cache, xd.kpe_cache, td, xd.seq_lens,
                                                x.sm_scale)
    torch.cuda.synchronize()
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(l), fin)
    assert np.max(np.abs(o - ref_out)) <= OUT_TOL
    assert np.max(np.abs(l[fin] - ref_lse[fin])) <= LSE_TOL
    # The same keys through the CSR entry point: the same kernel, bit for bit.
    ptr, idx = lib.block_table_to_csr(td, xd.seq_lens, page_size)
    out2, lse2 = lib.mla_paged_decode(xd.q_nope, xd.q_pe, xd.ckv_cache, xd.kpe_cache, ptr, idx, x.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_block_table_decode_in_a_cuda_graph(lib):
    """The conversion and the decode run inside a captured CUDA graph; a replay after the
    lengths changed in place gives the direct call's result for the new lengths."""
    require_gpu()
    lens = [300, 70, 1024, 5]
    x = wl.make_block_table_decode(lens, 128, 64, 20, seed=5400).to("cuda")
    seq = x.seq_lens.clone()
    out = torch.empty(4, 128, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(4, 128, dtype=torch.float32, device="cuda")
    dims = lib.make_dims(4, 128, x.num_pages, 64, 0)
    ws = torch.zeros(lib.lib().mla_workspace_bytes_block_table(ctypes.byref(dims), 20), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        lib.mla_paged_decode_block_table(x.q_nope, x.q_pe, x.ckv_cache, x.kpe_cache, x.block_table, seq,
                                         x.sm_scale, out=out, lse=lse, workspace=ws)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        lib.mla_paged_decode_block_table(x.q_nope, x.q_pe, x.ckv_cache, x.kpe_cache, x.block_table, seq,
                                         x.sm_scale, out=out, lse=lse, workspace=ws)
    for new_lens in ([300, 70, 1024, 5], [1, 1280, 64, 0]):
        seq.copy_(torch.tensor(new_lens, dtype=torch.int32))
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        ref_out, ref_lse = lib.mla_paged_decode_block_table(x.q_nope, x.q_pe, x.ckv_cache, x.kpe_cache,
                                                            x.block_table, seq.clone(), x.sm_scale)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
