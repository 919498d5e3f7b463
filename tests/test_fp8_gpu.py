"""FP8-KV decode on the GPU against the float64 oracle.

The cache is the 656-byte token layout of the FlashMLA notes ("FP8 KV Cache
Quantization and Dequantization"); the oracle dequantises it to BF16 first.  Besides
the parity tolerances, the kernel's dequantisation is checked exactly: the FP8 decode
must equal, bit for bit, the bf16 decode (same kernel instance family, same tile
order) run on the cache the oracle dequantised.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_head_latent_gb300 import workloads as wl
from tests.conftest import require_gpu
from tests.oracle_io import oracle_run

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2
LSE_TOL = 1e-3


def _close(out, lse, ref_out, ref_lse, what):
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(l), fin), what
    assert np.max(np.abs(o - ref_out)) <= OUT_TOL, what
    assert np.max(np.abs(l[fin] - ref_lse[fin])) <= LSE_TOL, what


def _dequantised_bf16(w):
    ckv, kpe = oracle.dequantize_fp8_cache(w.kv_fp8.numpy())
    return (torch.from_numpy(ckv).to(torch.bfloat16), torch.from_numpy(kpe).to(torch.bfloat16))


@pytest.mark.parametrize("page_size,heads", [(1, 16), (16, 128), (64, 128), (64, 16)])
def test_fp8_decode_small(lib, page_size, heads):
    require_gpu()
    lens = [1, 0, 63, 64, 65, 200, 1500, 3000]
    w = wl.quantize_fp8(wl.make_decode(lens, heads, page_size, seed=6000 + page_size + heads))
    ref_out, ref_lse = oracle_run(w)
    wd = w.to("cuda")
    out, lse = lib.run_workload(wd)
    torch.cuda.synchronize()
    _close(out, lse, ref_out, ref_lse, f"fp8 ps{page_size} h{heads}")
    if page_size % 64 != 0:
        # The bf16 decode of the oracle's dequantised cache runs the same copy-path
        # arithmetic on the same tiles: equal bit for bit iff the dequantisation is.
        ckv, kpe = _dequantised_bf16(w)
        o2, l2 = lib.mla_paged_decode(wd.q_nope, wd.q_pe, ckv.cuda(), kpe.cuda(), wd.kv_indptr, wd.kv_indices,
                                      w.sm_scale)
        torch.cuda.synchronize()
        assert torch.equal(out, o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("page_size,heads", [(32, 100), (1, 1), (64, 33)])
def test_fp8_decode_odd_shapes(lib, page_size, heads):
    require_gpu()
    lens = [2, 77, 640, 129, 1]
    w = wl.quantize_fp8(wl.make_decode(lens, heads, page_size, seed=6400 + page_size + heads))
    ref_out, ref_lse = oracle_run(w)
    out, lse = lib.run_workload(w.to("cuda"))
    torch.cuda.synchronize()
    _close(out, lse, ref_out, ref_lse, f"fp8 ps{page_size} h{heads}")


@pytest.mark.parametrize("workers", [1, 3, 40])
def test_fp8_split_counts(lib, workers):
    """Split rows (and, with one worker, one worker walking every tile through the FP8
    producer's staging ring many times over)."""
    require_gpu()
    w = wl.quantize_fp8(wl.make_decode([3000, 65, 1999, 700], 128, 64, seed=6500 + workers))
    ref_out, ref_lse = oracle_run(w)
    wd = w.to("cuda")
    ws = torch.zeros(lib.workload_workspace_bytes(wd, workers), dtype=torch.uint8, device="cuda")
    out, lse = lib.run_workload(wd, workspace=ws, num_workers=workers)
    torch.cuda.synchronize()
    assert lib.read_device_status(ws) == 0
    _close(out, lse, ref_out, ref_lse, f"fp8 workers={workers}")


def test_fp8_full_size_every_element(lib):
    require_gpu()
    w = wl.by_name("fp8_b64_h128_ps64")
    out, lse = lib.run_workload(w.to("cuda"))
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle_run(w)
    _close(out, lse, ref_out, ref_lse, "fp8_b64_h128_ps64")


def test_fp8_sparse(lib):
    require_gpu()
    w = wl.quantize_fp8(wl.make_sparse_decode([3000, 100, 5000, 64], 256, 128, 16, seed=6100))
    ref_out, ref_lse = oracle_run(w)
    out, lse = lib.run_workload(w.to("cuda"))
    torch.cuda.synchronize()
    _close(out, lse, ref_out, ref_lse, "fp8 sparse")


def test_fp8_unreferenced_nan_codes_and_out_of_range_slot(lib):
    """Tokens no request lists hold E4M3 NaN codes and NaN scales; one listed slot lies
    outside the cache (not a key).  Neither may reach the output."""
    require_gpu()
    w = wl.quantize_fp8(wl.make_decode([70, 200, 40], 16, 64, seed=6200))
    used = torch.zeros(w.num_pages * w.page_size, dtype=torch.bool)
    used[w.kv_indices.long()] = True
    kv = w.kv_fp8.clone().view(-1, 656)
    kv[~used] = 0x7F
    bad = w.kv_indices.clone()
    bad[5] = w.num_pages * w.page_size + 9
    keep = torch.ones(bad.numel(), dtype=torch.bool)
    keep[5] = False
    ip = w.kv_indptr.clone()
    ip[1:] -= 1
    import dataclasses
    w_bad = dataclasses.replace(w, kv_fp8=kv.view_as(w.kv_fp8), kv_indices=bad)
    w_ref = dataclasses.replace(w, kv_indices=bad[keep].clone(), kv_indptr=ip)
    ref_out, ref_lse = oracle_run(w_ref)
    out, lse = lib.run_workload(w_bad.to("cuda"))
    torch.cuda.synchronize()
    _close(out, lse, ref_out, ref_lse, "fp8 poisoned")


def test_fp8_rejects_misaligned_cache(lib):
    require_gpu()
    w = wl.quantize_fp8(wl.make_decode([70], 16, 64, seed=6300)).to("cuda")
    buf = torch.empty(w.kv_fp8.numel() + 16, dtype=torch.uint8, device="cuda")
    dims = lib.make_dims(1, 16, w.num_pages, 64, w.num_kv_indices)
    ws = torch.zeros(lib.workspace_bytes(dims, False), dtype=torch.uint8, device="cuda")
    out = torch.empty(1, 16, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 16, dtype=torch.float32, device="cuda")
    v = ctypes.c_void_p
    st = lib.lib().mla_paged_decode_fp8(v(w.q_nope.data_ptr()), v(w.q_pe.data_ptr()), v(buf.data_ptr() + 8),
                                        v(w.kv_indptr.data_ptr()), v(w.kv_indices.data_ptr()),
                                        ctypes.c_float(w.sm_scale), v(out.data_ptr()), v(lse.data_ptr()),
                                        ctypes.byref(dims), v(ws.data_ptr()), ws.numel(), 0, None)
    assert st == -3
