"""The allocation-free decode entry point (for callers that cannot allocate device
memory: the split-KV scratch is a static device array inside the library).

Called through the C ABI; its output must match the regular entry point's within the
parity tolerances, on two calls in a row (the static scratch keeps the previous call's
contents, which must not leak into the next result).  This file is collected last so
that a failure here never hides the other tests' results.
"""

import ctypes

import numpy as np
import pytest
import torch

from paged_head_latent_gb300 import workloads as wl
from tests.conftest import require_gpu

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2
LSE_TOL = 1e-3


def _noalloc_call(lib, w, out, lse):
    dims = lib.make_dims(w.batch, w.num_qo_heads, w.num_pages, w.page_size, w.num_kv_indices)
    v = ctypes.c_void_p
    st = lib.lib().mla_paged_decode_noalloc(
        v(w.q_nope.data_ptr()), v(w.q_pe.data_ptr()), v(w.ckv_cache.data_ptr()), v(w.kpe_cache.data_ptr()),
        v(w.kv_indptr.data_ptr()), v(w.kv_indices.data_ptr()), ctypes.c_float(w.sm_scale), v(out.data_ptr()),
        v(lse.data_ptr()), ctypes.byref(dims), 0, v(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.string_of(st)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().copy(), lse.cpu().numpy().copy()


@pytest.mark.parametrize("kv_lens", [[1, 63, 64, 200, 3000, 777, 0, 1500], [5000, 130, 9]])
def test_noalloc_matches_workspace_entry_point(lib, kv_lens):
    require_gpu()
    w = wl.make_decode(kv_lens, num_qo_heads=128, page_size=64, seed=3100 + len(kv_lens)).to("cuda")
    ref_out, ref_lse = lib.run_workload(w)
    torch.cuda.synchronize()
    ref_out = ref_out.float().cpu().numpy()
    ref_lse = ref_lse.cpu().numpy()
    out = torch.empty(w.batch, 128, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.batch, 128, dtype=torch.float32, device="cuda")
    for _ in range(2):  # two calls in a row share the static scratch
        out.fill_(7.0)
        lse.fill_(7.0)
        o, l = _noalloc_call(lib, w, out, lse)
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(l), fin)
        assert np.max(np.abs(o - ref_out)) <= OUT_TOL
        assert np.max(np.abs(l[fin] - ref_lse[fin])) <= LSE_TOL


def test_noalloc_rejects_flags_and_oversized_worker_count(lib):
    require_gpu()
    w = wl.make_decode([64, 65], num_qo_heads=128, page_size=64, seed=3200).to("cuda")
    out = torch.empty(2, 128, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(2, 128, dtype=torch.float32, device="cuda")
    v = ctypes.c_void_p
    args = [v(w.q_nope.data_ptr()), v(w.q_pe.data_ptr()), v(w.ckv_cache.data_ptr()), v(w.kpe_cache.data_ptr()),
            v(w.kv_indptr.data_ptr()), v(w.kv_indices.data_ptr()), ctypes.c_float(w.sm_scale), v(out.data_ptr()),
            v(lse.data_ptr())]
    dims = lib.make_dims(2, 128, w.num_pages, 64, w.num_kv_indices)
    assert lib.lib().mla_paged_decode_noalloc(*args, ctypes.byref(dims), 1, None) == -2
    big = lib.make_dims(2, 128, w.num_pages, 64, w.num_kv_indices, num_workers=4096)
    assert lib.lib().mla_paged_decode_noalloc(*args, ctypes.byref(big), 0, None) == -4
