"""The allocation-free decode entry point.

Some callers cannot call cudaMalloc (a plugin running inside another framework's memory
pool, code that must not allocate once it is serving, a context where an allocation
would synchronise the device); for them the library keeps the split-KV scratch in a
static device array.  These tests call that entry point through the C ABI and check its
output against the float64 oracle and against the regular entry point (with a freshly
zeroed workspace), within the parity tolerances, on consecutive calls: the static
scratch keeps the previous call's contents, which must never leak into the next result,
even when the previous call had another head count and worker layout.  This file is
collected last so that a failure here never hides the other tests' results.
"""

import ctypes

import numpy as np
import pytest
import torch

from paged_head_latent_gb300 import workloads as wl
from tests.conftest import require_gpu
from tests.oracle_io import oracle_run

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
    assert lib.noalloc_read_status() == 0, "device status of the allocation-free call reports an error"
    return out.float().cpu().numpy().copy(), lse.cpu().numpy().copy()


def _close(o, l, ref_o, ref_l, what):
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin), what
    assert np.max(np.abs(o - ref_o)) <= OUT_TOL, what
    assert np.max(np.abs(l[fin] - ref_l[fin])) <= LSE_TOL, what


def _workspace_call(lib, w):
    ws = torch.zeros(lib.workload_workspace_bytes(w), dtype=torch.uint8, device="cuda")
    o, l = lib.run_workload(w, workspace=ws)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), l.cpu().numpy()


@pytest.mark.parametrize("kv_lens", [[1, 63, 64, 200, 3000, 777, 0, 1500], [5000, 130, 9]])
def test_noalloc_matches_oracle_and_workspace_entry_point(lib, kv_lens):
    require_gpu()
    w_cpu = wl.make_decode(kv_lens, num_qo_heads=128, page_size=64, seed=3100 + len(kv_lens))
    ref_out, ref_lse = oracle_run(w_cpu)
    w = w_cpu.to("cuda")
    ws_out, ws_lse = _workspace_call(lib, w)
    out = torch.empty(w.batch, 128, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.batch, 128, dtype=torch.float32, device="cuda")
    for k in range(2):  # two calls in a row share the static scratch
        out.fill_(7.0)
        lse.fill_(7.0)
        o, l = _noalloc_call(lib, w, out, lse)
        _close(o, l, ref_out, ref_lse, f"call {k} vs oracle")
        _close(o, l, ws_out, ws_lse, f"call {k} vs workspace entry point")


def test_noalloc_after_a_call_with_another_layout(lib):
    """A 16-head call with split rows, then a 128-head call whose long request is merged
    in two levels: the second call's worker count, head count and so the scratch layout
    differ from the first's, and its long row needs the merge counters."""
    require_gpu()
    first = wl.make_decode([3000, 777, 1500, 64, 2049], num_qo_heads=16, page_size=64, seed=3150).to("cuda")
    o1 = torch.empty(first.batch, 16, 512, dtype=torch.bfloat16, device="cuda")
    l1 = torch.empty(first.batch, 16, dtype=torch.float32, device="cuda")
    second_cpu = wl.make_decode([131072] + [512] * 7, num_qo_heads=128, page_size=64, seed=3151)
    ref_out, ref_lse = oracle_run(second_cpu)
    second = second_cpu.to("cuda")
    ws_out, ws_lse = _workspace_call(lib, second)
    o2 = torch.empty(second.batch, 128, 512, dtype=torch.bfloat16, device="cuda")
    l2 = torch.empty(second.batch, 128, dtype=torch.float32, device="cuda")
    for k in range(2):
        _noalloc_call(lib, first, o1, l1)
        o2.fill_(7.0)
        l2.fill_(7.0)
        o, l = _noalloc_call(lib, second, o2, l2)
        _close(o, l, ref_out, ref_lse, f"round {k} vs oracle")
        _close(o, l, ws_out, ws_lse, f"round {k} vs workspace entry point")


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
