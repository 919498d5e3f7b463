"""The kernels' bounded waits: a wait that runs out gives up cleanly and is reported.

A test hook makes the attention kernel's producer (split-KV worker 0, first CTA of the
pair) skip one tile's loads and arrival, and shortens every wait's limit to 2 ms.  The
call must return (no hang), the device status word must read MLA_ERR_TIMEOUT, and once
the hook is off and the workspace zeroed again the next call on the same context must
match the oracle.  No fault, trap or endless loop is involved: the failure is a missing
arrival, and every wait has a limit.
"""

import numpy as np
import pytest
import torch

from paged_head_latent_gb300 import workloads as wl
from tests.conftest import require_gpu
from tests.oracle_io import oracle_run

OUT_TOL = 2e-2
LSE_TOL = 1e-3


def test_inject_hook_rejects_bad_arguments(lib):
    # host-side checks only (no CUDA call)
    assert lib.lib().mla_debug_inject_timeout(0, 1000) == -2
    assert lib.lib().mla_debug_inject_timeout(-5, 1000) == -2
    assert lib.lib().mla_debug_inject_timeout(-1, 0) == 0


CASES = {
    "bf16": lambda: wl.make_decode([1000, 300], num_qo_heads=16, page_size=64, seed=4000),
    # FP8 caches have their own producer: raw bytes by TMA boxes (page 64) or cp.async
    # (page 16), converted a tile later, with its own give-up and drain path.
    "fp8_tma": lambda: wl.quantize_fp8(wl.make_decode([1000, 300], num_qo_heads=16, page_size=64, seed=4001)),
    "fp8_copy": lambda: wl.quantize_fp8(wl.make_decode([1000, 300], num_qo_heads=16, page_size=16, seed=4002)),
}


@pytest.mark.gpu
@pytest.mark.parametrize("case", sorted(CASES))
def test_bounded_wait_gives_up_and_reports_timeout(lib, case):
    require_gpu()
    w_cpu = CASES[case]()
    w = w_cpu.to("cuda")
    ws = torch.zeros(lib.workload_workspace_bytes(w, 1), dtype=torch.uint8, device="cuda")
    assert lib.lib().mla_debug_inject_timeout(2, 2_000_000) == 0
    try:
        lib.run_workload(w, workspace=ws, num_workers=1)
        status = lib.read_device_status(ws)
    finally:
        assert lib.lib().mla_debug_inject_timeout(-1, 0) == 0
    assert status == -7, lib.string_of(status)  # MLA_ERR_TIMEOUT
    # The context is still usable: the same call, hook off, matches the oracle.
    ws.zero_()
    out, lse = lib.run_workload(w, workspace=ws, num_workers=1)
    assert lib.read_device_status(ws) == 0
    ref_out, ref_lse = oracle_run(w_cpu)
    assert np.max(np.abs(out.float().cpu().numpy() - ref_out)) <= OUT_TOL
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) <= LSE_TOL
