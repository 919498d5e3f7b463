"""Seeded random cases on the GPU against the float64 oracle.

Each case draws its kind (decode, causal prefill, packed multi-token decode, sparse top-k
decode, FP8-cache decode), batch, head count, page size, key lengths and split-KV worker
count from one seed, so the grid of hand-picked parity cases is crossed with shapes
nobody chose: odd head counts, page sizes that are neither 1 nor a multiple of 64,
empty and one-key requests, lengths on and next to 64-key tile boundaries, and worker
counts from one to more than there are SMs.  Every element of out and lse is compared,
and the device status word must stay clear.
"""

import numpy as np
import pytest
import torch

from paged_head_latent_gb300 import workloads as wl
from tests.conftest import require_gpu
from tests.oracle_io import oracle_run

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2
LSE_TOL = 1e-3

HEADS = [1, 3, 7, 16, 33, 64, 100, 128]
PAGE_SIZES = [1, 2, 16, 32, 64, 128]
WORKERS = [0, 1, 2, 3, 11, 76, 150]


def _lengths(rng, n, hi):
    """Key lengths: mostly uniform, with empty, single-key and tile-boundary values mixed in."""
    special = [0, 1, 63, 64, 65, 127, 128, 129]
    out = []
    for _ in range(n):
        r = rng.random()
        out.append(int(rng.choice(special)) if r < 0.35 else int(rng.integers(1, hi + 1)))
    return out


def _case(seed):
    rng = np.random.default_rng(9000 + seed)
    kind = ["decode", "decode", "prefill", "mtp", "sparse", "fp8"][seed % 6]
    heads = int(rng.choice(HEADS))
    ps = int(rng.choice(PAGE_SIZES))
    workers = int(rng.choice(WORKERS))
    if kind == "decode":
        w = wl.make_decode(_lengths(rng, int(rng.integers(1, 10)), 1500), heads, ps, seed=seed,
                           token_shuffle=bool(rng.integers(0, 2)))
    elif kind == "fp8":
        w = wl.quantize_fp8(wl.make_decode(_lengths(rng, int(rng.integers(1, 8)), 1200), heads, ps, seed=seed))
    elif kind == "prefill":
        n = int(rng.integers(1, 4))
        q_lens = [int(x) for x in rng.integers(1, 90, size=n)]
        prefixes = [int(rng.choice([0, 1, 63, 64, int(rng.integers(0, 300))])) for _ in range(n)]
        w = wl.make_prefill(q_lens, prefixes, num_qo_heads=heads, page_size=ps, seed=seed)
    elif kind == "mtp":
        q_len = int(rng.integers(2, 5))
        heads = min(heads, 128 // q_len)
        lens = [max(q_len, x) for x in _lengths(rng, int(rng.integers(1, 8)), 1200)]
        w = wl.make_mtp(lens, q_len, heads, ps, seed=seed)
    else:  # sparse
        topk = int(rng.choice([1, 37, 64, 130, 256]))
        w = wl.make_sparse_decode(_lengths(rng, int(rng.integers(1, 7)), 900), topk, heads, ps, seed=seed)
    return w, workers


@pytest.mark.parametrize("seed", range(120))
def test_random_case(lib, seed):
    require_gpu()
    w, workers = _case(seed)
    what = f"seed {seed}: {w.kind} heads {w.num_qo_heads} page {w.page_size} workers {workers}"
    wd = w.to("cuda")
    ws = torch.zeros(lib.workload_workspace_bytes(wd, workers), dtype=torch.uint8, device="cuda")
    out, lse = lib.run_workload(wd, workspace=ws, num_workers=workers)
    torch.cuda.synchronize()
    assert lib.read_device_status(ws) == 0, what
    ref_out, ref_lse = oracle_run(w)
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    assert o.shape == ref_out.shape and l.shape == ref_lse.shape, what
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(l), fin), what
    assert np.all(np.isneginf(l[~fin])), what
    if o.size:
        assert np.max(np.abs(o - ref_out)) <= OUT_TOL, what
    if fin.any():
        assert np.max(np.abs(l[fin] - ref_lse[fin])) <= LSE_TOL, what
