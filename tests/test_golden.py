"""Regression fixtures of the oracle (written by tests/golden/make_golden.py from oracle/ only).

They also pin the seeded generator: the same seed must give the same draws on
every machine that runs the GPU tests, or CPU and GPU runs would not compare
the same inputs.
"""

import json
import os

import numpy as np
import pytest

from paged_head_latent_gb300 import workloads as wl
from tests.oracle_io import oracle_run

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("name,make", [
    ("decode_b4_h16_ps64", wl.decode_b4_h16_ps64),
    ("prefill_small_q5_3_prefix2_64",
     lambda: wl.make_prefill([5, 3], [2, 64], num_qo_heads=2, page_size=64, seed=1099,
                             name="prefill_small_q5_3_prefix2_64")),
])
def test_oracle_matches_fixture(name, make):
    with open(os.path.join(HERE, name + ".json")) as f:
        g = json.load(f)
    out, lse = oracle_run(make())
    want_lse = np.array([[float(x) for x in row] for row in g["lse"]])
    want_out = np.array([[[float(x) for x in h] for h in r] for r in g["out"]])
    np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out[:, :, g["out_cols"]], want_out, rtol=0, atol=1e-12)
