"""Write the oracle's regression fixtures.  Calls only oracle/ and the seeded input generator.

The pages print no worked numeric example for paged MLA (flashinfer-bench
"MLA Paged" lists shapes only), so these fixtures are not the pages' numbers:
they freeze the oracle's float64 result on the small seeded decode workload
(batch 4, 16 heads, page 64, kv lens {1, 63, 64, 200}) and on a small causal
prefill, so that any later change to the oracle or to the generator's draws
shows up.  Run:  python tests/golden/make_golden.py
"""

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from paged_head_latent_gb300 import workloads as wl  # noqa: E402
from tests.oracle_io import oracle_run  # noqa: E402

COLS = [0, 1, 255, 256, 511]


def fixture(w):
    out, lse = oracle_run(w)
    return {
        "workload": w.name,
        "lse": [[repr(float(x)) for x in row] for row in lse],
        "out_cols": COLS,
        "out": [[[repr(float(out[r, h, c])) for c in COLS] for h in range(out.shape[1])]
                for r in range(out.shape[0])],
    }


def main():
    items = [wl.decode_b4_h16_ps64(),
             wl.make_prefill([5, 3], [2, 64], num_qo_heads=2, page_size=64, seed=1099,
                             name="prefill_small_q5_3_prefix2_64")]
    for w in items:
        with open(os.path.join(HERE, w.name + ".json"), "w") as f:
            json.dump(fixture(w), f, indent=0)
            f.write("\n")


if __name__ == "__main__":
    main()
