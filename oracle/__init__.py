"""Float64 CPU oracle for paged MLA (test infrastructure only).

Only tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  It shares no code with the CUDA path.
"""

from .mla_oracle import (attend, combine_partials, mla_decode, mla_decode_split, mla_prefill,
                         mla_sparse_decode, online_softmax_partial, scores, visible_len)
from .brute import brute_decode, brute_prefill

__all__ = ["attend", "combine_partials", "mla_decode", "mla_decode_split", "mla_prefill", "mla_sparse_decode",
           "online_softmax_partial", "scores", "visible_len", "brute_decode", "brute_prefill"]
