"""Float64 CPU oracle for paged MLA (test infrastructure only).

Only tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  It shares no code with the CUDA path.
"""

from .mla_oracle import (attend, block_table_to_csr, combine_partials, dequantize_fp8_cache, e4m3_to_float,
                         mla_decode, mla_decode_block_table, mla_decode_fp8, mla_sparse_decode_fp8,
                         mla_decode_split, mla_prefill, mla_sparse_decode, online_softmax_partial, scores,
                         visible_len)
from .brute import brute_decode, brute_prefill

__all__ = ["attend", "block_table_to_csr", "dequantize_fp8_cache", "e4m3_to_float", "mla_decode_fp8",
           "mla_sparse_decode_fp8", "mla_decode_block_table", "combine_partials", "mla_decode", "mla_decode_split", "mla_prefill", "mla_sparse_decode",
           "online_softmax_partial", "scores", "visible_len", "brute_decode", "brute_prefill"]
