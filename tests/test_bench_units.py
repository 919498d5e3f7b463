"""The bench's algorithmic work per call: the unit figures its roofline divides by.

Bytes: 1152 B of KV + 4 B of index per cached key of a request (a prefill request's
query rows share its keys, so each key counts once), plus 1152 B of q, 1024 B of out
and 4 B of lse per (query row, head).  Flops: 2 * (576 + 512) per (visible key, head),
a visible key being a (query row, key) pair that the bottom-right causal mask keeps.
"""
import importlib.util
import os

from paged_head_latent_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_decode_units():
    b = _bench()
    w = wl.make_decode([3, 64, 129], num_qo_heads=16, page_size=64, seed=3100)
    nbytes, flops, keys = b.algorithmic_work(w)
    assert keys == 3 + 64 + 129
    assert nbytes == keys * 1156 + 3 * 16 * (1152 + 1024 + 4)
    assert flops == keys * 16 * 2 * 1088


def test_prefill_counts_each_cached_key_once():
    b = _bench()
    # request 0: 4 query rows, no prefix (kv 4); request 1: 2 query rows after a prefix of 5 (kv 7)
    w = wl.make_prefill([4, 2], [0, 5], num_qo_heads=8, page_size=16, seed=3101)
    nbytes, flops, keys = b.algorithmic_work(w)
    visible = (1 + 2 + 3 + 4) + (6 + 7)  # causal, bottom-right aligned
    assert keys == visible
    assert nbytes == (4 + 7) * 1156 + 6 * 8 * (1152 + 1024 + 4)
    assert flops == visible * 8 * 2 * 1088
