"""Host logic of the N > 1 bench path, on CPU with gloo (no GPU).

The decode path has no data exchange between GPUs (requests are independent), so
`bench.py --gpus N` runs N independent replicas; the only cross-rank steps are the
barrier and the max over ranks of the step time, checked here with two gloo ranks.
"""
import argparse
import contextlib
import io
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.distributed.barrier()
        results[rank] = bench.max_over_ranks(1.5 + rank, world, "cpu")
    finally:
        torch.distributed.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        assert dict(results) == {0: 2.5, 1: 2.5}


def test_max_over_ranks_single_rank_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_other_ranks_do_no_work():
    args = argparse.Namespace(workload="decode_b4_h16_ps64", steps=1, warmup=0)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.reference_arm(args, rank=1, world=2)
    assert buf.getvalue() == ""
