"""The N > 1 path of bench.py on CPU: world-size-2 gloo ranks (no GPU).

Ranks are replicas with their own sequences; only the timing crosses ranks: the
whole-job value is the tokens of every rank over the slowest rank's time."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        times = [10.0 + 5.0 * rank, 7.0 - rank]          # rank 1 is slower in the first entry
        out[rank] = (bench.max_over_ranks(times), bench.rank_seed(3, rank))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timing_and_keep_distinct_sequences():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == [15.0, 7.0]
    assert res[0][1] != res[1][1]


def test_single_rank_and_whole_job_value():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.0, 2.0]) == [1.0, 2.0]
    # 2 ranks x batch 8 x 64 steps over the slowest rank's 400 ms
    assert bench.whole_job_tokens_per_s(8, 64, 2, 400.0) == pytest.approx(2560.0)
