"""The multi-GPU path is replicas only: every rank runs its own forward on
its own inputs, with no collective on the data path; bench.py times each
replica, takes the slowest rank's time and counts every rank's tokens.
This checks that host logic with two gloo ranks on the CPU (no GPU)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, got_local = bench.dist_env()
        # each replica's own step time; the job's is the slowest one
        mine = 1.5 + rank
        slowest = bench.max_over_ranks(mine, got_ws, torch.device("cpu"))
        # each replica draws its own inputs (seeded by rank)
        from state_space_sequence_cumsum_gb300.inputs import Shape, make_inputs
        x = make_inputs(Shape(1, 8, 2, 4, 4, 1, 4), seed=got_rank)["x"].float()
        xs = [torch.zeros_like(x) for _ in range(ws)]
        dist.all_gather(xs, x)
        distinct = not torch.equal(xs[0], xs[1])
        out[rank] = (got_ws, got_rank, got_local, slowest,
                     bench.job_throughput(got_ws, 1000.0, slowest), distinct)
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_rank_and_count_every_rank():
    ws = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(ws, port, out), nprocs=ws, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank, (got_ws, got_rank, got_local, slowest, thr, distinct) in res.items():
        assert (got_ws, got_rank, got_local) == (2, rank, rank)
        assert slowest == pytest.approx(2.5)          # rank 1's 2.5 ms, seen by both ranks
        assert thr == pytest.approx(2 * 1000.0 / 2.5e-3)
        assert distinct                                # replicas work on different inputs


def test_one_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25
    assert bench.job_throughput(1, 500.0, 2.0) == pytest.approx(250000.0)
