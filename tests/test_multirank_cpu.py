"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): every rank
draws its own batch of the same shape, the slowest rank's time is what every
rank reports, and the job throughput counts all ranks' tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workloads as wl
    my_ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
    slowest = bench.max_over_ranks(my_ms, dist, torch.device("cpu"))
    inp = wl.prefill_inputs([16, 8], 2, 8, 8, torch.float32, True, seed=bench.rank_seed(rank))
    out[rank] = (slowest, bench.job_throughput(1000, world, slowest),
                 tuple(inp["q"].shape), float(inp["q"].sum()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 15.0
    assert out[0][1] == pytest.approx(1000 * 2 / 0.015)
    assert out[0][2] == out[1][2]          # same shapes
    assert out[0][3] != out[1][3]          # independent draws
