"""Multi-rank host logic on CPU (gloo, world size 2): every rank draws its
own batch of the same shape, the slowest rank's time is what every rank
reports, and the job throughput counts all ranks' tokens; and one batch
sharded by sequence across the ranks, each shard run through the oracle,
gathers back to exactly the single-rank result."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import numpy as np


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


def _shard_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    import workloads as wl
    # one global batch, the same on every rank (same seed); ragged lengths,
    # an empty sequence, initial states
    full = wl.prefill_inputs([37, 0, 64, 5, 130, 1, 90], 2, 16, 8, torch.float32, True, seed=5,
                             init_state=True)
    part, seqs = wl.shard_sequences(full, rank, world)
    f = lambda t: None if t is None else t.double().numpy()
    o, S = oracle.delta(f(part["q"]), f(part["k"]), f(part["v"]), f(part["beta_logits"]),
                        f(part["gate_logits"]), part["cu_seqlens"].numpy(), init_S=f(part["init_S"]))
    # exchange the shards' outputs (gloo all_gather of padded tensors)
    n_tok = torch.tensor([o.shape[0]])
    sizes = [torch.zeros(1, dtype=torch.long) for _ in range(world)]
    dist.all_gather(sizes, n_tok)
    cap = int(max(s_.item() for s_ in sizes))
    pad = torch.zeros((cap,) + o.shape[1:], dtype=torch.float64)
    pad[:o.shape[0]] = torch.from_numpy(o)
    outs = [torch.zeros_like(pad) for _ in range(world)]
    dist.all_gather(outs, pad)
    if rank == 0:
        shards = []
        for r in range(world):
            _, seqs_r = wl.shard_sequences(full, r, world)
            shards.append((outs[r][:int(sizes[r].item())], seqs_r))
        got = wl.gather_sequences(shards, full["cu_seqlens"])
        ref, _ = oracle.delta(f(full["q"]), f(full["k"]), f(full["v"]), f(full["beta_logits"]),
                              f(full["gate_logits"]), full["cu_seqlens"].numpy(), init_S=f(full["init_S"]))
        out["equal"] = bool(np.array_equal(got.numpy(), ref))
        out["seqs"] = [wl.shard_sequences(full, r, world)[1] for r in range(world)]
    dist.barrier()
    dist.destroy_process_group()


def test_one_batch_sharded_by_sequence():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_shard_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out["seqs"] == [[0, 2, 4, 6], [1, 3, 5]]
    assert out["equal"]
