"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): each rank gets its own batch
of requests, the timing barrier works, and the reported time is the maximum over ranks."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r) == (world, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(dist)
    t = bench.max_over_ranks(dist, 1.5 + rank, torch.device("cpu"))
    from synth import workloads
    w = workloads.config1(seed=bench.rank_seed(0, rank), steps=1)
    first = next(iter(w.iter_steps(1))).topk
    out[rank] = (t, first.sum().item(), bench.rank_seed(7, rank))
    dist.destroy_process_group()


def test_two_ranks_weak_scaling_host_logic():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    (t0, s0, seed0), (t1, s1, seed1) = out[0], out[1]
    assert t0 == t1 == 2.5                 # max over ranks
    assert seed0 != seed1 and s0 != s1      # independent batches per rank
