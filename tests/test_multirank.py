"""Host logic of the multi-GPU bench path on CPU: two gloo ranks. Each rank
draws its own batch (different seeds, same shapes) and the reported step time
is the maximum over ranks; nothing is exchanged on the data path."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from mixture_experts_layer_99_b300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = W.small(W.WORKLOADS["switch_top1"], T=16, d=8, H=8)
    local = 1.0 + rank * 0.5
    got = bench.max_over_ranks(local, dist, torch.device("cpu"))
    x = W.make_inputs(w, seed=bench.rank_seed(w, rank, 0))["x"]
    gathered = [torch.empty_like(x) for _ in range(world)]
    dist.all_gather(gathered, x)
    dist.barrier()
    q.put((rank, got, [torch.equal(gathered[0], g) for g in gathered]))
    dist.destroy_process_group()


def test_two_rank_timing_and_seeds():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, same in res:
        assert got == 1.5                       # max over ranks
        assert same == [True, False]            # rank 1 drew a different batch


def test_single_process_max_is_identity():
    assert bench.max_over_ranks(3.25, None, torch.device("cpu")) == 3.25
