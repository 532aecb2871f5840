"""Host logic of the data-parallel (weak-scaling) bench path, world size 2 on gloo.

Every GPU run here has one GPU, so the N > 1 path is covered on the CPU: each rank
draws its own shard of the global batch (rank 0 = the single-GPU workload, the
others distinct), and the step time reported is the maximum over ranks.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workload


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, _ = bench.dist_env()
    cfg = workload.shard(workload.CONFIGS["decode"], r)
    inst = workload.draw(cfg)
    lens = torch.from_numpy(inst.prefix.astype(np.int64))
    gathered = [torch.zeros_like(lens) for _ in range(ws)]
    dist.all_gather(gathered, lens)
    slowest = bench.max_over_ranks(10.0 + r, ws, device="cpu")
    bench.barrier(ws)
    out[r] = (ws, [g.tolist() for g in gathered], slowest)
    dist.destroy_process_group()


def test_two_ranks_draw_disjoint_shards_and_report_the_slowest():
    mgr = mp.get_context("spawn").Manager()  # no fork of a multi-threaded process
    out = mgr.dict()
    mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
    single = workload.draw(workload.CONFIGS["decode"]).prefix.tolist()
    for r in (0, 1):
        ws, gathered, slowest = out[r]
        assert ws == 2
        assert gathered[0] == single            # rank 0 is the single-GPU workload
        assert gathered[1] != gathered[0]        # rank 1 draws its own sequences
        assert slowest == 11.0                   # max over ranks
