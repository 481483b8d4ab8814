"""Host logic of the multi-GPU benchmark on CPU: two gloo ranks.

Every rank verifies its own batch (weak scaling); the only collectives are the
barrier and the max over ranks of the timings.  Checked here without a GPU:
the per-rank seeds differ, the inputs of a rank are reproducible, and the
max-over-ranks reduction gives every rank the slowest rank's time.
"""
import os
import socket

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(10.0 + rank, dist, torch.device("cpu"))
    seed = bench.rank_seed(bench.workloads.CONFIGS["tiny"], rank)
    out[rank] = (t, seed)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_reduction_and_seeds():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 11.0          # slowest rank's time on both ranks
    assert out[0][1] != out[1][1]                  # each rank draws its own batch
