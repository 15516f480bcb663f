"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

Each rank runs an independent replica of the workload (weak scaling, no
data-path collective); the only cross-rank steps are the timing reductions:
the slowest rank's time and the sum of the bytes processed.
"""

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


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    times = [1.0 + rank, 10.0 - rank, 5.0 * (rank + 1)]
    red, total = bench.reduce_over_ranks(times, 1000 * (rank + 1), "cpu")
    spec = bench.workload_spec("longctx_8x2_B2_L4096", seed_offset=100 * rank)
    results[rank] = (red, total, spec.seed, spec.kv_bytes(), spec.ctx_lens)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_reduction_and_replica_specs():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
    r0, r1 = results[0], results[1]
    assert r0[0] == r1[0] == [2.0, 10.0, 10.0]          # max over ranks
    assert r0[1] == r1[1] == 3000.0                     # sum of bytes
    assert r0[2] != r1[2]                               # own seed per replica
    assert r0[3] == r1[3] and r0[4] == r1[4]            # same shapes: weak scaling


def test_single_rank_reduction_is_identity():
    import bench

    assert not dist.is_initialized()
    red, total = bench.reduce_over_ranks([3.0, 4.0], 77, "cpu")
    assert red == [3.0, 4.0] and total == 77.0
