"""The N > 1 path of bench.py on CPU: two gloo ranks shard tokens without a
collective on the data path and agree on the max-over-ranks time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, l = bench.dist_env()
    lo, hi = bench.shard_tokens(1000, w, r)
    t = bench.max_over_ranks(1.0 + r, w)
    dist.barrier()
    q.put((r, lo, hi, t))
    dist.destroy_process_group()


def test_two_rank_sharding_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][1:3] == (0, 1000) and res[1][1:3] == (1000, 2000)   # disjoint token ranges
    assert res[0][3] == res[1][3] == 2.0                               # slowest rank's time


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.per_token_bytes(4, 7168) == 71776
    assert bench.launch_bytes(32768, 4, 7168) == 32768 * 71776 + 4 * 24 * 28672
