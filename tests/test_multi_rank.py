"""The N > 1 path of bench.py on CPU: two gloo ranks shard tokens without a
collective on the forward's data path, agree on the max-over-ranks time,
and sum the backward's weight gradients over ranks (its one exchange)."""
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
    grads = {"grad_phi": torch.full((2, 3), float(r + 1)), "grad_alpha": torch.tensor([r, 1.0, 2.0]),
             "grad_bias": torch.ones(4) * (r + 1), "grad_gamma": None, "grad_x": torch.full((2,), float(r))}
    bench.allreduce_weight_grads(grads, w)
    dist.barrier()
    q.put((r, lo, hi, t, grads["grad_phi"].tolist(), grads["grad_alpha"].tolist(), grads["grad_bias"].tolist(),
           grads["grad_x"].tolist()))
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
    for r in res:
        assert r[4] == [[3.0] * 3] * 2 and r[5] == [1.0, 2.0, 4.0] and r[6] == [3.0] * 4   # summed
    assert res[0][7] == [0.0, 0.0] and res[1][7] == [1.0, 1.0]         # grad_x stays per rank


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.per_token_bytes(4, 7168) == 71776
    assert bench.launch_bytes(32768, 4, 7168) == 32768 * 71776 + 4 * 24 * 28672
