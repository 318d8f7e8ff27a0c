"""The N > 1 path of bench.py on CPU: two gloo ranks take their shards of one
global batch through the same calls bench.py makes (rank_shard, shard_tokens),
with no collective on the forward's data path, agree on the max-over-ranks
time, and sum the backward's weight gradients over ranks (its one exchange)."""
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
    # the inputs bench.py gives this rank: its shard of one global batch
    from mhc_synth import make_case, make_post_case
    part = bench.rank_shard(lambda **k: make_case("tiny", device="cpu", pre_mix=True, **k), 40, w, r)
    xs = [torch.empty_like(part.x.float()) for _ in range(w)]
    dist.all_gather(xs, part.x.float().contiguous())          # bf16 values, exact in fp32
    pms = [torch.empty_like(part.pre_mix) for _ in range(w)]
    dist.all_gather(pms, part.pre_mix.contiguous())
    post = bench.rank_shard(lambda **k: make_post_case(device="cpu", **k), 24, w, r)
    shard_info = (part.T, tuple(part.x.shape), torch.cat(xs).numpy().tobytes(), torch.cat(pms).numpy().tobytes(),
                  post.T, tuple(post.residual.shape))
    t = bench.max_over_ranks(1.0 + r, w)
    grads = {"grad_phi": torch.full((2, 3), float(r + 1)), "grad_alpha": torch.tensor([r, 1.0, 2.0]),
             "grad_bias": torch.ones(4) * (r + 1), "grad_gamma": None, "grad_x": torch.full((2,), float(r))}
    bench.allreduce_weight_grads(grads, w)
    dist.barrier()
    q.put((r, lo, hi, t, grads["grad_phi"].tolist(), grads["grad_alpha"].tolist(), grads["grad_bias"].tolist(),
           grads["grad_x"].tolist(), shard_info))
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
    # each rank held its own 40 tokens, and together they are the global batch
    # of 80 tokens drawn from one seed, in rank order
    from mhc_synth import make_case
    full = make_case("tiny", device="cpu", T=80, seed=0, pre_mix=True)
    for r in res:
        T_r, shape, xs, pms, post_T, post_shape = r[8]
        assert T_r == 40 and shape == (40, 4, 256) and post_T == 24 and post_shape == (24, 4, 256)
        assert xs == full.x.float().numpy().tobytes()
        assert pms == full.pre_mix.numpy().tobytes()


def test_take_tokens_cuts_only_per_token_tensors():
    from mhc_synth import make_bwd_grads, make_case
    c = make_case("tiny", device="cpu", T=10, gamma=True, pre_mix=True)
    p = bench.take_tokens(c, 3, 7)
    assert p.T == 4 and torch.equal(p.x, c.x[3:7]) and torch.equal(p.pre_mix, c.pre_mix[3:7])
    assert p.phi is c.phi and p.gamma is c.gamma and p.bias is c.bias
    g = make_bwd_grads(device="cpu", T=10, grad_x_post=True)
    q = bench.take_tokens(g, 2, 5)
    assert torch.equal(q.g_in, g.g_in[2:5]) and torch.equal(q.g_res, g.g_res[2:5])
    assert torch.equal(q.g_x_post, g.g_x_post[2:5])
    assert bench.rank_shard(lambda **k: make_case("tiny", device="cpu", **k), 16, 1, 0).T == 16


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.per_token_bytes(4, 7168) == 71776
    assert bench.launch_bytes(32768, 4, 7168) == 32768 * 71776 + 4 * 24 * 28672


def test_algorithmic_bytes_of_every_workload():
    """The per-token byte counts the roofline divides by, for each workload:
    x in, y out, the gate outputs (comb only with three gates), pre_mix in,
    and the backward outputs (invRms, hMix, every Sinkhorn step's sums and
    matrices) when asked for."""
    assert bench.per_token_bytes(4, 256) == 2 * 4 * 256 + 2 * 256 + 4 * 24            # tiny: 2,656
    assert bench.per_token_bytes(4, 256) == 2656
    assert bench.per_token_bytes(4, 4096, need_backward=True) == 41056 + 3300         # training
    assert bench.per_token_bytes(4, 7168) == 71776                                     # decode, prefill
    assert bench.per_token_bytes(8, 2048, pre_mix=True) == 37216                       # generic A
    assert bench.per_token_bytes(8, 2048, alpha_len=2) == 36928                        # generic B
    # two gates with the backward outputs: invRms and the 2n mixes, no Sinkhorn steps
    assert bench.per_token_bytes(4, 64, need_backward=True, alpha_len=2) == 2 * 256 + 128 + 32 + 4 + 32
    # the backward and its contraction kernel; the post-mapping
    assert bench.bwd_token_bytes(4, 7168) == 132436
    assert bench.bwd_main_token_bytes(4, 7168) == 129024
    # x read (2D), residual read and out written (2nD each), post (4n) and comb (4n^2) read
    assert bench.post_token_bytes(4, 7168) == 2 * 7168 + 2 * (2 * 4 * 7168) + 4 * 4 + 4 * 16 == 129104
