#!/usr/bin/env python3
"""Benchmark of the mHC pre-mapping forward on GB300 (one JSON line on stdout).

Workload: the prefill shape the metric is quoted on -- T = 32768 tokens
(b = 4, s = 8192), n = 4 streams, D = 7168, phi [24, 28672] fp32, alpha[3],
bias[24], no gamma, 20 Sinkhorn iterations, fp32 projection mode.  A step is
one whole forward (plane preparation + fused kernel) over that batch; inputs
(2.35 GB of algorithmic traffic) are larger than L2, so no flush is needed
between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torch.distributed.run, one rank per GPU: every rank processes
its own batch of T tokens (tokens are independent, so the work shards with no
collective on the data path; "weak" scaling); the barrier and max-over-ranks
timing use the process group only for the clock.

--impl reference times the CPU oracle (the only other implementation of the
operator here) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s and achieved HBM GB/s (% of roofline), mHC pre fwd n=4 D=7168 20 iters"
WORKLOAD = dict(name="prefill", T=32768, n=4, D=7168, impl_mode=0, num_iters=20)


def per_token_bytes(n, D, need_backward=False, pre_mix=False, alpha_len=3, iters=20):
    """Algorithmic bytes per token: x in, y out, hPost + hPre out, and comb
    with three gates (the two-gate form's optional comb is all zeros and not
    counted)."""
    R = n * n + 2 * n if alpha_len == 3 else 2 * n
    b = 2 * n * D + 2 * D + 4 * (2 * n) + (4 * n * n if alpha_len == 3 else 0)
    if pre_mix:
        b += 4 * n
    if need_backward:
        b += 4 + 4 * R + (2 * iters * 4 * (n + n * n) if alpha_len == 3 else 0)
    return b


def launch_bytes(T, n, D, alpha_len=3):
    R = n * n + 2 * n if alpha_len == 3 else 2 * n
    return T * per_token_bytes(n, D) + 4 * R * n * D      # phi once per launch


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def shard_tokens(T_per_rank: int, world: int, rank: int):
    """Token range of one rank in the global batch (weak scaling: each rank
    owns its own T_per_rank tokens)."""
    return rank * T_per_rank, (rank + 1) * T_per_rank


# Per-token fields of the input records (cut along their first dimension).
TOKEN_FIELDS = ("x", "pre_mix", "residual", "post", "comb", "g_in", "g_post", "g_res", "g_x_post")


def take_tokens(rec, lo: int, hi: int):
    """Tokens [lo, hi) of an input record (a dataclass of tensors): its
    per-token tensors cut, everything else (weights) kept."""
    import dataclasses
    changes = {}
    for f in dataclasses.fields(rec):
        v = getattr(rec, f.name)
        if f.name == "T":
            changes["T"] = hi - lo
        elif f.name in TOKEN_FIELDS and v is not None:
            changes[f.name] = v[lo:hi].clone()
    return dataclasses.replace(rec, **changes)


def rank_shard(make, T_per_rank: int, world: int, rank: int):
    """This rank's part of one global batch: `make(T=world * T_per_rank,
    seed=0)` draws the whole batch from one seed, and the rank keeps the
    tokens shard_tokens gives it."""
    full = make(T=world * T_per_rank, seed=0)
    if world == 1:
        return full
    lo, hi = shard_tokens(T_per_rank, world, rank)
    part = take_tokens(full, lo, hi)
    del full
    return part


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = [l for (t, l) in self.lines if self.t0 and self.t1 and self.t0 <= t <= self.t1]
        if not rows:  # timed region shorter than the sampling period: use the nearest samples
            rows = [l for (_, l) in self.lines[-3:]]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- peaks

def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


KERNEL_SOURCES = {"mhc_pre_tc_kernel": "mhc_pre_tc.cu", "mhc_pre_tc_kernel_resident": "mhc_pre_tc.cu",
                  "mhc_pre_gw_kernel": "mhc_pre_gw.cu", "bw_main_kernel": "mhc_bwd.cu"}


def _code_only(text):
    """Source text without // comments, trailing blanks and blank lines, so
    that editing a comment leaves the hash of the code alone."""
    out = []
    for line in text.splitlines():
        i = line.find("//")
        if i >= 0:
            line = line[:i]
        line = line.rstrip()
        if line:
            out.append(line)
    return "\n".join(out)


def kernel_hash(kernel):
    """Hash of a fused kernel's device code (its traffic record is void once
    the code changes; comments do not count)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "mhc_hyper_connection_gb300", "csrc")
    for name in ("mhc_common.cuh", "mhc_ptx.cuh", KERNEL_SOURCES[kernel]):
        with open(os.path.join(d, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, T):
    """DRAM bytes per launch of the fused kernel from the committed ncu summary,
    scaled to T tokens; None once the kernel source changed since capture."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_hash") != kernel_hash(kernel):
        return None
    return rec["dram_bytes_per_token"] * T + rec.get("dram_bytes_fixed", 0)


# ----------------------------------------------------------------- CPU oracle

def oracle_rate(case, budget_s: float, max_tokens: int):
    """Tokens/s of the oracle, on all host cores, over passes of up to
    max_tokens of the workload's tokens until about budget_s has elapsed."""
    import numpy as np
    import torch
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    phi, alpha, bias = case.phi.cpu().numpy(), case.alpha.cpu().numpy(), case.bias.cpu().numpy()
    count = max(1, min(max_tokens, case.T))
    x = case.x[:count].view(torch.int16).cpu().numpy().view(np.uint16)
    done, t_total, passes = 0, 0.0, 0
    while passes == 0 or t_total < budget_s:
        t0 = time.perf_counter()
        oracle.run(x, phi, alpha, bias, num_iters=case.num_iters, backward=False, threads=threads,
                   x_fp16=case.x.dtype == torch.float16)
        t_total += time.perf_counter() - t0
        done += count
        passes += 1
    return done / t_total, threads, f"{passes} pass(es) over {count} tokens", t_total


# ----------------------------------------------------------------- post-mapping

POST_METRIC = "tokens/s and achieved HBM GB/s (% of roofline), mHC post (hc_post) n=4 D=7168"


def post_token_bytes(n, D):
    """x + residual read, out written (bf16), post + comb read (fp32)."""
    return 2 * D + 2 * n * D + 2 * n * D + 4 * n + 4 * n * n


def bench_post(args, device, world, rank, local):
    """hc_post at the prefill shape: device-timed steps, the roofline of its
    one kernel, and the oracle on host cores for a bounded sample."""
    import torch
    from mhc_synth import make_post_case
    T, n, D = args.tokens, WORKLOAD["n"], WORKLOAD["D"]
    cfg = {"workload": f"hc_post T={T} n={n} D={D} (b=4, s=8192)", "tokens_per_rank": T, "n": n, "D": D,
           "l2": "inputs exceed L2; no flush needed", "parallelism": f"token-sharded x{world} (no collective)"}
    case = rank_shard(lambda **k: make_post_case(device=device, n=n, D=D, **k), T, world, rank)
    if args.impl == "reference":
        if rank != 0:
            return 0
        rate, threads, sample, dt = post_oracle_rate(case, 60.0 * args.steps / (args.steps + args.warmup))
        print(json.dumps({"impl": "reference", "metric": POST_METRIC, "value": rate, "unit": "tokens/s",
                          "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": 1e3 * T / rate, "higher_is_better": True, "scaling": "weak",
                          "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
                          "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                           "sample": sample},
                          "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}))
        return 0
    from mhc_hyper_connection_gb300 import build as mbuild, hc_post
    mbuild.build()
    stream = torch.cuda.current_stream(device)
    out = torch.empty((T, n, D), dtype=torch.bfloat16, device=device)

    def step():
        hc_post(case.x, case.residual, case.post, case.comb, out=out, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    K = args.steps
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    clocks.mark(True)
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark(False)
    time.sleep(0.2)
    clocks.stop()
    elapsed = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, device)
    per_step = elapsed / K
    lb = T * post_token_bytes(n, D)
    peak, peak_src = hbm_peak()
    achieved = lb / per_step / 1e9
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, threads, sample, dt = post_oracle_rate(case, 10.0)
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps({
            "metric": POST_METRIC, "value": world * T * K / elapsed, "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": None, "kernel": "mhc_post_kernel", "kernel_ms": per_step * 1e3,
                         "algorithmic_bytes": lb, "peak_source": f"hbm_gbs of {peak_src}"},
            "cpu_baseline": cpu, "gpu_launches": K * world, "clocks": clocks.summary()}))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def post_oracle_rate(case, budget_s: float):
    """Tokens/s of the post-mapping oracle on all host cores, over passes of a
    bounded token sample, until about budget_s has elapsed."""
    import numpy as np
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    count = max(1, min(case.T, 2048))
    xb = case.x[:count].contiguous().view(torch_int16()).cpu().numpy().view(np.uint16)
    rb = case.residual[:count].contiguous().view(torch_int16()).cpu().numpy().view(np.uint16)
    post = case.post[:count].cpu().numpy()
    comb = case.comb[:count].cpu().numpy()
    done, t_total, passes = 0, 0.0, 0
    while passes == 0 or t_total < budget_s:
        t0 = time.perf_counter()
        oracle.run_post(xb, rb, post, comb, threads=threads)
        t_total += time.perf_counter() - t0
        done += count
        passes += 1
    return done / t_total, threads, f"{passes} pass(es) over {count} tokens of the hc_post workload ({t_total:.1f} s, double precision)", t_total


# ----------------------------------------------------------------- backward

BWD_METRIC = "tokens/s and achieved HBM GB/s (% of roofline), mHC pre backward (Sinkhorn form) n=4 D=7168"


def bwd_token_bytes(n, D, iters=20, grad_x_post=False):
    """Per token: x, grad_h_in, grad_h_post, grad_h_res, invRms, hMix, hPre,
    hPost, sumOut, normOut read, grad_x written (+ grad_x_post read)."""
    R = n * n + 2 * n
    b = 2 * n * D + 2 * D + 4 * n + 4 * n * n + 4 + 4 * R + 4 * n + 4 * n
    b += 2 * iters * 4 * (n + n * n) + 2 * n * D
    return b + (2 * n * D if grad_x_post else 0)


def bwd_main_token_bytes(n, D):
    """The contraction kernel's share: x and grad_h_in read, grad_x written."""
    return 2 * n * D + 2 * D + 2 * n * D


def bwd_inputs(device, T, n, D, world, rank, mode):
    """Forward inputs, the forward's saved intermediates (made by the library's
    own forward: these are benchmark inputs, not parity references) and
    upstream gradients, for this rank's shard of the global batch."""
    import torch
    from mhc_hyper_connection_gb300 import MhcPre
    from mhc_synth import make_bwd_grads, make_case
    case = rank_shard(lambda **k: make_case("prefill", device=device, impl_mode=mode, need_backward=True, **k),
                      T, world, rank)
    fwd = MhcPre(n, D, alpha_len=3, num_iters=20, impl_mode=mode, need_backward=True)
    out = fwd.allocate(T, device)
    fwd.run(case.x, case.phi, case.alpha, case.bias, out)
    torch.cuda.synchronize()
    if fwd.status(out) != 0:
        raise RuntimeError("device-side error in the forward that makes the saved intermediates")
    saved = {k: out[k] for k in ("inv_rms", "h_mix", "h_pre", "h_post", "sum_out", "norm_out")}
    g = rank_shard(lambda **k: make_bwd_grads(device=device, n=n, D=D, **k), T, world, rank)
    return case, saved, g


def allreduce_weight_grads(grads, world: int):
    """Data-parallel backward: the weight gradients (grad_phi, grad_alpha,
    grad_bias and grad_gamma when present) are sums over every rank's tokens,
    the one exchange step of the sharded backward; grad_x stays per rank."""
    if world <= 1:
        return
    import torch.distributed as dist
    for k in ("grad_phi", "grad_alpha", "grad_bias", "grad_gamma"):
        t = grads.get(k)
        if t is not None:
            dist.all_reduce(t, op=dist.ReduceOp.SUM)


def bwd_reference_inputs(device, T, n, D, mode, max_tokens):
    """Inputs of the reference arm: the first max_tokens tokens of the same
    workload, their saved intermediates from the oracle's forward (fp32, as
    the forward hands them on); no kernel of the library runs."""
    import types
    import numpy as np
    import torch
    import oracle
    from mhc_synth import make_bwd_grads, make_case
    case = make_case("prefill", device=device, T=T, impl_mode=mode, seed=0, need_backward=True)
    Ts = min(T, max_tokens)
    x = case.x[:Ts].contiguous()
    fw = oracle.run(x.view(torch_int16()).cpu().numpy().view(np.uint16), case.phi.cpu().numpy(),
                    case.alpha.cpu().numpy(), case.bias.cpu().numpy(), num_iters=case.num_iters, backward=True,
                    threads=os.cpu_count() or 1)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    saved = {"inv_rms": f32(fw.inv_rms), "h_mix": f32(fw.h_mix), "h_pre": f32(fw.h_pre),
             "h_post": f32(fw.h_post), "sum_out": f32(fw.sum_out), "norm_out": f32(fw.norm_out)}
    g = make_bwd_grads(seed=0, device=device, T=T, n=n, D=D)
    sub = types.SimpleNamespace(x=x, phi=case.phi, alpha=case.alpha, T=Ts, num_iters=case.num_iters)
    gs = types.SimpleNamespace(g_in=g.g_in[:Ts].contiguous(), g_post=g.g_post[:Ts], g_res=g.g_res[:Ts])
    return sub, saved, gs


def bwd_oracle_rate(case, saved, g, budget_s: float, max_tokens: int):
    """Tokens/s of the backward oracle on all host cores over passes of a
    bounded token sample (all five gradients of that sample)."""
    import numpy as np
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    count = max(1, min(case.T, max_tokens))
    bits = lambda t: t[:count].contiguous().view(torch_int16()).cpu().numpy().view(np.uint16)
    sv = {k: v[:count].cpu().numpy() if k not in ("sum_out", "norm_out") else v[:, :count].contiguous().cpu().numpy()
          for k, v in saved.items()}
    args = (bits(case.x), case.phi.cpu().numpy(), case.alpha.cpu().numpy(), None, bits(g.g_in),
            g.g_post[:count].cpu().numpy(), g.g_res[:count].cpu().numpy(), sv["inv_rms"], sv["h_mix"],
            sv["h_pre"], sv["h_post"], sv["sum_out"], sv["norm_out"])
    done, t_total, passes = 0, 0.0, 0
    while passes == 0 or t_total < budget_s:
        t0 = time.perf_counter()
        oracle.run_backward(*args, num_iters=case.num_iters, threads=threads)
        t_total += time.perf_counter() - t0
        done += count
        passes += 1
    return done / t_total, threads, (f"{passes} pass(es) over {count} tokens of the backward workload "
                                     f"({t_total:.1f} s, double precision, all five gradients)"), t_total


def bench_bwd(args, device, world, rank, local):
    """The backward at the prefill shape (Sinkhorn form, no gamma): device-timed
    steps of the five launches, the roofline of the contraction kernel, an
    end-to-end number with host buffers, and the oracle on host cores."""
    import torch
    T, n, D = args.tokens, WORKLOAD["n"], WORKLOAD["D"]
    mode_name = "fp32" if args.mode == 0 else "tf32"
    cfg = {"workload": f"pre backward T={T} n={n} D={D} iters=20 {mode_name} Sinkhorn form (b=4, s=8192)",
           "tokens_per_rank": T, "n": n, "D": D, "num_iters": 20, "impl_mode": mode_name, "gamma": None,
           "grad_x_post": None, "l2": "inputs (4.3 GB/step) exceed L2; no flush needed",
           "parallelism": f"token-sharded x{world}" + (" + all-reduce of grad_phi/alpha/bias" if world > 1 else "")}
    if args.impl == "reference":
        # the oracle alone: its own forward makes the saved intermediates of
        # the sampled tokens, then its backward is timed on them
        if rank != 0:
            return 0
        case, saved, g = bwd_reference_inputs(device, T, n, D, args.mode, 20000)
        per_step = 60.0 / (args.steps + args.warmup)
        probe, _, _, _ = bwd_oracle_rate(case, saved, g, 0.0, 64)
        tokens = int(max(1, min(case.T, probe * per_step)))
        rate, threads, sample, dt = bwd_oracle_rate(case, saved, g, 60.0 * args.steps / (args.steps + args.warmup),
                                                    tokens)
        print(json.dumps({"impl": "reference", "metric": BWD_METRIC, "value": rate, "unit": "tokens/s",
                          "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": 1e3 * T / rate, "higher_is_better": True, "scaling": "weak",
                          "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
                          "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                           "sample": sample},
                          "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}))
        return 0
    from mhc_hyper_connection_gb300 import build as mbuild
    mbuild.build()
    case, saved, g = bwd_inputs(device, T, n, D, world, rank, args.mode)
    from mhc_hyper_connection_gb300 import MhcPre, mhc_pre_last_launch, mhc_pre_set_profile_events
    op = MhcPre(n, D, alpha_len=3, num_iters=20, impl_mode=args.mode, need_backward=True)
    grads = op.allocate_backward(T, device)
    stream = torch.cuda.current_stream(device)

    def step(gr=grads):
        op.backward(case.x, case.phi, case.alpha, None, g.g_in, g.g_post, g.g_res, saved, gr, stream=stream)
        allreduce_weight_grads(gr, world)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if op.status(grads) != 0:
        raise RuntimeError("device-side error during warm-up")
    K = args.steps
    ev_k = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in ev_k:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    clocks.mark(True)
    e0.record(stream)
    for i in range(K):
        mhc_pre_set_profile_events(op.handle, ev_k[i][0].cuda_event, ev_k[i][1].cuda_event)
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark(False)
    if world > 1:
        torch.distributed.barrier()
    mhc_pre_set_profile_events(op.handle, 0, 0)
    time.sleep(0.2)
    clocks.stop()
    if op.status(grads) != 0:
        raise RuntimeError("device-side error during the timed steps")
    cfg["launch"] = mhc_pre_last_launch(op.handle)[1]
    cfg["launch"]["kernel"] = "bw_main_kernel"
    elapsed = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, device)
    kern = statistics.median(a.elapsed_time(b) for a, b in ev_k) / 1e3   # median launch
    per_step = elapsed / K

    # ---- end to end with host buffers: every step copies its inputs in from
    # pinned host memory and the four fp32/bf16 gradients back out.  Steps are
    # pipelined over three streams with two buffer sets (copy-in of step i+1,
    # compute of step i, copy-out of step i-1 overlap).
    e2e = None
    if not args.no_e2e:
        names_in = [("x", case.x), ("g_in", g.g_in), ("g_post", g.g_post), ("g_res", g.g_res)] + \
                   [(k, v) for k, v in saved.items()]
        host_in = {k: v.cpu().pin_memory() for k, v in names_in}
        dev_in = [{k: torch.empty_like(v) for k, v in names_in} for _ in range(2)]
        outs = ("grad_x", "grad_phi", "grad_alpha", "grad_bias")
        gsets = [grads, op.allocate_backward(T, device)]
        host_out = [{k: torch.empty_like(grads[k], device="cpu").pin_memory() for k in outs} for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
        ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "comp", "out")}

        def e2e_steps(n_steps, first):
            for i in range(n_steps):
                bi = i % 2
                if i >= 2 or not first:
                    s_in.wait_event(ev["comp"][bi])          # buffer bi's inputs are free
                with torch.cuda.stream(s_in):
                    for k, v in host_in.items():
                        dev_in[bi][k].copy_(v, non_blocking=True)
                ev["in"][bi].record(s_in)
                stream.wait_event(ev["in"][bi])
                if i >= 2 or not first:
                    stream.wait_event(ev["out"][bi])         # buffer bi's gradients are copied out
                d = dev_in[bi]
                op.backward(d["x"], case.phi, case.alpha, None, d["g_in"], d["g_post"], d["g_res"],
                            {k: d[k] for k in saved}, gsets[bi], stream=stream)
                ev["comp"][bi].record(stream)
                s_out.wait_event(ev["comp"][bi])
                with torch.cuda.stream(s_out):
                    for k in outs:
                        host_out[bi][k].copy_(gsets[bi][k], non_blocking=True)
                ev["out"][bi].record(s_out)

        e2e_steps(2, True)
        torch.cuda.synchronize()
        Ke = max(3, min(K, 10))
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s_in)
        e2e_steps(Ke, False)
        b.record(s_out)
        torch.cuda.synchronize()
        t_e2e = max_over_ranks(a.elapsed_time(b) / 1e3, world, device)
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = sum(v.numel() * v.element_size() for v in host_out[0].values())
        e2e = {"value": world * T * Ke / t_e2e, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": Ke}
        del host_in, dev_in, host_out, gsets

    peak, peak_src = hbm_peak()
    lb_main = T * bwd_main_token_bytes(n, D)
    lb_step = T * bwd_token_bytes(n, D) + 2 * 4 * (n * n + 2 * n) * n * D
    achieved = lb_main / kern / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": recorded_traffic("bw_main_kernel", T), "kernel": "bw_main_kernel", "kernel_ms": kern * 1e3,
            "algorithmic_bytes": lb_main, "peak_source": f"hbm_gbs of {peak_src}"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        probe, _, _, _ = bwd_oracle_rate(case, saved, g, 0.0, 64)
        rate, threads, sample, dt = bwd_oracle_rate(case, saved, g, 10.0, int(max(64, min(T, probe * 3))))
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps({
            "metric": BWD_METRIC, "value": world * T * K / elapsed, "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
            "hbm_gbs_step": lb_step / per_step / 1e9, "hbm_frac_step": lb_step / per_step / 1e9 / peak,
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 5 * K * world,
            "clocks": clocks.summary()}))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def torch_int16():
    import torch
    return torch.int16


# ----------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--tokens", type=int, default=WORKLOAD["T"])
    ap.add_argument("--mode", type=int, default=WORKLOAD["impl_mode"], choices=[0, 1])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--x-dtype", choices=["bf16", "fp16"], default="bf16",
                    help="element type of x and y (forward)")
    ap.add_argument("--route", choices=["fused", "composite"], default="fused",
                    help="forward: the fused kernel, or the composite three-launch route (a debug aid)")
    ap.add_argument("--batch-consistent", action="store_true",
                    help="forward in batch-consistent mode (results per token independent of T)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel", choices=["auto", "cluster", "grid", "resident"], default="auto",
                    help="forward: force a fused kernel (default: the library's choice)")
    ap.add_argument("--cluster", type=int, default=0, help="forward: force a cluster size (0: the library's)")
    ap.add_argument("--tm-buffers", type=int, default=0, help="resident forward: TMEM chunk buffers (0: the library's)")
    ap.add_argument("--prepared-weights", action="store_true",
                    help="forward: prepare phi's planes once (mhc_pre_prepare_weights) and time steady-state calls")
    ap.add_argument("--op", choices=["pre", "post", "bwd"], default="pre",
                    help="pre: the pre-mapping forward (the headline); post: the post-mapping (hc_post); "
                         "bwd: the pre-mapping backward")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo",
                                init_method="env://")
    device = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    if device.type == "cuda":
        torch.cuda.set_device(device)
    from mhc_synth import make_case

    T, n, D = args.tokens, WORKLOAD["n"], WORKLOAD["D"]
    mode_name = "fp32" if args.mode == 0 else "tf32"
    cfg = {"workload": f"prefill T={T} n={n} D={D} iters=20 {mode_name} (b=4, s=8192)",
           "tokens_per_rank": T, "n": n, "D": D, "num_iters": 20, "impl_mode": mode_name,
           "gamma": None, "l2": "inputs (2.35 GB/step) exceed L2; no flush needed",
           "parallelism": f"token-sharded x{world} (no collective)"}
    if args.route == "composite":
        cfg["route"] = "composite (inv_rms, mixes, sinkhorn launches)"
        cfg["workload"] += " composite route"
    if args.x_dtype != "bf16" or args.batch_consistent:
        cfg["x_dtype"] = args.x_dtype
        cfg["batch_consistent"] = bool(args.batch_consistent)
        cfg["workload"] += f" x={args.x_dtype}" + (" batch-consistent" if args.batch_consistent else "")

    if args.op == "post":
        return bench_post(args, device, world, rank, local)
    if args.op == "bwd":
        return bench_bwd(args, device, world, rank, local)

    if args.impl == "reference":
        if rank != 0:
            return 0
        case = make_case("prefill", device=device, T=T, impl_mode=args.mode)
        # bounded: each step is a sample sized so the whole run takes about a minute
        per_step = 60.0 / (args.steps + args.warmup)
        probe, _, _, _ = oracle_rate(case, 0.0, 256)
        tokens = int(max(1, min(case.T, probe * per_step)))
        rate, threads, sample, dt = oracle_rate(case, 60.0 * args.steps / (args.steps + args.warmup), tokens)
        line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * T / rate, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
                "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                 "sample": f"{sample} of the prefill workload ({dt:.1f} s)"},
                "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    from mhc_hyper_connection_gb300 import (MhcPre, mhc_pre_last_kernel, mhc_pre_last_launch,
                                            mhc_pre_set_profile_events)
    from mhc_hyper_connection_gb300 import build as mbuild, MHC_DTYPE_BF16, MHC_DTYPE_FP16
    mbuild.build()
    xdt = torch.float16 if args.x_dtype == "fp16" else torch.bfloat16
    case = rank_shard(lambda **k: make_case("prefill", device=device, impl_mode=args.mode, x_dtype=xdt, **k),
                      T, world, rank)
    kernel_code = {"auto": 0, "cluster": 1, "grid": 2, "resident": 3}[args.kernel]
    op = MhcPre(n, D, alpha_len=3, num_iters=20, impl_mode=args.mode, batch_consistent=args.batch_consistent,
                x_dtype=MHC_DTYPE_FP16 if args.x_dtype == "fp16" else MHC_DTYPE_BF16,
                kernel=kernel_code, cluster=args.cluster, tm_buffers=args.tm_buffers)
    out = op.allocate(T, device)
    stream = torch.cuda.current_stream(device)
    weights = op.prepare_weights(case.phi, stream=stream) if args.prepared_weights else None
    if weights is not None:
        cfg["weights"] = "prepared once (mhc_pre_prepare_weights); a step is the header copy and the fused kernel"
        cfg["workload"] += " prepared weights"

    def step():
        if args.route == "composite":
            op.run_composite(case.x, case.phi, case.alpha, case.bias, out, stream=stream)
        else:
            op.run(case.x, case.phi, case.alpha, case.bias, out, stream=stream, weights=weights)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if op.status(out) != 0:
        raise RuntimeError("device-side error during warm-up")

    # ---- device-timed steps (whole step), plus the fused kernel alone
    K = args.steps
    ev_k = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(K)]
    for a, b in ev_k:                 # materialise the CUDA events
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    clocks.mark(True)
    e0.record(stream)
    for i in range(K):
        mhc_pre_set_profile_events(op.handle, ev_k[i][0].cuda_event, ev_k[i][1].cuda_event)
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark(False)
    if world > 1:
        torch.distributed.barrier()
    mhc_pre_set_profile_events(op.handle, 0, 0)
    time.sleep(0.2)
    clocks.stop()
    if op.status(out) != 0:
        raise RuntimeError("device-side error during the timed steps")
    cfg["launch"] = mhc_pre_last_launch(op.handle)[1]
    cfg["launch"]["kernel"] = mhc_pre_last_kernel(op.handle)
    elapsed = e0.elapsed_time(e1) / 1e3
    kern = statistics.median(a.elapsed_time(b) for a, b in ev_k) / 1e3   # median launch
    elapsed_max = max_over_ranks(elapsed, world, device)
    if args.route == "composite":
        # three launches and no single fused kernel: the roofline is the route's
        cfg["launch"] = {"kernel": "composite route (stage_inv_rms, stage_mixes, stage_sinkhorn)"}
        kern = elapsed_max / K
    value = world * T * K / elapsed_max

    # ---- end to end through the C ABI with host buffers
    # Each step copies its x from pinned host memory, runs the forward and
    # copies y, hPost and comb back.  Steps are pipelined over three streams
    # with two buffer sets (copy-in of step i+1, compute of step i and
    # copy-out of step i-1 overlap), as a caller streaming batches would.
    e2e = None
    if not args.no_e2e:
        x_host = case.x.cpu().pin_memory()
        outs = [out, op.allocate(T, device)]
        x_devs = [torch.empty_like(case.x), torch.empty_like(case.x)]
        hosts = [[torch.empty_like(o[k], device="cpu").pin_memory() for k in ("y", "h_post", "h_res")]
                 for o in outs]
        s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
        ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "comp", "out")}
        Ke = max(3, min(K, 20))

        def e2e_steps(n_steps, first):
            for i in range(n_steps):
                bi = i % 2
                if i >= 2 or not first:
                    s_in.wait_event(ev["comp"][bi])          # buffer bi's x is free
                with torch.cuda.stream(s_in):
                    x_devs[bi].copy_(x_host, non_blocking=True)
                ev["in"][bi].record(s_in)
                stream.wait_event(ev["in"][bi])
                if i >= 2 or not first:
                    stream.wait_event(ev["out"][bi])         # buffer bi's outputs are copied out
                op.run(x_devs[bi], case.phi, case.alpha, case.bias, outs[bi], stream=stream, weights=weights)
                ev["comp"][bi].record(stream)
                s_out.wait_event(ev["comp"][bi])
                with torch.cuda.stream(s_out):
                    for hbuf, k in zip(hosts[bi], ("y", "h_post", "h_res")):
                        hbuf.copy_(outs[bi][k], non_blocking=True)
                ev["out"][bi].record(s_out)

        e2e_steps(2, True)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s_in)
        e2e_steps(Ke, False)
        b.record(s_out)
        torch.cuda.synchronize()
        t_e2e = max_over_ranks(a.elapsed_time(b) / 1e3, world, device)
        h2d = case.x.numel() * case.x.element_size()
        d2h = sum(t.numel() * t.element_size() for t in (out["y"], out["h_post"], out["h_res"]))
        e2e = {"value": world * T * Ke / t_e2e, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": Ke}
        del x_host, hosts, x_devs, outs

    # ---- roofline of the fused kernel
    peak, peak_src = hbm_peak()
    lb = launch_bytes(T, n, D)
    achieved = lb / kern / 1e9
    kernel = cfg["launch"]["kernel"]
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": recorded_traffic(kernel, T) if kernel in KERNEL_SOURCES else None,
            "kernel": kernel, "kernel_ms": kern * 1e3,
            "algorithmic_bytes": lb, "peak_source": f"hbm_gbs of {peak_src}"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, threads, sample, dt = oracle_rate(case, 10.0, case.T)
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{sample} of the prefill workload ({dt:.1f} s, double precision)"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": K, "warmup": args.warmup, "ms_per_step": elapsed_max / K * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.x_dtype,
                "data": "synthetic", "config": cfg,
                "hbm_gbs_step": lb / (elapsed_max / K) / 1e9,
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": (3 if args.route == "composite" else (1 if weights is not None else 2)) * K * world,
                "clocks": clocks.summary()}
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
