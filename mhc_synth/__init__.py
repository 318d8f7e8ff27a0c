"""Seeded synthetic inputs for the mHC pre-mapping forward.

This module only draws random numbers and lays them out in the shapes the
operator takes. It holds none of the operator's arithmetic, and it imports
neither the CUDA library nor the oracle, so both sides can be fed from it.

Generator
---------
Small tensors (and x up to ``SPLITMIX_X_LIMIT`` elements) come from a
counter-based SplitMix64 stream: the i-th 64-bit word of the stream with key
``s`` is ``mix64(s + (i + 1) * 0x9E3779B97F4A7C15)``, where ``mix64`` is the
SplitMix64 finaliser (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014).  Uniforms take the top 53 bits; normals use
Box-Muller on two consecutive words (cosine branch only).

Large x (prefill-sized, ~1e9 elements) is drawn on the target device with
torch's own seeded generator, which is what keeps a full-size benchmark from
spending a minute on the host.  Whatever produces x, the oracle is always
given a host copy of the very same values.

Shapes and distributions follow the five workloads the operator is measured
on (tiny / training-shaped / decode-shaped / prefill / generic-n).  ``N(0,s)``
means mean 0 and standard deviation s.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
SPLITMIX_X_LIMIT = 1 << 25   # elements of x drawn on the host with SplitMix64

# One key per tensor so that changing one shape never shifts another stream.
_TAGS = {"x": 1, "phi": 2, "alpha": 3, "bias": 4, "gamma": 5, "pre_mix": 6,
         "outlier": 7, "misc": 8, "post": 9, "comb": 10, "g_post": 11, "g_res": 12}


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tag: str) -> np.uint64:
    """Key of the SplitMix64 stream for one named tensor."""
    base = np.array([(int(seed) & 0xFFFFFFFF) | (_TAGS[tag] << 40)], dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(base)[0]


def words(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Words start .. start+count-1 of the stream with this key."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + idx * GOLDEN)


def uniform(key: np.uint64, count: int, start: int = 0) -> np.ndarray:
    """U[0,1) doubles, 53-bit."""
    return (words(key, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(key: np.uint64, count: int, std: float = 1.0, mean: float = 0.0,
           chunk: int = 1 << 22) -> np.ndarray:
    """N(mean, std) doubles via Box-Muller on word pairs (2i, 2i+1)."""
    out = np.empty(count, dtype=np.float64)
    for s in range(0, count, chunk):
        m = min(chunk, count - s)
        u = uniform(key, 2 * m, start=2 * s)
        u1 = 1.0 - u[0::2]          # (0, 1]
        u2 = u[1::2]
        out[s:s + m] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return out * std + mean


def to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float64/float32 -> bf16 bit patterns (round to nearest even)."""
    f = np.ascontiguousarray(v, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounding = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return ((u + rounding) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Case:
    """One workload: operator attributes plus the input tensors (torch)."""
    name: str
    T: int
    n: int
    D: int
    alpha_len: int
    num_iters: int
    norm_eps: float
    hc_eps: float
    impl_mode: int
    need_backward: bool
    x: torch.Tensor                  # bf16 [T, n, D]
    phi: torch.Tensor                # f32 [R, n*D]
    alpha: torch.Tensor              # f32 [alpha_len]
    bias: torch.Tensor               # f32 [R]
    gamma: Optional[torch.Tensor]    # f32 [n, D] or None
    pre_mix: Optional[torch.Tensor]  # f32 [T, n] or None

    @property
    def R(self) -> int:
        return self.n * self.n + 2 * self.n if self.alpha_len == 3 else 2 * self.n

    @property
    def K(self) -> int:
        return self.n * self.D


# Workload recipes (T, n, D, extras).  The phi scale 1/sqrt(nD) keeps the
# projection O(1), which is the stable-input range the pages recommend.
WORKLOADS = {
    "tiny": dict(T=64, n=4, D=256, alpha="fixed", alpha_vals=(0.8, 1.2, 1.0),
                 gamma=False, pre_mix=False, need_backward=False, impl_mode=0),
    "training": dict(T=4096, n=4, D=4096, alpha="uniform", gamma=True,
                     pre_mix=False, need_backward=True, impl_mode=0),
    "decode": dict(T=64, n=4, D=7168, alpha="fixed", alpha_vals=(1.0, 1.0, 1.0),
                   gamma=False, pre_mix=False, need_backward=False, impl_mode=0,
                   outliers=True),
    "prefill": dict(T=32768, n=4, D=7168, alpha="uniform", gamma=False,
                    pre_mix=False, need_backward=False, impl_mode=0),
    "generic_a": dict(T=16384, n=8, D=2048, alpha="uniform", gamma=False,
                      pre_mix=True, need_backward=False, impl_mode=0),
    "generic_b": dict(T=16384, n=8, D=2048, alpha="uniform2", gamma=False,
                      pre_mix=False, need_backward=False, impl_mode=0),
}


def _x_tensor(seed, T, n, D, outliers, device, dtype=None):
    """x drawn N(0, 1) (with the decode workload's outliers), rounded to
    bf16 (default) or to fp16 (round to nearest even in both)."""
    dtype = torch.bfloat16 if dtype is None else dtype
    numel = T * n * D
    if numel <= SPLITMIX_X_LIMIT:
        v = normal(stream_key(seed, "x"), numel)
        if outliers:
            hit = uniform(stream_key(seed, "outlier"), numel) < 0.01
            v = np.where(hit, v * 20.0, v)
        if dtype == torch.float16:
            return torch.from_numpy(v.astype(np.float16).reshape(T, n, D)).to(device)
        bits = to_bf16_bits(v).view(np.int16).reshape(T, n, D)
        return torch.from_numpy(bits.copy()).view(torch.bfloat16).to(device)
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + 17)
    x = torch.randn((T, n, D), generator=g, device=device, dtype=torch.float32)
    if outliers:
        hit = torch.rand((T, n, D), generator=g, device=device) < 0.01
        x = torch.where(hit, x * 20.0, x)
    return x.to(dtype)


def make_case(name: str, *, seed: int = 0, device="cpu", T: Optional[int] = None,
              n: Optional[int] = None, D: Optional[int] = None,
              impl_mode: Optional[int] = None, num_iters: int = 20,
              need_backward: Optional[bool] = None, gamma: Optional[bool] = None,
              pre_mix: Optional[bool] = None, alpha_len: Optional[int] = None,
              x_dtype=None) -> Case:
    """Build a workload by name; any shape or flag may be overridden
    (x_dtype: torch.bfloat16, the default, or torch.float16)."""
    w = dict(WORKLOADS[name])
    T = w["T"] if T is None else T
    n = w["n"] if n is None else n
    D = w["D"] if D is None else D
    if alpha_len is None:
        alpha_len = 2 if w["alpha"] == "uniform2" else 3
    K = n * D
    R_full = n * n + 2 * n
    R = R_full if alpha_len == 3 else 2 * n

    x = _x_tensor(seed, T, n, D, w.get("outliers", False), device, x_dtype)
    # phi: N(0, 1/sqrt(K)) over the full [n^2+2n, K] matrix; the two-gate
    # variant takes its first 2n rows (same stream, so rows agree).
    phi_full = normal(stream_key(seed, "phi"), R_full * K, std=1.0 / math.sqrt(K))
    phi = phi_full.reshape(R_full, K)[:R].astype(np.float32)
    if w["alpha"] == "fixed":
        alpha = np.array(w["alpha_vals"][:alpha_len], dtype=np.float32)
    else:
        alpha = (0.5 + uniform(stream_key(seed, "alpha"), 3))[:alpha_len].astype(np.float32)
    bias = normal(stream_key(seed, "bias"), R_full, std=0.1)[:R].astype(np.float32)
    use_gamma = w["gamma"] if gamma is None else gamma
    g_t = None
    if use_gamma:
        g_t = torch.from_numpy(
            normal(stream_key(seed, "gamma"), n * D, std=0.05, mean=1.0)
            .astype(np.float32).reshape(n, D)).to(device)
    use_pm = w["pre_mix"] if pre_mix is None else pre_mix
    pm_t = None
    if use_pm:
        pm_t = torch.from_numpy(uniform(stream_key(seed, "pre_mix"), T * n)
                                .astype(np.float32).reshape(T, n)).to(device)
    return Case(
        name=name, T=T, n=n, D=D, alpha_len=alpha_len, num_iters=num_iters,
        norm_eps=1e-6, hc_eps=1e-6,
        impl_mode=w["impl_mode"] if impl_mode is None else impl_mode,
        need_backward=w["need_backward"] if need_backward is None else need_backward,
        x=x, phi=torch.from_numpy(np.ascontiguousarray(phi)).to(device),
        alpha=torch.from_numpy(alpha).to(device),
        bias=torch.from_numpy(bias).to(device), gamma=g_t, pre_mix=pm_t)


def sample_tokens(T: int, count: int, seed: int = 0, tile: int = 128) -> np.ndarray:
    """Token indices for sampled checks: first/last tokens, tile edges and a
    seeded random spread, sorted and unique."""
    picks = {0, T - 1}
    for edge in range(tile, T, tile * max(1, (T // tile) // 16)):
        picks.update({edge - 1, edge})
    rnd = (uniform(stream_key(seed, "misc"), count) * T).astype(np.int64)
    picks.update(int(v) for v in rnd)
    out = np.array(sorted(p for p in picks if 0 <= p < T), dtype=np.int64)
    return out


@dataclasses.dataclass
class PostCase:
    """Inputs of the post-mapping: layer output x bf16 [T, D], residual
    streams bf16 [T, n, D], post fp32 [T, n] in (0, 2), comb fp32 [T, n, n]
    with entries in [0, 1/n) (the scale of a doubly stochastic mix)."""
    T: int
    n: int
    D: int
    x: torch.Tensor
    residual: torch.Tensor
    post: torch.Tensor
    comb: torch.Tensor


def make_post_case(*, seed: int = 0, device="cpu", T: int = 64, n: int = 4, D: int = 256) -> PostCase:
    x = _x_tensor(seed * 7 + 1, T, 1, D, False, device).reshape(T, D)
    residual = _x_tensor(seed * 7 + 2, T, n, D, False, device)
    post = torch.from_numpy((2.0 * uniform(stream_key(seed, "post"), T * n)).astype(np.float32)
                            .reshape(T, n)).to(device)
    comb = torch.from_numpy((uniform(stream_key(seed, "comb"), T * n * n) / n).astype(np.float32)
                            .reshape(T, n, n)).to(device)
    return PostCase(T=T, n=n, D=D, x=x, residual=residual, post=post, comb=comb)


@dataclasses.dataclass
class BwdGrads:
    """Upstream gradients of the pre-mapping's outputs: grad_h_in bf16 [T, D]
    (of y), grad_h_post fp32 [T, n], grad_h_res fp32 [T, n, n] (of the
    Sinkhorn output, or of the res logits), and optionally grad_x_post bf16
    [T, n, D] (the post-mapping's gradient of x).  All N(0, 1)."""
    g_in: torch.Tensor
    g_post: torch.Tensor
    g_res: torch.Tensor
    g_x_post: Optional[torch.Tensor]


def make_bwd_grads(*, seed: int = 0, device="cpu", T: int = 64, n: int = 4, D: int = 256,
                   grad_x_post: bool = False) -> BwdGrads:
    g_in = _x_tensor(seed * 7 + 3, T, 1, D, False, device).reshape(T, D)
    g_post = torch.from_numpy(normal(stream_key(seed, "g_post"), T * n).astype(np.float32)
                              .reshape(T, n)).to(device)
    g_res = torch.from_numpy(normal(stream_key(seed, "g_res"), T * n * n).astype(np.float32)
                             .reshape(T, n, n)).to(device)
    gxp = _x_tensor(seed * 7 + 4, T, n, D, False, device) if grad_x_post else None
    return BwdGrads(g_in=g_in, g_post=g_post, g_res=g_res, g_x_post=gxp)
