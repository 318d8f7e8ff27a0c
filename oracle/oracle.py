"""TEST INFRASTRUCTURE: build and call the C oracle; a Decimal brute force.

Only tests, the smoke check and the benchmark's CPU baseline use this file.

Two independent statements of the same operator live here:

* ``run`` -- the C oracle in ``mhc_pre_oracle.c`` (double precision, threads
  over tokens), used for every parity comparison;
* ``brute_force_decimal`` -- a 50-digit ``decimal`` evaluation written from
  the pages in a different shape (explicit segment slicing, Sinkhorn as
  diagonal scalings of the softmax), used only on tiny inputs to pin the C
  oracle's loops and indexing.

``run_post`` is the C oracle of the post-mapping (``mhc_post_oracle.c``);
``run_backward`` that of the pre-mapping's backward (``mhc_pre_bwd_oracle.c``).
"""
from __future__ import annotations

import ctypes
import dataclasses
import decimal
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, f) for f in ("mhc_pre_oracle.c", "mhc_post_oracle.c", "mhc_pre_bwd_oracle.c")]
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libmhc_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags: no -march, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or any(os.path.getmtime(_SO) < os.path.getmtime(f) for f in _SRCS):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", "-fno-fast-math", *_SRCS, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            f = lib.mhc_oracle_pre
            P = ctypes.c_void_p
            f.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                          ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_int,
                          P, P, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_int]
            f.restype = ctypes.c_int
            f16 = lib.mhc_oracle_pre_f16
            f16.argtypes = f.argtypes
            f16.restype = ctypes.c_int
            hv = lib.mhc_oracle_half_value
            hv.argtypes = [ctypes.c_uint16]
            hv.restype = ctypes.c_double
            g = lib.mhc_oracle_post
            g.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P, P, P, P, P, ctypes.c_int]
            g.restype = ctypes.c_int
            b = lib.mhc_oracle_pre_backward
            I64 = ctypes.c_int64
            b.argtypes = [I64, I64, I64, ctypes.c_int, ctypes.c_double,
                          P, P, P, P, P, P, P, P, P, P, P, P, P, P,
                          I64, P, I64, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_int]
            b.restype = ctypes.c_int
            _lib = lib
    return _lib


@dataclasses.dataclass
class OracleOut:
    y: np.ndarray          # [T, D]  exact weighted sum (not rounded to bf16)
    h_post: np.ndarray     # [T, n]
    h_res: np.ndarray      # [T, n, n] (comb after Sinkhorn; zeros for two gates)
    h_pre: np.ndarray      # [T, n]
    inv_rms: np.ndarray    # [T]
    h_mix: np.ndarray      # [T, R]
    sum_out: Optional[np.ndarray]   # [2I, T, n]
    norm_out: Optional[np.ndarray]  # [2I, T, n, n]


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def run(x_bits: np.ndarray, phi: np.ndarray, alpha: np.ndarray, bias: np.ndarray,
        gamma: Optional[np.ndarray] = None, pre_mix: Optional[np.ndarray] = None, *,
        num_iters: int = 20, norm_eps: float = 1e-6, hc_eps: float = 1e-6,
        hf32: int = 0, backward: bool = True, threads: Optional[int] = None,
        x_fp16: bool = False) -> OracleOut:
    """Evaluate the oracle.  x_bits: uint16/int16 bit patterns [T, n, D] of bf16
    values, or of IEEE fp16 values with x_fp16=True.  hf32: 0 exact projection;
    1 (or True) the HcPre page's HF32 simulation on the operands x (.) gamma and
    phi; 2 that truncation on the folded weight gamma (.) phi (rounded to fp32
    first), x exact."""
    hf32 = int(hf32)
    if hf32 not in (0, 1, 2):
        raise ValueError("hf32 must be 0, 1 or 2")
    x_bits = np.ascontiguousarray(x_bits).view(np.uint16)
    T, n, D = x_bits.shape
    alpha = np.ascontiguousarray(alpha, dtype=np.float32)
    alpha_len = int(alpha.shape[0])
    R = n * n + 2 * n if alpha_len == 3 else 2 * n
    phi = np.ascontiguousarray(phi, dtype=np.float32).reshape(R, n * D)
    bias = np.ascontiguousarray(bias, dtype=np.float32).reshape(R)
    if gamma is not None:
        gamma = np.ascontiguousarray(gamma, dtype=np.float32).reshape(n * D)
    if pre_mix is not None:
        pre_mix = np.ascontiguousarray(pre_mix, dtype=np.float32).reshape(T, n)
    y = np.zeros((T, D))
    h_post = np.zeros((T, n))
    h_res = np.zeros((T, n, n))
    h_pre = np.zeros((T, n))
    inv_rms = np.zeros(T)
    h_mix = np.zeros((T, R))
    sb = backward and alpha_len == 3
    sum_out = np.zeros((2 * num_iters, T, n)) if sb else None
    norm_out = np.zeros((2 * num_iters, T, n, n)) if sb else None
    if threads is None:
        threads = os.cpu_count() or 1
    fn = _load().mhc_oracle_pre_f16 if x_fp16 else _load().mhc_oracle_pre
    rc = fn(
        T, n, D, alpha_len, num_iters, norm_eps, hc_eps, int(hf32),
        _ptr(x_bits), _ptr(phi), _ptr(alpha), _ptr(bias), _ptr(gamma), _ptr(pre_mix),
        _ptr(y), _ptr(h_post), _ptr(h_res), _ptr(h_pre), _ptr(inv_rms), _ptr(h_mix),
        _ptr(sum_out), _ptr(norm_out), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return OracleOut(y, h_post, h_res, h_pre, inv_rms, h_mix, sum_out, norm_out)


def half_value(bits: int) -> float:
    """The oracle's decoding of one IEEE fp16 bit pattern (for its pin)."""
    return float(_load().mhc_oracle_half_value(int(bits) & 0xFFFF))


def run_post(x_bits: np.ndarray, residual_bits: np.ndarray, post: np.ndarray, comb: np.ndarray, *,
             threads: Optional[int] = None) -> np.ndarray:
    """Post-mapping oracle: out[t, j, d] = post[t, j] x[t, d] + sum_i comb[t, i, j]
    residual[t, i, d], in double, unrounded.  x_bits: bf16 bits [T, D];
    residual_bits: bf16 bits [T, n, D]; post [T, n]; comb [T, n, n]."""
    residual_bits = np.ascontiguousarray(residual_bits).view(np.uint16)
    T, n, D = residual_bits.shape
    x_bits = np.ascontiguousarray(x_bits).view(np.uint16).reshape(T, D)
    post = np.ascontiguousarray(post, dtype=np.float32).reshape(T, n)
    comb = np.ascontiguousarray(comb, dtype=np.float32).reshape(T, n, n)
    out = np.zeros((T, n, D))
    if threads is None:
        threads = os.cpu_count() or 1
    rc = _load().mhc_oracle_post(T, n, D, _ptr(x_bits), _ptr(residual_bits), _ptr(post), _ptr(comb),
                                 _ptr(out), int(threads))
    if rc != 0:
        raise ValueError("post oracle rejected its arguments")
    return out


@dataclasses.dataclass
class BwdOut:
    grad_x: Optional[np.ndarray]          # [tokens, n, D] (selected tokens), unrounded
    grad_x_abs: Optional[np.ndarray]      # sum of |terms| of each grad_x element
    grad_phi: Optional[np.ndarray]        # [R, columns]
    grad_phi_abs: Optional[np.ndarray]
    grad_gamma: Optional[np.ndarray]      # [columns] (with gamma)
    grad_gamma_abs: Optional[np.ndarray]
    grad_alpha: np.ndarray                # [3]
    grad_alpha_abs: np.ndarray
    grad_bias: np.ndarray                 # [R]
    grad_bias_abs: np.ndarray


def _f64(a, shape=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a if shape is None else a.reshape(shape)


def run_backward(x_bits, phi, alpha, gamma, grad_h_in_bits, grad_h_post, grad_h_res,
                 inv_rms, h_mix, h_pre, h_post, sum_out=None, norm_out=None,
                 grad_x_post_bits=None, *, num_iters: int = 20, hc_eps: float = 1e-6,
                 tokens=None, columns=None, want_grad_x: bool = True, want_grad_phi: bool = True,
                 threads: Optional[int] = None) -> BwdOut:
    """Backward oracle of the pre-mapping with Sinkhorn (three gates).

    x_bits, grad_x_post_bits: bf16 bits [T, n, D]; grad_h_in_bits: bf16 bits
    [T, D]; every other array is taken in float64 exactly as given (pass the
    forward's fp32 intermediates to mirror the device, or double ones for the
    analytic pins).  With sum_out / norm_out, grad_h_res is the gradient of
    the Sinkhorn output; without them, of the res logits.  ``tokens`` selects
    the rows of grad_x, ``columns`` the columns of grad_phi / grad_gamma."""
    x_bits = np.ascontiguousarray(x_bits).view(np.uint16)
    T, n, D = x_bits.shape
    R, K = n * n + 2 * n, n * D
    gh = np.ascontiguousarray(grad_h_in_bits).view(np.uint16).reshape(T, D)
    gxp = None if grad_x_post_bits is None else \
        np.ascontiguousarray(grad_x_post_bits).view(np.uint16).reshape(T, n, D)
    phi = _f64(phi, (R, K))
    alpha = _f64(alpha, (3,))
    gamma = _f64(gamma, (K,))
    ghp, ghr = _f64(grad_h_post, (T, n)), _f64(grad_h_res, (T, n, n))
    ir, hm, hp, hq = _f64(inv_rms, (T,)), _f64(h_mix, (T, R)), _f64(h_pre, (T, n)), _f64(h_post, (T, n))
    so = _f64(sum_out, (2 * num_iters, T, n))
    no = _f64(norm_out, (2 * num_iters, T, n, n))
    tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
    col = None if columns is None else np.ascontiguousarray(columns, dtype=np.int64)
    nt = T if tok is None else len(tok)
    nc = K if col is None else len(col)
    gx = np.zeros((nt, n, D)) if want_grad_x else None
    gxa = np.zeros((nt, n, D)) if want_grad_x else None
    gp = np.zeros((R, nc)) if want_grad_phi else None
    gpa = np.zeros((R, nc)) if want_grad_phi else None
    gg = np.zeros(nc) if (want_grad_phi and gamma is not None) else None
    gga = np.zeros(nc) if gg is not None else None
    ga, gaa = np.zeros(3), np.zeros(3)
    gb, gba = np.zeros(R), np.zeros(R)
    if threads is None:
        threads = os.cpu_count() or 1
    rc = _load().mhc_oracle_pre_backward(
        T, n, D, num_iters, hc_eps, _ptr(x_bits), _ptr(phi), _ptr(alpha), _ptr(gamma), _ptr(gh),
        _ptr(ghp), _ptr(ghr), _ptr(ir), _ptr(hm), _ptr(hp), _ptr(hq), _ptr(so), _ptr(no), _ptr(gxp),
        nt, _ptr(tok), nc, _ptr(col), _ptr(gx), _ptr(gxa), _ptr(gp), _ptr(gpa), _ptr(gg), _ptr(gga),
        _ptr(ga), _ptr(gaa), _ptr(gb), _ptr(gba), int(threads))
    if rc != 0:
        raise ValueError("backward oracle rejected its arguments" if rc == 1 else "backward oracle: out of memory")
    return BwdOut(gx, gxa, gp, gpa, gg, gga, ga, gaa, gb, gba)


# ---------------------------------------------------------------------------
# 50-digit brute force (tiny inputs only).
# ---------------------------------------------------------------------------

def brute_force_decimal(x_vals, phi, alpha, bias, gamma=None, pre_mix=None, *,
                        num_iters=20, norm_eps=1e-6, hc_eps=1e-6, digits=50):
    """Evaluate the forward in ``decimal`` arithmetic.

    x_vals: float array [T, n, D] of the (already bf16-exact) input values.
    Written independently of the C oracle: phi is cut into its pre / post /
    res row blocks first ("phi split along rows into three segments", Sinkhorn
    page §3.1); the Sinkhorn output is formed as diag(r) E diag(c) -- running
    row and column scale vectors applied to the exponentiated logits -- rather
    than by normalising a matrix in place.  Returns a dict of float lists.
    """
    D_ = decimal.Decimal
    ctx = decimal.Context(prec=digits)
    x_vals = np.asarray(x_vals, dtype=np.float64)
    T, n, D = x_vals.shape
    K = n * D
    alpha = [D_(float(a)) for a in np.asarray(alpha, dtype=np.float32)]
    two_gate = len(alpha) == 2
    phi = np.asarray(phi, dtype=np.float32).reshape(-1, K)
    bias = [D_(float(b)) for b in np.asarray(bias, dtype=np.float32).reshape(-1)]
    eps_h = D_(hc_eps)
    eps_n = D_(norm_eps)
    gam = None if gamma is None else [D_(float(v)) for v in np.asarray(gamma, np.float32).reshape(-1)]
    one = D_(1)

    def sig(z):
        return one / (one + ctx.exp(-z))

    seg_pre = phi[0:n]
    seg_post = phi[n:2 * n]
    seg_res = None if two_gate else phi[2 * n:2 * n + n * n]
    out = {k: [] for k in ("y", "h_pre", "h_post", "h_res", "inv_rms", "h_mix")}
    for t in range(T):
        flat = [D_(float(v)) for v in x_vals[t].reshape(-1)]
        ms = ctx.divide(sum((ctx.multiply(v, v) for v in flat), D_(0)), D_(K))
        r = one / ctx.sqrt(ms + eps_n)
        xg = flat if gam is None else [ctx.multiply(a, b) for a, b in zip(flat, gam)]

        def proj(rows):
            return [sum((ctx.multiply(xg[k], D_(float(row[k]))) for k in range(K)), D_(0))
                    for row in rows]

        mix_pre, mix_post = proj(seg_pre), proj(seg_post)
        mix_res = [] if two_gate else proj(seg_res)
        out["h_mix"].append([float(v) for v in mix_pre + mix_post + mix_res])
        out["inv_rms"].append(float(r))
        hp = [sig(alpha[0] * (m * r) + bias[i]) + eps_h for i, m in enumerate(mix_pre)]
        hq = [2 * sig(alpha[1] * (m * r) + bias[n + i]) + (eps_h if two_gate else 0)
              for i, m in enumerate(mix_post)]
        out["h_pre"].append([float(v) for v in hp])
        out["h_post"].append([float(v) for v in hq])
        if two_gate:
            out["h_res"].append([[0.0] * n for _ in range(n)])
        else:
            L = [[alpha[2] * (mix_res[i * n + j] * r) + bias[2 * n + i * n + j]
                  for j in range(n)] for i in range(n)]
            # Softmax rows, plus eps; from then on keep E fixed and carry the
            # scalings: M = diag(rs) E' diag(cs) with E' = softmax + eps.
            E = []
            for i in range(n):
                mx = max(L[i])
                ex = [ctx.exp(v - mx) for v in L[i]]
                s = sum(ex, D_(0))
                E.append([e / s + eps_h for e in ex])
            rs = [one] * n
            cs = [one] * n

            def entry(i, j):
                return rs[i] * E[i][j] * cs[j]

            for it in range(num_iters):
                if it > 0:  # row pass (the softmax stands in for the first one)
                    sums = [sum((entry(i, j) for j in range(n)), D_(0)) + eps_h for i in range(n)]
                    rs = [rs[i] / sums[i] for i in range(n)]
                sums = [sum((entry(i, j) for i in range(n)), D_(0)) + eps_h for j in range(n)]
                cs = [cs[j] / sums[j] for j in range(n)]
            out["h_res"].append([[float(entry(i, j)) for j in range(n)] for i in range(n)])
        w = hp if pre_mix is None else [D_(float(v)) for v in np.asarray(pre_mix, np.float32)[t]]
        out["y"].append([float(sum((w[i] * flat[i * D + d] for i in range(n)), D_(0)))
                         for d in range(D)])
    return out
