"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs, and compare within the stated
tolerances.

Reference: the oracle in the handle's precision mode -- the exact projection
in fp32 mode; in tf32 mode the HcPre page's HF32 simulation (its 精度验证
method: an fp32 golden whose matmul operands are truncated to HF32), applied
to the folded weight gamma (.) phi as the library does (oracle hf32=2;
without gamma it is the page's own operand-wise simulation).

Tolerances (against that reference):
  * hPre, hPost, comb: max |err| <= 1e-4 in both modes; in tf32 mode the
    gates are also held to 3e-3 against the exact oracle (check_tf32_exact);
  * y (bf16 or fp16): |err| <= 2^-7 |ref| + 1e-3 elementwise, both modes, no
    other term;
  * intermediates: invRms rel 1e-4; hMix |err| <= 2e-4 (1 + |ref|) -- fp32
    accumulation over n*D products; sumOut rel 1e-4; normOut 1e-4.
    The invRms bound: Sigma x^2 is accumulated in fp32, each token's squares
    split over 2 C partial sums (C = cluster size, two halves of the
    streams per member) of 8 running sums each, so a running sum takes
    n*D/(16 C) additions; with each addition off by at most an ulp (2^-23)
    in the same direction the total is off by at most (n*D/(16 C)) 2^-23
    -- 1.07e-4 at n*D = 28672, C = 2 -- and invRms by half of that, 5.3e-5
    (measured up to 2.6e-5).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mhc_hyper_connection_gb300 import MhcPre

TOL = {0: 1e-4, 1: 3e-3}     # gates against the exact oracle, per mode
TOL_MODE = 1e-4               # gates against the oracle in the handle's own mode


def make_op(case, **launch):
    """A handle for the case's shape and mode; launch-choice keywords (kernel,
    cluster, ...) force a kernel or launch shape."""
    from mhc_hyper_connection_gb300 import MHC_DTYPE_BF16, MHC_DTYPE_FP16
    return MhcPre(case.n, case.D, alpha_len=case.alpha_len, num_iters=case.num_iters,
                  norm_eps=case.norm_eps, hc_eps=case.hc_eps, impl_mode=case.impl_mode,
                  need_backward=case.need_backward,
                  x_dtype=MHC_DTYPE_FP16 if case.x.dtype == torch.float16 else MHC_DTYPE_BF16, **launch)


def run_cuda(case, stream=None, out=None, op=None, **launch):
    op = op or make_op(case, **launch)
    if out is None:
        out = op.allocate(case.T, case.x.device)
    op.run(case.x, case.phi, case.alpha, case.bias, out, gamma=case.gamma,
           pre_mix=case.pre_mix, stream=stream)
    st = op.status(out)
    assert st == 0, f"device status {st}"
    return op, out


def x_bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def run_oracle(case, tokens=None, hf32=None):
    """The oracle on the case's inputs (optionally only `tokens`); hf32=None
    picks the handle's mode: exact for fp32 mode, the folded HF32 simulation
    for tf32 mode."""
    if hf32 is None:
        hf32 = 2 if case.impl_mode == 1 else 0
    x = case.x if tokens is None else case.x[torch.as_tensor(tokens, device=case.x.device)]
    pm = None
    if case.pre_mix is not None:
        pm = case.pre_mix if tokens is None else case.pre_mix[torch.as_tensor(tokens, device=case.pre_mix.device)]
        pm = pm.cpu().numpy()
    return oracle.run(x_bits(x), case.phi.cpu().numpy(), case.alpha.cpu().numpy(),
                      case.bias.cpu().numpy(),
                      None if case.gamma is None else case.gamma.cpu().numpy(), pm,
                      num_iters=case.num_iters, norm_eps=case.norm_eps, hc_eps=case.hc_eps,
                      hf32=hf32, backward=case.need_backward, x_fp16=case.x.dtype == torch.float16)


def _sel(t, tokens, axis=0):
    a = t.float().cpu().numpy() if isinstance(t, torch.Tensor) else t
    if tokens is None:
        return a
    return np.take(a, tokens, axis=axis)


def compare(case, out, ref, tokens=None, tol=None, check_intermediates=True, exact_check=True):
    """Assert the CUDA outputs match the oracle `ref` (run in the handle's
    mode, see run_oracle); in tf32 mode also the gates against the exact
    oracle (exact_check).  Returns a dict of max errors."""
    tol = TOL_MODE if tol is None else tol
    errs = {}
    gp = _sel(out["h_post"], tokens)
    errs["h_post"] = float(np.abs(gp - ref.h_post).max())
    if out.get("h_pre") is not None:
        errs["h_pre"] = float(np.abs(_sel(out["h_pre"], tokens) - ref.h_pre).max())
    if out.get("h_res") is not None:
        errs["comb"] = float(np.abs(_sel(out["h_res"], tokens) - ref.h_res).max())
    for k in ("h_post", "h_pre", "comb"):
        if k in errs:
            assert errs[k] <= tol, f"{case.name}: {k} max err {errs[k]:.3g} > {tol}"
    y = _sel(out["y"], tokens).astype(np.float64)
    bad = np.abs(y - ref.y) > 2.0 ** -7 * np.abs(ref.y) + 1e-3
    errs["y_viol"] = int(bad.sum())
    errs["y"] = float(np.abs(y - ref.y).max())
    assert not bad.any(), (f"{case.name}: {bad.sum()} y elements outside 2^-7|ref|+1e-3, "
                           f"max err {errs['y']:.3g}")
    if case.need_backward and check_intermediates:
        ir = _sel(out["inv_rms"], tokens)
        errs["inv_rms"] = float(np.abs(ir / ref.inv_rms - 1).max())
        assert errs["inv_rms"] <= 1e-4, errs
        hm = _sel(out["h_mix"], tokens)
        errs["h_mix"] = float((np.abs(hm - ref.h_mix) / (1 + np.abs(ref.h_mix))).max())
        assert errs["h_mix"] <= 2e-4, errs
        if case.alpha_len == 3:
            so = _sel(out["sum_out"], tokens, axis=1)
            no = _sel(out["norm_out"], tokens, axis=1)
            errs["sum_out"] = float((np.abs(so - ref.sum_out) / np.abs(ref.sum_out)).max())
            errs["norm_out"] = float(np.abs(no - ref.norm_out).max())
            assert errs["sum_out"] <= 1e-4 and errs["norm_out"] <= 1e-4, errs
    if case.impl_mode == 1 and exact_check:
        errs.update(check_tf32_exact(case, out, tokens))
    return errs


def check_tf32_exact(case, out, tokens=None):
    """tf32 mode: the gates within 3e-3 of the exact (fp32-mode) oracle."""
    ref = run_oracle(case, tokens, hf32=0)
    errs = {}
    for k, r in (("h_post", ref.h_post), ("h_pre", ref.h_pre), ("h_res", ref.h_res)):
        if out.get(k) is None:
            continue
        e = float(np.abs(_sel(out[k], tokens) - r).max())
        errs[k + "_vs_exact"] = e
        assert e <= TOL[1], f"{case.name}: tf32 {k} vs exact oracle {e:.3g} > {TOL[1]}"
    return errs
