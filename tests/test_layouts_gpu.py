"""Batch-consistent mode and the BSND layout, through the C ABI.

* Batch consistency (the Sinkhorn page's §8.1, off by default): with
  batch_consistent = 1 every token's outputs are bitwise the same whatever
  batch it is part of -- checked on prefixes and slices of one batch, at
  sizes that make the default mode pick different cluster sizes -- and they
  still match the oracle (the tolerances of tests/gpu_helpers.py).
* BSND: x [B, S, n, D] (contiguous) is the same memory as [B*S, n, D]; the
  forward, the backward and hc_post on the 4-D views give bitwise the same
  results as on the 3-D tensors, shaped by (B, S).
"""
import numpy as np
import pytest
import torch

from mhc_synth import make_bwd_grads, make_case, make_post_case
from gpu_helpers import compare, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mhc_hyper_connection_gb300 import build
    build.build()


def _fwd(case, x, consistent, lead=None):
    from mhc_hyper_connection_gb300 import MhcPre
    op = MhcPre(case.n, case.D, num_iters=case.num_iters, impl_mode=case.impl_mode, need_backward=True,
                batch_consistent=consistent)
    out = op.allocate(lead if lead is not None else x.shape[0], x.device)
    op.run(x, case.phi, case.alpha, case.bias, out, gamma=case.gamma)
    torch.cuda.synchronize()
    assert op.status(out) == 0
    return op, out


KEYS = ("y", "h_post", "h_res", "h_pre", "inv_rms", "h_mix")


@pytest.mark.parametrize("D", [256, 7168])
def test_batch_consistent_tokens_do_not_depend_on_the_batch(cuda_device, D):
    case = make_case("training", device=cuda_device, T=1100, D=D, seed=D, need_backward=True)
    _, full = _fwd(case, case.x, True)
    for lo, hi in [(0, 1), (0, 37), (0, 64), (0, 300), (500, 564), (1099, 1100)]:
        _, part = _fwd(case, case.x[lo:hi].contiguous(), True)
        for k in KEYS:
            assert torch.equal(part[k], full[k][lo:hi]), (k, lo, hi)
        for k in ("sum_out", "norm_out"):
            assert torch.equal(part[k], full[k][:, lo:hi]), (k, lo, hi)
    ref = run_oracle(case)
    compare(case, full, ref)


def test_bsnd_forward_backward_post(cuda_device):
    from mhc_hyper_connection_gb300 import MhcPre, hc_post
    B, S, D = 3, 50, 512
    case = make_case("training", device=cuda_device, T=B * S, D=D, seed=9, need_backward=True)
    op, flat = _fwd(case, case.x, False)
    _, bsnd = _fwd(case, case.x.view(B, S, case.n, D), False, lead=(B, S))
    assert bsnd["y"].shape == (B, S, D) and bsnd["h_res"].shape == (B, S, case.n, case.n)
    assert bsnd["norm_out"].shape == (40, B, S, case.n, case.n)
    for k in KEYS + ("sum_out", "norm_out"):
        assert torch.equal(bsnd[k].reshape(flat[k].shape), flat[k]), k
    # backward on the BSND views
    g = make_bwd_grads(device=cuda_device, T=B * S, n=case.n, D=D, seed=9)
    saved = {k: flat[k] for k in ("inv_rms", "h_mix", "h_pre", "h_post", "sum_out", "norm_out")}
    gf = op.allocate_backward(B * S, cuda_device, gamma=True)
    op.backward(case.x, case.phi, case.alpha, case.gamma, g.g_in, g.g_post, g.g_res, saved, gf)
    saved4 = {k: bsnd[k] for k in saved}
    gb = op.allocate_backward((B, S), cuda_device, gamma=True)
    op.backward(case.x.view(B, S, case.n, D), case.phi, case.alpha, case.gamma, g.g_in.view(B, S, D),
                g.g_post.view(B, S, case.n), g.g_res.view(B, S, case.n, case.n), saved4, gb)
    torch.cuda.synchronize()
    assert gb["grad_x"].shape == (B, S, case.n, D)
    for k in ("grad_x", "grad_phi", "grad_alpha", "grad_bias", "grad_gamma"):
        assert torch.equal(gb[k].reshape(gf[k].shape), gf[k]), k
    # hc_post on BSND
    pc = make_post_case(device=cuda_device, T=B * S, n=case.n, D=D, seed=2)
    o3 = hc_post(pc.x, pc.residual, pc.post, pc.comb)
    o4 = hc_post(pc.x.view(B, S, D), pc.residual.view(B, S, case.n, D), pc.post.view(B, S, case.n),
                 pc.comb.view(B, S, case.n, case.n))
    torch.cuda.synchronize()
    assert o4.shape == (B, S, case.n, D) and torch.equal(o4.reshape(o3.shape), o3)
