"""Pins of the backward oracle (``oracle.run_backward``) against what the
mathematics fixes, independently of the oracle's own stages.

The backward page defines every output as a gradient of the forward
("MhcPreBackward 反向梯度算子实现与 aclnn 调用指南" §一).  So the pin is automatic
differentiation (torch, float64, CPU) of a loss built on a forward written
here in tensor form -- one matmul for the projection, ``torch.softmax`` and
whole-matrix divisions for Sinkhorn -- after that forward has been checked
against the C forward oracle on the same inputs.  Any dropped term, wrong
sign, transposed index or wrong Sinkhorn step in the stage-by-stage oracle
shows up as a mismatch here.  Further pins: the logit form of grad_h_res,
grad_x_post passing straight through, zero upstream gradients, token and
column selection, thread-count independence.
"""
import numpy as np
import pytest
import torch

import oracle


def _bf16_bits(a):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _bits_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(T, n, D, seed, with_gamma=True, num_iters=20):
    rng = np.random.default_rng(seed)
    K, R = n * D, n * n + 2 * n
    c = {
        "x": _bf16_bits(rng.standard_normal((T, n, D))),
        "phi": (rng.standard_normal((R, K)) / np.sqrt(K)).astype(np.float32),
        "alpha": rng.uniform(0.5, 1.5, 3).astype(np.float32),
        "bias": (0.1 * rng.standard_normal(R)).astype(np.float32),
        "gamma": (1 + 0.05 * rng.standard_normal((n, D))).astype(np.float32) if with_gamma else None,
        "g_in": _bf16_bits(rng.standard_normal((T, D))),
        "g_post": rng.standard_normal((T, n)),
        "g_res": rng.standard_normal((T, n, n)),
        "g_xp": _bf16_bits(rng.standard_normal((T, n, D))),
        "num_iters": num_iters,
    }
    return c


def _torch_forward(x, phi, alpha, bias, gamma, num_iters, norm_eps=1e-6, hc_eps=1e-6):
    """The forward in tensor form: returns y, hPost, comb, hPre, invRms, hMix
    and the res logits H."""
    T, n, D = x.shape
    flat = x.reshape(T, n * D)
    inv = torch.rsqrt((flat * flat).mean(dim=1) + norm_eps)
    xg = flat if gamma is None else flat * gamma.reshape(1, -1)
    hmix = xg @ phi.T
    w = hmix * inv[:, None]
    pre = torch.sigmoid(alpha[0] * w[:, :n] + bias[:n]) + hc_eps
    post = 2.0 * torch.sigmoid(alpha[1] * w[:, n:2 * n] + bias[n:2 * n])
    H = (alpha[2] * w[:, 2 * n:] + bias[2 * n:]).reshape(T, n, n)
    P = torch.softmax(H, dim=-1) + hc_eps
    P = P / (P.sum(dim=1, keepdim=True) + hc_eps)
    for _ in range(num_iters - 1):
        P = P / (P.sum(dim=2, keepdim=True) + hc_eps)
        P = P / (P.sum(dim=1, keepdim=True) + hc_eps)
    y = (pre[:, :, None] * x).sum(dim=1)
    return y, post, P, pre, inv, hmix, H


def _autograd(c, logit_form=False):
    f = lambda a: torch.tensor(np.asarray(a, dtype=np.float64), requires_grad=True)
    x = f(_bits_to_f64(c["x"]))
    phi, alpha, bias = f(c["phi"]), f(c["alpha"]), f(c["bias"])
    gamma = None if c["gamma"] is None else f(c["gamma"])
    y, post, comb, pre, inv, hmix, H = _torch_forward(x, phi, alpha, bias, gamma, c["num_iters"])
    g_in = torch.from_numpy(_bits_to_f64(c["g_in"]))
    loss = (g_in * y).sum() + (torch.from_numpy(c["g_post"]) * post).sum()
    loss = loss + (torch.from_numpy(c["g_res"]) * (H if logit_form else comb)).sum()
    loss.backward()
    out = {"x": x.grad.numpy(), "phi": phi.grad.numpy(), "alpha": alpha.grad.numpy(),
           "bias": bias.grad.numpy()}
    if gamma is not None:
        out["gamma"] = gamma.grad.numpy().reshape(-1)
    fwd = {k: v.detach().numpy() for k, v in
           zip(("y", "h_post", "h_res", "h_pre", "inv_rms", "h_mix"), (y, post, comb, pre, inv, hmix))}
    return out, fwd


def _oracle_backward(c, logit_form=False, g_xp=False, threads=None, **kw):
    fw = oracle.run(c["x"], c["phi"], c["alpha"], c["bias"], c["gamma"], num_iters=c["num_iters"])
    return oracle.run_backward(
        c["x"], c["phi"], c["alpha"], c["gamma"], c["g_in"], c["g_post"], c["g_res"],
        fw.inv_rms, fw.h_mix, fw.h_pre, fw.h_post,
        None if logit_form else fw.sum_out, None if logit_form else fw.norm_out,
        c["g_xp"] if g_xp else None, num_iters=c["num_iters"], threads=threads, **kw), fw


def _close(got, want, scale, rel=1e-10):
    got, want, scale = map(np.asarray, (got, want, scale))
    bad = np.abs(got - want) > rel * (np.abs(scale) + np.abs(want)) + 1e-13
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], want[bad][:5])


@pytest.mark.parametrize("with_gamma", [False, True])
@pytest.mark.parametrize("num_iters", [1, 2, 20])
def test_matches_autograd(with_gamma, num_iters):
    c = _case(3, 4, 8, seed=10 + num_iters, with_gamma=with_gamma, num_iters=num_iters)
    want, fwd = _autograd(c)
    got, fw = _oracle_backward(c)
    # the tensor-form forward is the C forward oracle's function
    assert np.allclose(fwd["h_res"], fw.h_res, rtol=0, atol=1e-13)
    assert np.allclose(fwd["h_mix"], fw.h_mix, rtol=0, atol=1e-13)
    assert np.allclose(fwd["y"], fw.y, rtol=0, atol=1e-12)
    _close(got.grad_x, want["x"], got.grad_x_abs)
    _close(got.grad_phi, want["phi"], got.grad_phi_abs)
    _close(got.grad_alpha, want["alpha"], got.grad_alpha_abs)
    _close(got.grad_bias, want["bias"], got.grad_bias_abs)
    if with_gamma:
        _close(got.grad_gamma, want["gamma"], got.grad_gamma_abs)
    else:
        assert got.grad_gamma is None


@pytest.mark.parametrize("n", [6, 8])
def test_matches_autograd_wider(n):
    c = _case(2, n, 4, seed=n, num_iters=3)
    want, _ = _autograd(c)
    got, _ = _oracle_backward(c)
    _close(got.grad_x, want["x"], got.grad_x_abs)
    _close(got.grad_phi, want["phi"], got.grad_phi_abs)
    _close(got.grad_gamma, want["gamma"], got.grad_gamma_abs)
    _close(got.grad_bias, want["bias"], got.grad_bias_abs)
    _close(got.grad_alpha, want["alpha"], got.grad_alpha_abs)


def test_logit_form_of_grad_h_res():
    """Without sum_out / norm_out, grad_h_res is the gradient of the res
    logits and no Sinkhorn backward runs."""
    c = _case(3, 4, 8, seed=3)
    want, _ = _autograd(c, logit_form=True)
    got, _ = _oracle_backward(c, logit_form=True)
    _close(got.grad_x, want["x"], got.grad_x_abs)
    _close(got.grad_phi, want["phi"], got.grad_phi_abs)
    _close(got.grad_bias, want["bias"], got.grad_bias_abs)
    _close(got.grad_alpha, want["alpha"], got.grad_alpha_abs)


def test_sinkhorn_changes_the_res_gradient():
    """The Sinkhorn backward is not the identity: the two forms differ."""
    c = _case(2, 4, 8, seed=4)
    a, _ = _oracle_backward(c)
    b, _ = _oracle_backward(c, logit_form=True)
    assert np.abs(a.grad_bias[8:] - b.grad_bias[8:]).max() > 1e-3
    assert np.array_equal(a.grad_bias[:8], b.grad_bias[:8])


def test_grad_x_post_adds_through():
    c = _case(3, 4, 16, seed=5)
    a, _ = _oracle_backward(c)
    b, _ = _oracle_backward(c, g_xp=True)
    assert np.allclose(b.grad_x - a.grad_x, _bits_to_f64(c["g_xp"]), rtol=0, atol=1e-14)
    assert np.array_equal(a.grad_phi, b.grad_phi)
    assert np.array_equal(a.grad_alpha, b.grad_alpha)


def test_zero_upstream_gradient():
    c = _case(2, 4, 8, seed=6)
    c["g_in"] = np.zeros_like(c["g_in"])
    c["g_post"] = np.zeros_like(c["g_post"])
    c["g_res"] = np.zeros_like(c["g_res"])
    got, _ = _oracle_backward(c)
    for a in (got.grad_x, got.grad_phi, got.grad_gamma, got.grad_alpha, got.grad_bias):
        assert not np.any(a)


def test_selection_and_threads():
    c = _case(9, 4, 16, seed=7)
    full, _ = _oracle_backward(c, threads=1)
    many, _ = _oracle_backward(c, threads=5)
    for f in ("grad_x", "grad_phi", "grad_gamma", "grad_alpha", "grad_bias", "grad_phi_abs"):
        assert np.array_equal(getattr(full, f), getattr(many, f)), f
    toks, cols = [7, 0, 7, 3], [63, 1, 17]
    sel, _ = _oracle_backward(c, tokens=toks, columns=cols)
    assert np.array_equal(sel.grad_x, full.grad_x[toks])
    assert np.array_equal(sel.grad_phi, full.grad_phi[:, cols])
    assert np.array_equal(sel.grad_gamma, full.grad_gamma[cols])
    assert np.array_equal(sel.grad_bias, full.grad_bias)
