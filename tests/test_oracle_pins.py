"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every test here runs on the CPU.  Each one would fail under a plausible slip
in the oracle: a dropped eps, the softmax over the wrong axis, the Sinkhorn
steps in the wrong order, a transposed phi, the RMS mean over D instead of
n*D, gamma applied to the RMS, segments read in the wrong order, y built
from gamma-scaled x, pre_mix ignored, hcEps missing on the two-gate hPost.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from mhc_synth import make_case, normal, stream_key, to_bf16_bits, bf16_bits_to_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
EPS = 1e-6


def sig(z):
    return 1.0 / (1.0 + np.exp(-z))


def rand_inputs(T, n, D, alpha_len=3, seed=3, phi_scale=None, gamma=False, pre_mix=False):
    R = n * n + 2 * n if alpha_len == 3 else 2 * n
    K = n * D
    x = to_bf16_bits(normal(stream_key(seed, "x"), T * K)).reshape(T, n, D)
    scale = phi_scale if phi_scale is not None else 1.0 / math.sqrt(K)
    phi = normal(stream_key(seed, "phi"), R * K, std=scale).astype(np.float32).reshape(R, K)
    alpha = np.array([0.8, 1.3, 0.9][:alpha_len], dtype=np.float32)
    bias = normal(stream_key(seed, "bias"), R, std=0.3).astype(np.float32)
    g = normal(stream_key(seed, "gamma"), K, 0.2, 1.0).astype(np.float32).reshape(n, D) if gamma else None
    pm = (np.abs(normal(stream_key(seed, "pre_mix"), T * n)).astype(np.float32).reshape(T, n)
          if pre_mix else None)
    return x, phi, alpha, bias, g, pm


def xval(x_bits):
    return bf16_bits_to_f32(x_bits).astype(np.float64)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("D", [1, 2, 4])
@pytest.mark.parametrize("variant", ["plain", "gamma", "pre_mix", "two_gate"])
@pytest.mark.parametrize("iters", [1, 2, 20])
def test_decimal_brute_force_agrees(D, variant, iters):
    n, T = 4, 3
    alpha_len = 2 if variant == "two_gate" else 3
    x, phi, alpha, bias, g, pm = rand_inputs(T, n, D, alpha_len, seed=D * 7 + iters,
                                             gamma=variant == "gamma",
                                             pre_mix=variant == "pre_mix", phi_scale=0.7)
    o = oracle.run(x, phi, alpha, bias, g, pm, num_iters=iters)
    b = oracle.brute_force_decimal(xval(x), phi, alpha, bias, g, pm, num_iters=iters)
    for key in ("y", "h_pre", "h_post", "h_res", "inv_rms", "h_mix"):
        got = getattr(o, key)
        ref = np.asarray(b[key], dtype=np.float64).reshape(got.shape)
        np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12, err_msg=key)


# ----------------------------------------------------------- closed forms

def test_alpha_zero_closed_form():
    """alpha = 0: the gates see the bias alone, whatever x and phi are."""
    T, n, D = 5, 4, 32
    x, phi, _, bias, _, _ = rand_inputs(T, n, D)
    alpha = np.zeros(3, dtype=np.float32)
    o = oracle.run(x, phi, alpha, bias)
    b = bias.astype(np.float64)
    np.testing.assert_allclose(o.h_pre, np.tile(sig(b[:n]) + EPS, (T, 1)), rtol=0, atol=1e-15)
    np.testing.assert_allclose(o.h_post, np.tile(2 * sig(b[n:2 * n]), (T, 1)), rtol=0, atol=1e-15)
    # comb is the same matrix for every token.
    assert np.all(o.h_res == o.h_res[0:1])
    # y is the weighted sum of raw x with those constant weights.
    y = np.einsum("tid,i->td", xval(x), sig(b[:n]) + EPS)
    np.testing.assert_allclose(o.y, y, rtol=1e-14, atol=1e-14)


def test_two_gate_variant():
    """alpha of length 2: no residual path, hPost picks up hcEps."""
    T, n, D = 4, 4, 16
    x, phi, alpha, bias, _, _ = rand_inputs(T, n, D, alpha_len=2)
    o = oracle.run(x, phi, alpha, bias)
    assert o.h_mix.shape == (T, 2 * n)
    assert np.all(o.h_res == 0.0)
    assert o.sum_out is None
    w = o.h_mix * o.inv_rms[:, None]
    np.testing.assert_allclose(o.h_post, 2 * sig(alpha[1] * w[:, n:] + bias[n:]) + EPS,
                               rtol=1e-14)
    z = oracle.run(x, phi, np.zeros(2, np.float32), bias)
    np.testing.assert_allclose(z.h_post, np.tile(2 * sig(bias[n:].astype(np.float64)) + EPS,
                                                 (T, 1)), rtol=0, atol=1e-15)


def _uniform_scalar_map(n, iters, eps):
    a = 1.0 / n + eps            # softmax of equal logits, plus eps
    a = a / (n * a + eps)        # first column step
    for _ in range(iters - 1):
        a = a / (n * a + eps)    # row step
        a = a / (n * a + eps)    # column step
    return a


@pytest.mark.parametrize("n", [4, 6, 8])
def test_uniform_logits_reduce_to_scalar_map(n):
    """Equal residual logits: every entry follows a <- a/(n a + eps) and tends
    to the fixed point (1 - eps)/n."""
    T, D = 3, 8
    x, phi, alpha, bias, _, _ = rand_inputs(T, n, D)
    alpha[2] = 0.0
    bias[2 * n:] = 0.37
    o = oracle.run(x, phi, alpha, bias)
    a = _uniform_scalar_map(n, 20, EPS)
    np.testing.assert_allclose(o.h_res, np.full((T, n, n), a), rtol=0, atol=1e-16)
    assert abs(a - (1 - EPS) / n) < 1e-15
    if n == 4:
        assert a == pytest.approx(0.24999975000000002, abs=1e-17)


def test_hand_built_softmax_and_first_column_step():
    """phi = 0 makes w = 0, so the logits are the bias block as given.
    Row 0 = [0, ln2, ln3, ln4] has softmax [1,2,3,4]/10 (rows, not columns)."""
    n, D, T = 4, 4, 1
    x = to_bf16_bits(np.ones(n * D)).reshape(1, n, D)
    phi = np.zeros((24, n * D), np.float32)
    alpha = np.array([1, 1, 1], np.float32)
    H = np.array([[0, math.log(2), math.log(3), math.log(4)],
                  [1.0, 1.0, 1.0, 1.0],
                  [0.0, 0.0, 0.0, 2.0],
                  [-1.0, 0.0, 1.0, 0.5]])
    bias = np.zeros(24, np.float32)
    bias[8:] = H.reshape(-1).astype(np.float32)
    Hf = bias[8:].astype(np.float64).reshape(n, n)
    o = oracle.run(x, phi, alpha, bias, num_iters=2)
    # normOut[0]: softmax along each row, plus eps.
    E = np.exp(Hf - Hf.max(axis=1, keepdims=True))
    sm = E / E.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(o.norm_out[0, 0], sm + EPS, rtol=1e-15)
    assert o.norm_out[0, 0, 0, 1] == pytest.approx(0.2 + EPS, rel=1e-7)   # 2/10 (+eps)
    np.testing.assert_allclose(o.sum_out[0, 0], E.sum(axis=1), rtol=1e-15)
    # step 1 divides by column sums + eps.
    c = (sm + EPS).sum(axis=0) + EPS
    np.testing.assert_allclose(o.sum_out[1, 0], c, rtol=1e-15)
    np.testing.assert_allclose(o.norm_out[1, 0], (sm + EPS) / c[None, :], rtol=1e-15)
    # step 2 divides by row sums + eps.
    P1 = (sm + EPS) / c[None, :]
    r = P1.sum(axis=1) + EPS
    np.testing.assert_allclose(o.norm_out[2, 0], P1 / r[:, None], rtol=1e-14)
    # the output is the last column step.
    np.testing.assert_array_equal(o.h_res[0], o.norm_out[3, 0])


def test_final_column_sums_identity_and_row_convergence():
    """After the last column step, column j sums to S_j/(S_j + eps), S_j the
    pre-step column sum (exact identity, any logits).  At the workloads' logit
    scale (phi std 1/sqrt(nD)) S_j is near 1 after 20 iterations, so column
    sums are 1 within 1e-6; row sums approach 1 monotonically as iterations
    grow."""
    T, n, D = 6, 4, 32
    x, phi, alpha, bias, _, _ = rand_inputs(T, n, D, phi_scale=0.5)   # peaked logits
    for iters in (1, 3, 20):
        o = oracle.run(x, phi, alpha, bias, num_iters=iters)
        S = o.sum_out[2 * iters - 1] - EPS
        np.testing.assert_allclose(o.h_res.sum(axis=1), S / (S + EPS), rtol=0, atol=1e-13)
    x, phi, alpha, bias, _, _ = rand_inputs(T, n, D)
    prev = None
    for iters in (1, 2, 5, 20, 60):
        o = oracle.run(x, phi, alpha, bias, num_iters=iters)
        dev = np.abs(o.h_res.sum(axis=2) - 1.0).max()
        if prev is not None:
            assert dev <= prev + 1e-12
        prev = dev
        if iters >= 20:   # eps/(S+eps) with S within 1e-3 of 1
            assert np.all(np.abs(o.h_res.sum(axis=1) - 1.0) <= 1.001e-6)
    assert prev < 1e-5


def test_rms_mean_over_all_streams():
    """Constant x per stream: invRms = 1/sqrt(mean_i c_i^2 + eps), a mean over
    n*D elements, not D."""
    n, D = 4, 16
    c = np.array([1.0, 2.0, 0.5, 4.0])
    x = to_bf16_bits(np.repeat(c, D)).reshape(1, n, D)
    _, phi, alpha, bias, _, _ = rand_inputs(1, n, D)
    o = oracle.run(x, phi, alpha, bias)
    assert o.inv_rms[0] == pytest.approx(1 / math.sqrt(np.mean(c ** 2) + EPS), rel=1e-15)


def test_gamma_scales_projection_not_rms_or_y():
    """gamma = 2 doubles hMix, leaves invRms and the y weights' source x alone."""
    T, n, D = 3, 4, 8
    x, phi, alpha, bias, _, _ = rand_inputs(T, n, D)
    g = np.full((n, D), 2.0, np.float32)
    a = oracle.run(x, phi, alpha, bias, g)
    b = oracle.run(x, (phi * 2).astype(np.float32), alpha, bias)
    np.testing.assert_allclose(a.h_mix, b.h_mix, rtol=1e-15)
    np.testing.assert_array_equal(a.inv_rms, b.inv_rms)
    np.testing.assert_allclose(a.y, b.y, rtol=1e-15)
    y = np.einsum("tid,ti->td", xval(x), a.h_pre)
    np.testing.assert_allclose(a.y, y, rtol=1e-14)


def test_segment_order_pre_post_res():
    """Only the post rows of phi non-zero: hPre and comb see the bias alone."""
    T, n, D = 3, 4, 8
    x, phi, alpha, bias, _, _ = rand_inputs(T, n, D, phi_scale=0.5)
    phi[:n] = 0
    phi[2 * n:] = 0
    o = oracle.run(x, phi, alpha, bias)
    np.testing.assert_allclose(o.h_pre, np.tile(sig(bias[:n].astype(np.float64)) + EPS, (T, 1)),
                               atol=1e-15)
    assert np.all(o.h_res == o.h_res[0:1])
    assert np.ptp(o.h_post, axis=0).max() > 1e-3
    # phi row r pairs with x element k of the flattened [n, D] token (no transpose).
    r, k = n + 1, 3 * D + 5
    phi2 = np.zeros_like(phi)
    phi2[r, k] = 1.0
    o2 = oracle.run(x, phi2, alpha, bias)
    assert o2.h_mix[1, r] == xval(x)[1].reshape(-1)[k]
    assert np.count_nonzero(o2.h_mix[1]) == (1 if xval(x)[1].reshape(-1)[k] != 0 else 0)


def test_pre_mix_replaces_weights():
    T, n, D = 4, 8, 8
    x, phi, alpha, bias, _, pm = rand_inputs(T, n, D, pre_mix=True)
    o = oracle.run(x, phi, alpha, bias, None, pm)
    plain = oracle.run(x, phi, alpha, bias)
    np.testing.assert_allclose(o.y, np.einsum("tid,ti->td", xval(x), pm.astype(np.float64)),
                               rtol=1e-14)
    np.testing.assert_array_equal(o.h_pre, plain.h_pre)    # hc_pre is still returned
    assert np.abs(o.y - plain.y).max() > 1e-3


def test_all_ones_example():
    """The MhcPreV2 page's worked call (§九: x = phi = alpha = bias = gamma = 1,
    n = 4, D = 2560) in closed form; tokens are identical so T is cut to 2."""
    with open(os.path.join(GOLDEN, "mhc_pre_v2_all_ones_example.json")) as f:
        ex = json.load(f)
    n, D, T = ex["n"], ex["D"], 2
    K = n * D
    x = to_bf16_bits(np.ones(T * K)).reshape(T, n, D)
    R = n * n + 2 * n
    o = oracle.run(x, np.ones((R, K), np.float32), np.ones(3, np.float32),
                   np.ones(R, np.float32), np.ones((n, D), np.float32))
    inv = 1 / math.sqrt(1 + EPS)
    np.testing.assert_allclose(o.inv_rms, inv, rtol=1e-15)
    np.testing.assert_allclose(o.h_mix, float(K), rtol=0)
    np.testing.assert_allclose(o.h_pre, 1 + EPS, rtol=1e-15)          # sigmoid saturates
    np.testing.assert_allclose(o.h_post, 2.0, rtol=1e-15)
    np.testing.assert_allclose(o.h_res, _uniform_scalar_map(n, 20, EPS), rtol=1e-14)
    np.testing.assert_allclose(o.y, n * (1 + EPS), rtol=1e-15)
    assert ex["expected_y_bf16"] == 4.0


def test_stable_inputs_example():
    """The Sinkhorn page's stable inputs (phi = 1/sqrt(nD), alpha = 0.25,
    bias = 0): every projection row equals sum(x)/sqrt(nD), so all hPre_i
    agree and comb is exactly the uniform scalar map."""
    T, n, D = 3, 4, 64
    K = n * D
    x, _, _, _, _, _ = rand_inputs(T, n, D)
    phi = np.full((24, K), 1.0 / math.sqrt(K), np.float32)
    o = oracle.run(x, phi, np.full(3, 0.25, np.float32), np.zeros(24, np.float32))
    s = xval(x).reshape(T, -1).sum(axis=1) * np.float64(np.float32(1.0 / math.sqrt(K)))
    np.testing.assert_allclose(o.h_mix, np.repeat(s[:, None], 24, axis=1), rtol=1e-12, atol=1e-12)
    w = s * o.inv_rms
    np.testing.assert_allclose(o.h_pre, np.repeat((sig(0.25 * w) + EPS)[:, None], n, 1), rtol=1e-12)
    np.testing.assert_allclose(o.h_res, _uniform_scalar_map(n, 20, EPS), rtol=1e-14)


def test_scale_and_permutation():
    """With normEps = 0 the gates and comb are invariant under x -> 2x (exact
    in bf16) while hMix and y double; tokens are independent, so permuting
    them permutes every output."""
    T, n, D = 5, 4, 16
    x, phi, alpha, bias, _, _ = rand_inputs(T, n, D)
    a = oracle.run(x, phi, alpha, bias, norm_eps=0.0)
    x2 = to_bf16_bits(2 * xval(x)).reshape(x.shape)
    b = oracle.run(x2, phi, alpha, bias, norm_eps=0.0)
    for key in ("h_pre", "h_post", "h_res"):
        np.testing.assert_allclose(getattr(b, key), getattr(a, key), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(b.y, 2 * a.y, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(b.h_mix, 2 * a.h_mix, rtol=1e-15)
    np.testing.assert_allclose(b.inv_rms, a.inv_rms / 2, rtol=1e-15)
    perm = np.array([3, 0, 4, 1, 2])
    a = oracle.run(x, phi, alpha, bias)
    c = oracle.run(x[perm], phi, alpha, bias)
    for key in ("y", "h_pre", "h_post", "h_res", "inv_rms", "h_mix"):
        np.testing.assert_array_equal(getattr(c, key), getattr(a, key)[perm])


def test_hf32_truncates_operands():
    """HF32 simulation: the result equals the exact product of operands whose
    low 13 mantissa bits were cleared, and moves by about 2^-11 relative."""
    T, n, D = 3, 4, 64
    x, phi, alpha, bias, _, _ = rand_inputs(T, n, D)
    ph = (phi.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
    a = oracle.run(x, phi, alpha, bias, hf32=True)
    b = oracle.run(x, ph, alpha, bias)
    np.testing.assert_allclose(a.h_mix, b.h_mix, rtol=1e-15, atol=1e-15)
    c = oracle.run(x, phi, alpha, bias)
    rel = np.abs(a.h_mix - c.h_mix).max() / np.abs(c.h_mix).max()
    assert 1e-6 < rel < 2e-3


def test_hf32_on_the_folded_weight():
    """hf32=2 truncates the folded weight gamma (.) phi (rounded to fp32), x
    exact.  Closed form from the HF32 format (10 fraction bits): with
    phi = gamma = 1 + 2^-10 (both exact in HF32) the fp32 product is
    1 + 2^-9 + 2^-20, which HF32 cuts to 1 + 2^-9; the operand-wise
    simulation (hf32=1) keeps both factors and so the 2^-20 term.  With
    x = 1 everywhere each projection row is then K (1 + 2^-9) against
    K (1 + 2^-9 + 2^-20).  Without gamma the two variants agree exactly."""
    T, n, D = 2, 4, 8
    K = n * D
    R = n * n + 2 * n
    x = np.full((T, n, D), 0x3F80, dtype=np.uint16)            # bf16 1.0
    v = np.float32(1.0 + 2.0 ** -10)
    phi = np.full((R, K), v, dtype=np.float32)
    gamma = np.full((n, D), v, dtype=np.float32)
    alpha = np.array([0.5, 0.5, 0.5], dtype=np.float32)
    bias = np.zeros(R, dtype=np.float32)
    folded = oracle.run(x, phi, alpha, bias, gamma, hf32=2)
    operand = oracle.run(x, phi, alpha, bias, gamma, hf32=1)
    exact = oracle.run(x, phi, alpha, bias, gamma)
    np.testing.assert_array_equal(folded.h_mix, np.full((T, R), K * (1 + 2.0 ** -9)))
    np.testing.assert_array_equal(operand.h_mix, np.full((T, R), K * (1 + 2.0 ** -9 + 2.0 ** -20)))
    np.testing.assert_array_equal(exact.h_mix, operand.h_mix)
    # random inputs without gamma: 1 and 2 are the same simulation
    x, phi, alpha, bias, _, _ = rand_inputs(3, 4, 64)
    a = oracle.run(x, phi, alpha, bias, hf32=1)
    b = oracle.run(x, phi, alpha, bias, hf32=2)
    for key in ("y", "h_pre", "h_post", "h_res", "h_mix"):
        np.testing.assert_array_equal(getattr(a, key), getattr(b, key))
    # with gamma, the folded variant equals the exact projection of the
    # truncated fp32 product weights
    x, phi, alpha, bias, g, _ = rand_inputs(3, 4, 64, gamma=True)
    w = (phi.astype(np.float32) * g.reshape(-1).astype(np.float32)).astype(np.float32)
    w = (w.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
    c = oracle.run(x, phi, alpha, bias, g, hf32=2)
    d = oracle.run(x, w, alpha, bias)
    np.testing.assert_allclose(c.h_mix, d.h_mix, rtol=1e-15, atol=1e-15)


def test_empty_and_threads_agree():
    x, phi, alpha, bias, g, _ = rand_inputs(7, 4, 16, gamma=True)
    a = oracle.run(x, phi, alpha, bias, g, threads=1)
    b = oracle.run(x, phi, alpha, bias, g, threads=5)
    for key in ("y", "h_pre", "h_res", "sum_out", "norm_out"):
        np.testing.assert_array_equal(getattr(a, key), getattr(b, key))
    e = oracle.run(x[:0], phi, alpha, bias)
    assert e.y.shape == (0, 16)


def test_synth_tiny_workload_is_sane():
    c = make_case("tiny")
    assert tuple(c.x.shape) == (64, 4, 256) and c.phi.shape == (24, 1024)
    o = oracle.run(c.x.view(__import__("torch").int16).numpy(), c.phi.numpy(), c.alpha.numpy(),
                   c.bias.numpy())
    assert np.all(np.isfinite(o.y)) and np.all(o.h_pre > 0) and np.all(o.h_pre < 1 + 2e-6)
    assert 0.5 < np.abs(o.h_mix).std() < 2.0   # projection is O(1) at phi std 1/sqrt(K)
