"""Pins of the post-mapping oracle (hc_post) against what the mathematics
fixes, independently of the oracle's own loops:

* identity comb with post = 0 returns the residual streams exactly;
* comb = 0 returns post (outer) x exactly;
* a comb with a single 1 at (i, j) moves residual stream i into output
  stream j (the mixing orientation: out_j = sum_i comb[i][j] residual_i);
* a permutation comb permutes the streams;
* exact rational evaluation (fractions) on tiny random inputs.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _bits(a):
    return (np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _vals(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(T, n, D, seed):
    rng = np.random.default_rng(seed)
    x = _bits(rng.standard_normal((T, D)))
    res = _bits(rng.standard_normal((T, n, D)))
    post = (2.0 * rng.random((T, n))).astype(np.float32)
    comb = rng.random((T, n, n)).astype(np.float32)
    return x, res, post, comb


@pytest.mark.parametrize("n", [4, 6, 8])
def test_identity_comb_returns_residual(n):
    x, res, _, _ = _case(5, n, 24, seed=n)
    comb = np.broadcast_to(np.eye(n, dtype=np.float32), (5, n, n)).copy()
    out = oracle.run_post(x, res, np.zeros((5, n), np.float32), comb)
    assert np.array_equal(out, _vals(res))


def test_zero_comb_is_post_times_x():
    x, res, post, _ = _case(7, 4, 40, seed=1)
    out = oracle.run_post(x, res, post, np.zeros((7, 4, 4), np.float32))
    want = post.astype(np.float64)[:, :, None] * _vals(x)[:, None, :]
    assert np.array_equal(out, want)


def test_mixing_orientation():
    T, n, D = 3, 4, 16
    x, res, post, _ = _case(T, n, D, seed=2)
    comb = np.zeros((T, n, n), np.float32)
    comb[:, 0, 1] = 1.0                       # stream 0 feeds output stream 1
    out = oracle.run_post(x, res, post, comb)
    base = post.astype(np.float64)[:, :, None] * _vals(x)[:, None, :]
    want = base.copy()
    want[:, 1, :] += _vals(res)[:, 0, :]
    assert np.array_equal(out, want)


def test_permutation_comb():
    T, n, D = 4, 6, 8
    x, res, _, _ = _case(T, n, D, seed=3)
    perm = np.array([3, 0, 5, 1, 2, 4])
    comb = np.zeros((T, n, n), np.float32)
    comb[:, np.arange(n), perm] = 1.0         # stream i goes to output perm[i]
    out = oracle.run_post(x, res, np.zeros((T, n), np.float32), comb)
    for i in range(n):
        assert np.array_equal(out[:, perm[i], :], _vals(res)[:, i, :])


def test_exact_rational_evaluation():
    T, n, D = 2, 4, 6
    x, res, post, comb = _case(T, n, D, seed=4)
    out = oracle.run_post(x, res, post, comb)
    xv, rv = _vals(x), _vals(res)
    for t in range(T):
        for j in range(n):
            for d in range(D):
                exact = Fraction(float(post[t, j])) * Fraction(xv[t, d])
                for i in range(n):
                    exact += Fraction(float(comb[t, i, j])) * Fraction(rv[t, i, d])
                assert abs(out[t, j, d] - float(exact)) <= 1e-12 * (1 + abs(float(exact)))
