"""Pins of the oracle's fp16 x path (the Sinkhorn page lists fp16 as the
other x type): the binary16 decoding against numpy's float16 on every one
of the 65536 bit patterns, and the fp16 forward against the bf16 forward on
values that both formats hold exactly (so every output must agree to the
last bit of the double result)."""
import numpy as np

import oracle


def test_half_decoding_all_patterns():
    bits = np.arange(65536, dtype=np.uint32)
    want = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle.half_value(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_fp16_forward_equals_bf16_forward_on_shared_values():
    rng = np.random.default_rng(0)
    T, n, D = 5, 4, 32
    K, R = n * D, n * n + 2 * n
    # values with at most 8 significant bits and moderate exponents: exact
    # in bf16 and in fp16
    mant = rng.integers(-255, 256, size=(T, n, D))
    vals = (mant * 2.0 ** rng.integers(-12, -2, size=(T, n, D))).astype(np.float32)
    bf = (vals.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bf.astype(np.uint32) << 16).view(np.float32), vals)
    hf = vals.astype(np.float16)
    assert np.array_equal(hf.astype(np.float32), vals)
    phi = (rng.standard_normal((R, K)) / np.sqrt(K)).astype(np.float32)
    alpha = np.array([0.9, 1.1, 1.0], np.float32)
    bias = (0.1 * rng.standard_normal(R)).astype(np.float32)
    a = oracle.run(bf, phi, alpha, bias)
    b = oracle.run(hf.view(np.uint16), phi, alpha, bias, x_fp16=True)
    for k in ("y", "h_post", "h_res", "h_pre", "inv_rms", "h_mix", "sum_out", "norm_out"):
        assert np.array_equal(getattr(a, k), getattr(b, k)), k
