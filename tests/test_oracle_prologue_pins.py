"""Pins of the oracle's block prologue ([paper] §3.4 "Token mixing block", Fig. 1).

q, k, v come from their projections through a short causal convolution and
SiLU; alpha uses Mamba2's parameterisation and beta a sigmoid.  Each test
checks the oracle against something other than itself: closed forms, numpy's
convolution, shifting, state carry across calls and causality.
"""
import math

import numpy as np
import pytest

import oracle


def silu(z):
    return z / (1.0 + np.exp(-z))


def test_current_token_tap_is_silu_of_the_input():
    rng = np.random.default_rng(30)
    x = rng.standard_normal((2, 9, 3, 5))
    w = np.zeros((3, 5, 4))
    w[..., 3] = 1.0                       # tap K-1 multiplies the current token
    y, _ = oracle.short_conv_silu(x, w)
    np.testing.assert_allclose(y, silu(x), atol=1e-14)


def test_oldest_tap_is_a_delay_of_k_minus_one():
    rng = np.random.default_rng(31)
    x = rng.standard_normal((1, 12, 2, 4))
    w = np.zeros((2, 4, 4))
    w[..., 0] = 1.0
    y, _ = oracle.short_conv_silu(x, w)
    np.testing.assert_allclose(y[:, 3:], silu(x[:, :-3]), atol=1e-14)
    np.testing.assert_allclose(y[:, :3], 0.0, atol=0)   # zero history, silu(0) = 0


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_conv_equals_numpy_convolve(K):
    rng = np.random.default_rng(32 + K)
    B, T, H, d = 2, 17, 2, 3
    x = rng.standard_normal((B, T, H, d))
    w = rng.standard_normal((H, d, K))
    y, _ = oracle.short_conv_silu(x, w)
    for b in range(B):
        for h in range(H):
            for c in range(d):
                z = np.convolve(x[b, :, h, c], w[h, c, ::-1])[:T]
                np.testing.assert_allclose(y[b, :, h, c], silu(z), atol=1e-13)


def test_causal():
    rng = np.random.default_rng(36)
    x = rng.standard_normal((1, 20, 2, 4))
    w = rng.standard_normal((2, 4, 4))
    y1, _ = oracle.short_conv_silu(x, w)
    x2 = x.copy()
    x2[:, 11:] += rng.standard_normal(x2[:, 11:].shape)
    y2, _ = oracle.short_conv_silu(x2, w)
    np.testing.assert_array_equal(y1[:, :11], y2[:, :11])
    assert np.abs(y1[:, 11:] - y2[:, 11:]).max() > 1e-3


def test_state_carry_two_calls_equal_one():
    rng = np.random.default_rng(37)
    B, T, H, d, K = 2, 23, 2, 3, 4
    x = rng.standard_normal((B, T, H, d))
    w = rng.standard_normal((H, d, K))
    s0 = rng.standard_normal((B, K - 1, H, d))
    y, s = oracle.short_conv_silu(x, w, state_in=s0)
    for T1 in (1, 2, 9):
        ya, sa = oracle.short_conv_silu(x[:, :T1], w, state_in=s0)
        yb, sb = oracle.short_conv_silu(x[:, T1:], w, state_in=sa)
        np.testing.assert_allclose(np.concatenate([ya, yb], 1), y, atol=1e-14)
        np.testing.assert_allclose(sb, s, atol=0)
    # the carried state is the last K-1 inputs, oldest first
    np.testing.assert_array_equal(s, x[:, -(K - 1):])
    # a call shorter than K-1 keeps the older history in its state
    _, s1 = oracle.short_conv_silu(x[:, :1], w, state_in=s0)
    np.testing.assert_array_equal(s1[:, :K - 2], s0[:, 1:])
    np.testing.assert_array_equal(s1[:, K - 2], x[:, 0])


def test_varlen_equals_separate_calls():
    rng = np.random.default_rng(38)
    lens = [5, 0, 1, 12, 3]
    H, d, K = 2, 3, 4
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x = rng.standard_normal((1, T, H, d))
    w = rng.standard_normal((H, d, K))
    s0 = rng.standard_normal((len(lens), K - 1, H, d))
    y, s = oracle.short_conv_silu(x, w, state_in=s0, cu_seqlens=cu)
    for n, L in enumerate(lens):
        yn, sn = oracle.short_conv_silu(x[:, cu[n]:cu[n + 1]], w, state_in=s0[n:n + 1])
        np.testing.assert_allclose(y[:, cu[n]:cu[n + 1]], yn, atol=1e-14)
        np.testing.assert_allclose(s[n:n + 1], sn, atol=0)
    np.testing.assert_array_equal(s[1], s0[1])    # an empty sequence keeps its history


def test_gate_activations_closed_forms():
    """g = log alpha = -exp(A_log) softplus(a + dt_bias) (Mamba2), beta = sigmoid(b)."""
    rng = np.random.default_rng(39)
    H = 4
    A_log = rng.standard_normal(H)
    dt_bias = rng.standard_normal(H)
    # a = -dt_bias: softplus(0) = log 2
    g, beta = oracle.gate_activations(-dt_bias[None], np.zeros((1, H)), A_log, dt_bias)
    np.testing.assert_allclose(g[0], -np.exp(A_log) * math.log(2.0), rtol=1e-14)
    np.testing.assert_allclose(beta[0], 0.5, atol=0)
    # large argument: softplus(z) -> z; very negative: -> e^z
    a = np.array([[40.0 - dt_bias[h] for h in range(H)]])
    g, _ = oracle.gate_activations(a, np.zeros((1, H)), A_log, dt_bias)
    np.testing.assert_allclose(g[0], -np.exp(A_log) * 40.0, rtol=1e-14)
    a = np.array([[-30.0 - dt_bias[h] for h in range(H)]])
    g, _ = oracle.gate_activations(a, np.zeros((1, H)), A_log, dt_bias)
    np.testing.assert_allclose(g[0], -np.exp(A_log) * math.exp(-30.0), rtol=1e-12)
    # alpha in (0, 1) and beta symmetric about 1/2
    a = 3 * rng.standard_normal((50, H))
    b = 3 * rng.standard_normal((50, H))
    g, beta = oracle.gate_activations(a, b, A_log, dt_bias)
    _, beta_m = oracle.gate_activations(a, -b, A_log, dt_bias)
    assert (g < 0).all()
    np.testing.assert_allclose(beta + beta_m, 1.0, atol=1e-15)
