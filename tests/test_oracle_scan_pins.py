"""Pins for the selective-scan oracle.

Source: "Long context, fast inference, smart decoding, and life beyond
attention", chapter "05 · State-space models: the architectural alternative":
the recurrence h_t = A_bar_t h_{t-1} + B_bar_t x_t unrolls into a sum over
past inputs (the page's h_t = sum_k A_bar^(t-k) B_bar x_k for fixed
parameters, here with time-varying ones), and with fixed parameters the output
is a convolution with the kernel (C B_bar, C A_bar B_bar, C A_bar^2 B_bar, ...).

* the unrolled sum, written as explicit loops, pins the recurrence;
* with constant delta, B and C the output is that convolution;
* softplus matches torch's;
* delta -> -inf (dt = 0) freezes the state; segments and decode steps chain.
"""
import numpy as np
import torch

from oracle.selective_scan import selective_scan, selective_scan_decode, softplus


def _rand(rng, B, T, D, N):
    x = rng.standard_normal((B, T, D))
    delta = rng.standard_normal((B, T, D)) - 1.0
    Bm = rng.standard_normal((B, T, N))
    Cm = rng.standard_normal((B, T, N))
    A = -np.exp(rng.random((D, N)))
    return x, delta, Bm, Cm, A


def test_softplus_matches_torch():
    x = np.linspace(-40, 40, 4001)
    ref = torch.nn.functional.softplus(torch.tensor(x, dtype=torch.float64), threshold=1000).numpy()
    np.testing.assert_allclose(softplus(x), ref, rtol=1e-14, atol=1e-300)


def test_recurrence_equals_unrolled_sum():
    """y_t[d] = sum_{s<=t} sum_n C_t[n] (prod_{r=s+1..t} exp(dt_r A)) dt_s B_s[n] x_s[d]
    + sum_n C_t[n] prod_{r<=t} exp(dt_r A) h0[d, n]."""
    rng = np.random.default_rng(0)
    x, delta, Bm, Cm, A = _rand(rng, 2, 11, 3, 4)
    h0 = rng.standard_normal((2, 3, 4))
    y, h = selective_scan(x, delta, Bm, Cm, A, h0)
    dt = softplus(delta)
    for b in range(2):
        for d in range(3):
            for t in range(11):
                acc = 0.0
                for n in range(4):
                    dec = np.exp(A[d, n] * dt[b, :t + 1, d].sum())
                    acc += Cm[b, t, n] * dec * h0[b, d, n]
                    for s in range(t + 1):
                        dec = np.exp(A[d, n] * dt[b, s + 1:t + 1, d].sum())
                        acc += Cm[b, t, n] * dec * dt[b, s, d] * Bm[b, s, n] * x[b, s, d]
                np.testing.assert_allclose(y[b, t, d], acc, rtol=1e-11, atol=1e-12)


def test_fixed_parameters_give_the_convolution():
    """Constant delta, B, C: y = x * K with K_k = sum_n C[n] A_bar^k B_bar[n]."""
    rng = np.random.default_rng(1)
    T, D, N = 25, 2, 3
    x = rng.standard_normal((1, T, D))
    A = -np.exp(rng.random((D, N)))
    d0, b0, c0 = rng.standard_normal(D) - 1.0, rng.standard_normal(N), rng.standard_normal(N)
    delta = np.broadcast_to(d0, (1, T, D)).copy()
    Bm = np.broadcast_to(b0, (1, T, N)).copy()
    Cm = np.broadcast_to(c0, (1, T, N)).copy()
    y, _ = selective_scan(x, delta, Bm, Cm, A)
    dt = softplus(d0)
    for d in range(D):
        A_bar = np.exp(dt[d] * A[d])
        K = np.array([(c0 * A_bar ** k * dt[d] * b0).sum() for k in range(T)])
        conv = np.convolve(x[0, :, d], K)[:T]
        np.testing.assert_allclose(y[0, :, d], conv, rtol=1e-11, atol=1e-12)


def test_zero_step_freezes_the_state():
    rng = np.random.default_rng(2)
    x, _, Bm, Cm, A = _rand(rng, 1, 6, 2, 3)
    delta = np.full((1, 6, 2), -800.0)  # softplus -> 0 (underflows to exactly 0)
    h0 = rng.standard_normal((1, 2, 3))
    y, h = selective_scan(x, delta, Bm, Cm, A, h0)
    np.testing.assert_array_equal(h, h0)
    np.testing.assert_allclose(y[0], np.einsum("dn,tn->td", h0[0], Cm[0]), rtol=1e-14)


def test_segments_and_decode_steps_chain():
    rng = np.random.default_rng(3)
    x, delta, Bm, Cm, A = _rand(rng, 2, 14, 3, 4)
    y, h = selective_scan(x, delta, Bm, Cm, A)
    y1, h1 = selective_scan(x[:, :9], delta[:, :9], Bm[:, :9], Cm[:, :9], A)
    y2, h2 = selective_scan(x[:, 9:], delta[:, 9:], Bm[:, 9:], Cm[:, 9:], A, h1)
    np.testing.assert_allclose(np.concatenate([y1, y2], 1), y, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(h2, h, rtol=1e-12)
    pool = np.zeros((5, 3, 4))
    pool[[4, 1]] = h1
    for t in range(9, 14):
        yd, pool = selective_scan_decode(x[:, t], delta[:, t], Bm[:, t], Cm[:, t], A, pool, [4, 1])
        np.testing.assert_allclose(yd, y[:, t], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(pool[[4, 1]], h, rtol=1e-12)
