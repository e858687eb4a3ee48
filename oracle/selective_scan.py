"""Mamba's selective scan, plain fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``): the tests, ``smoke()`` and
the benchmark's CPU leg call it; the CUDA path never does.

Source: "Long context, fast inference, smart decoding, and life beyond
attention", chapter "05 · State-space models: the architectural alternative",
section "Mamba: making the recurrence input-dependent, and the engineering that
makes that fast anyway", and the chapter's sequential listing of the scan.  B,
C and the step size are functions of the input; with dt = softplus(delta) per
channel d and a fixed A [D, N]:

    A_bar = exp(dt_t[d] A[d, n]),   B_bar = dt_t[d] B_t[n],
    h_t[d, n] = A_bar h_{t-1}[d, n] + B_bar x_t[d],
    y_t[d] = sum_n h_t[d, n] C_t[n].

The projections that produce delta, B and C (learned linear layers) are not
part of the scan: the scan takes their outputs, and applies the softplus.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def softplus(x):
    """log(1 + exp(x)), written to stay finite for large x."""
    x = _f64(x)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def selective_scan(x, delta, Bm, Cm, A, h0=None, return_states=False):
    """x, delta [B,T,D]; Bm, Cm [B,T,N]; A [D,N]; h0 [B,D,N] or None (zeros).
    Returns (y [B,T,D], h_T [B,D,N]) and, with ``return_states``, h after
    every token [B,T,D,N]."""
    x, delta, Bm, Cm, A = _f64(x), _f64(delta), _f64(Bm), _f64(Cm), _f64(A)
    B, T, D = x.shape
    N = A.shape[1]
    h = np.zeros((B, D, N)) if h0 is None else _f64(h0).copy()
    y = np.zeros((B, T, D))
    hs = np.zeros((B, T, D, N)) if return_states else None
    for t in range(T):
        dt = softplus(delta[:, t])                         # [B, D]
        A_bar = np.exp(dt[:, :, None] * A[None])           # [B, D, N]
        B_bar = dt[:, :, None] * Bm[:, t][:, None, :]      # [B, D, N]
        h = A_bar * h + B_bar * x[:, t][:, :, None]
        y[:, t] = (h * Cm[:, t][:, None, :]).sum(-1)
        if return_states:
            hs[:, t] = h
    return (y, h, hs) if return_states else (y, h)


def selective_scan_decode(x, delta, Bm, Cm, A, pool, slot_ids):
    """One step for R requests: x, delta [R,D]; Bm, Cm [R,N]; pool [P,D,N];
    by definition a one-token scan from each request's slot.  Returns
    (y [R,D], pool')."""
    pool = _f64(pool).copy()
    y = np.zeros(np.shape(x))
    for r, s in enumerate(int(v) for v in slot_ids):
        yr, hr = selective_scan(np.asarray(x[r])[None, None], np.asarray(delta[r])[None, None],
                                np.asarray(Bm[r])[None, None], np.asarray(Cm[r])[None, None], A, pool[s][None])
        y[r], pool[s] = yr[0, 0], hr[0]
    return y, pool
