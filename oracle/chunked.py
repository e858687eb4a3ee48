"""Second, independent fp64 path: the chunked form of the same layer.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).  It exists to pin the
recurrence in ``glinattn_oracle.c`` against a different formulation, and to
write down, in plain numpy, the chunk algebra that the prefill kernels use.

"Inference for linear attention and hybrid architectures", section "Two ways
to write the same computation", gives the chunked form of gated linear
attention: within a chunk, g is the cumulative log decay, position i sees
position j <= i with decay exp(g_i - g_j), the intra-chunk part is a C x C
decay-masked "attention", the inter-chunk part is exp(g) * (q S), and the
state moves on as S <- exp(g_C) S + (exp(g_C - g) * K)^T V.  For DeltaNet the
page says only that the error-correcting updates inside a chunk must first be
written in matrix form.  The matrix form used here is derived from the
recurrence S_t = alpha_t S_{t-1} + k_t^T u_t with
u_t = beta_t (v_t - alpha_t k_t S_{t-1}):

    with start state S and gamma_i = exp(g_i) inside the chunk,
    u_i = beta_i (v_i - gamma_i k_i S - sum_{j<i} (gamma_i/gamma_j)(k_i . k_j) u_j)
    => (I + A) U = diag(beta) V - diag(beta gamma) K S,
       A_ij = beta_i exp(g_i - g_j) (k_i . k_j) for j < i, else 0
    => U = U~ - W S,  U~ = (I + A)^-1 diag(beta) V,  W = (I + A)^-1 diag(beta gamma) K
    O      = diag(gamma) Q S + ((Q K^T) * D) U,   D_ij = exp(g_i - g_j) [j <= i]
    S_next = gamma_C S + (diag(exp(g_C - g)) K)^T U

Gated linear attention is the case U = V.  Every exponent g_i - g_j (j <= i)
and g_C - g_j is <= 0, so no 1/gamma is ever formed.  (I + A) is unit lower
triangular; it is solved with scipy's triangular solver.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular

GLA, GDN = 0, 1


def chunked_one(variant, q, k, v, alpha, beta=None, S0=None, C=64):
    """One (batch, head) sequence: q, k [T,dk], v [T,dv], alpha/beta [T].
    Returns (o [T,dv], S_T [dk,dv])."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    alpha = np.asarray(alpha, dtype=np.float64)
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((T, dv))
    for s in range(0, T, C):
        e = min(s + C, T)
        Q, K, V = q[s:e], k[s:e], v[s:e]
        n = e - s
        g = np.cumsum(np.log(alpha[s:e]))
        diff = g[:, None] - g[None, :]
        lower = np.tril(np.ones((n, n), dtype=bool))
        D = np.where(lower, np.exp(np.where(lower, diff, 0.0)), 0.0)
        gamma = np.exp(g)
        if variant == GDN:
            b = np.asarray(beta[s:e], dtype=np.float64)
            A = np.tril(b[:, None] * (K @ K.T) * D, -1)
            IA = np.eye(n) + A
            W = solve_triangular(IA, (b * gamma)[:, None] * K, lower=True, unit_diagonal=True)
            Ut = solve_triangular(IA, b[:, None] * V, lower=True, unit_diagonal=True)
            U = Ut - W @ S
        else:
            U = V
        o[s:e] = gamma[:, None] * (Q @ S) + ((Q @ K.T) * D) @ U
        S = gamma[-1] * S + (np.exp(g[-1] - g)[:, None] * K).T @ U
    return o, S


def chunked(variant, q, k, v, alpha, beta=None, S0=None, C=64):
    """Batched wrapper: q, k [B,T,H,dk], v [B,T,H,dv], alpha/beta [B,T,H],
    S0 [B,H,dk,dv] or None.  Returns (o [B,T,H,dv], S_T [B,H,dk,dv])."""
    q = np.asarray(q, dtype=np.float64)
    B, T, H, dk = q.shape
    dv = np.shape(v)[-1]
    o = np.zeros((B, T, H, dv))
    S = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            o[b, :, h], S[b, h] = chunked_one(
                variant, q[b, :, h], np.asarray(k)[b, :, h], np.asarray(v)[b, :, h],
                np.asarray(alpha)[b, :, h], None if beta is None else np.asarray(beta)[b, :, h],
                None if S0 is None else np.asarray(S0)[b, h], C)
    return o, S
