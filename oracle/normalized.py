"""Normalised kernelised linear attention, plain fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``): the tests, ``smoke()`` and
the benchmark's CPU leg call it; the CUDA path never does.

Source: "Long context, fast inference, smart decoding, and life beyond
attention", chapter "01 · Long-context architectures", section "Linear
attention: removing softmax entirely".  With a positive feature map phi,

    Attention_i = sum_{j<=i} (phi(q_i) . phi(k_j)) v_j / sum_{j<=i} phi(q_i) . phi(k_j),

and reassociating the sums gives a running d_k x d_v state and a running
normaliser:

    S_i = S_{i-1} + phi(k_i)^T v_i,   z_i = z_{i-1} + phi(k_i),
    o_i = phi(q_i) S_i / (phi(q_i) . z_i + eps).

The page's sequential version uses phi(x) = elu(x) + 1 (positive) and
eps = 1e-6 in the denominator.  With bf16 activations the feature values are
rounded to bf16 before use, as the GPU's tensor-core operands are (the same
reading as the other front-end outputs).  Grouped q / k heads are expanded
with ``oracle.expand_groups``.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def feature_map(x):
    """phi(x) = elu(x) + 1: x + 1 for x > 0, exp(x) otherwise."""
    x = _f64(x)
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def features(q, k, act_bf16):
    from . import round_bf16
    fq, fk = feature_map(q), feature_map(k)
    if act_bf16:
        fq, fk = round_bf16(fq), round_bf16(fk)
    return fq, fk


def nla_prefill(q, k, v, S0=None, z0=None, act_bf16=True, return_states=False):
    """q, k [B,T,Hq,dk] (raw; Hq divides H), v [B,T,H,dv]; S0 [B,H,dk,dv] and
    z0 [B,H,dk] or None (zeros).  Returns (o [B,T,H,dv], S_T, z_T) and, with
    ``return_states``, the (S, z) after every token."""
    from . import expand_groups
    v = _f64(v)
    B, T, H, dv = v.shape
    fq, fk = features(q, k, act_bf16)
    fq, fk = expand_groups(fq, H), expand_groups(fk, H)
    dk = fq.shape[-1]
    S = np.zeros((B, H, dk, dv)) if S0 is None else _f64(S0).copy()
    z = np.zeros((B, H, dk)) if z0 is None else _f64(z0).copy()
    o = np.zeros((B, T, H, dv))
    Ss = np.zeros((B, T, H, dk, dv)) if return_states else None
    zs = np.zeros((B, T, H, dk)) if return_states else None
    for b in range(B):
        for h in range(H):
            Sb, zb = S[b, h], z[b, h]
            for t in range(T):
                Sb += np.outer(fk[b, t, h], v[b, t, h])
                zb += fk[b, t, h]
                o[b, t, h] = (fq[b, t, h] @ Sb) / (fq[b, t, h] @ zb + EPS)
                if return_states:
                    Ss[b, t, h], zs[b, t, h] = Sb, zb
    if return_states:
        return o, S, z, Ss, zs
    return o, S, z


def nla_decode(q, k, v, pool, zpool, slot_ids, act_bf16=True):
    """One token per request: q, k [N,Hq,dk], v [N,H,dv]; pool [P,H,dk,dv],
    zpool [P,H,dk].  By definition a one-token prefill from each request's
    slot.  Returns (o [N,H,dv], pool', zpool')."""
    pool, zpool = _f64(pool).copy(), _f64(zpool).copy()
    N = np.shape(v)[0]
    o = np.zeros(np.shape(v))
    for n, s in enumerate(int(x) for x in slot_ids):
        on, Sn, zn = nla_prefill(np.asarray(q[n])[None, None], np.asarray(k[n])[None, None],
                                 np.asarray(v[n])[None, None], pool[s][None], zpool[s][None], act_bf16)
        o[n], pool[s], zpool[s] = on[0, 0], Sn[0], zn[0]
    return o, pool, zpool


def nla_spec_decode(q, k, v, pool, zpool, src_slot, dst_slots, act_bf16=True):
    """D draft tokens per request from src_slot[n]; the state (and normaliser)
    after draft i goes to dst_slots[n][i].  Returns (o [N,D,H,dv], pool', zpool')."""
    pool, zpool = _f64(pool).copy(), _f64(zpool).copy()
    N, D = np.shape(v)[:2]
    o = np.zeros(np.shape(v))
    for n in range(N):
        S, z = pool[int(src_slot[n])][None].copy(), zpool[int(src_slot[n])][None].copy()
        for i in range(D):
            on, S, z = nla_prefill(np.asarray(q[n, i])[None, None], np.asarray(k[n, i])[None, None],
                                   np.asarray(v[n, i])[None, None], S, z, act_bf16)
            o[n, i] = on[0, 0]
            pool[int(dst_slots[n][i])], zpool[int(dst_slots[n][i])] = S[0], z[0]
    return o, pool, zpool
