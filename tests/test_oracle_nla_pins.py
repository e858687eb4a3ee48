"""Pins for the normalised kernelised linear attention oracle.

Source: "Long context, fast inference, smart decoding, and life beyond
attention", chapter "01 · Long-context architectures", section "Linear
attention: removing softmax entirely": the kernelised attention
sum_j (phi(q_i).phi(k_j)) v_j / sum_j phi(q_i).phi(k_j) equals the running
state form; phi = elu + 1, eps = 1e-6.

* the parallel (quadratic) form, written with matrices, pins the recurrence;
* phi is torch's elu plus one;
* constant values pass through (the weights are normalised);
* segments handing (S, z) on, and decode steps, equal one prefill.
"""
import numpy as np
import torch

from oracle.normalized import EPS, feature_map, nla_decode, nla_prefill, nla_spec_decode


def _rand(rng, B, T, H, Hq, dk, dv):
    q = rng.standard_normal((B, T, Hq, dk))
    k = rng.standard_normal((B, T, Hq, dk))
    v = rng.standard_normal((B, T, H, dv))
    return q, k, v


def test_feature_map_is_elu_plus_one():
    x = np.linspace(-30, 30, 2001)
    ref = torch.nn.functional.elu(torch.tensor(x, dtype=torch.float64)).numpy() + 1.0
    # elu(x) + 1 = (exp(x) - 1) + 1 loses the low bits of exp(x) for x << 0
    np.testing.assert_allclose(feature_map(x), ref, rtol=1e-15, atol=1e-16)
    assert (feature_map(x) > 0).all()


def test_recurrence_equals_parallel_form():
    """O = (A V) / (A 1 + eps), A = tril(phi(Q) phi(K)^T), from zero state."""
    rng = np.random.default_rng(1)
    q, k, v = _rand(rng, 2, 23, 3, 3, 6, 5)
    o, S, z = nla_prefill(q, k, v, act_bf16=False)
    for b in range(2):
        for h in range(3):
            fq, fk = feature_map(q[b, :, h]), feature_map(k[b, :, h])
            A = np.tril(fq @ fk.T)
            want = (A @ v[b, :, h]) / (A.sum(axis=1, keepdims=True) + EPS)
            np.testing.assert_allclose(o[b, :, h], want, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(S[b, h], fk.T @ v[b, :, h], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(z[b, h], fk.sum(axis=0), rtol=1e-12)


def test_grouped_heads_use_their_group():
    rng = np.random.default_rng(2)
    q, k, v = _rand(rng, 1, 9, 4, 2, 4, 3)
    o, _, _ = nla_prefill(q, k, v, act_bf16=False)
    for h in range(4):
        fq, fk = feature_map(q[0, :, h // 2]), feature_map(k[0, :, h // 2])
        A = np.tril(fq @ fk.T)
        np.testing.assert_allclose(o[0, :, h], (A @ v[0, :, h]) / (A.sum(1, keepdims=True) + EPS),
                                   rtol=1e-12, atol=1e-13)


def test_constant_values_pass_through():
    rng = np.random.default_rng(3)
    q, k, _ = _rand(rng, 1, 30, 1, 1, 8, 4)
    c = rng.standard_normal(4)
    v = np.broadcast_to(c, (1, 30, 1, 4)).copy()
    o, _, _ = nla_prefill(q, k, v, act_bf16=False)
    np.testing.assert_allclose(o[0, :, 0], np.broadcast_to(c, (30, 4)), rtol=1e-5)


def test_segments_and_decode_steps_equal_one_prefill():
    rng = np.random.default_rng(4)
    q, k, v = _rand(rng, 1, 20, 2, 2, 5, 3)
    o, S, z = nla_prefill(q, k, v, act_bf16=False)
    o1, S1, z1 = nla_prefill(q[:, :12], k[:, :12], v[:, :12], act_bf16=False)
    o2, S2, z2 = nla_prefill(q[:, 12:], k[:, 12:], v[:, 12:], S1, z1, act_bf16=False)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S2, S, rtol=1e-12)
    pool, zpool = np.zeros((3,) + S.shape[1:]), np.zeros((3,) + z.shape[1:])
    pool[1], zpool[1] = S1[0], z1[0]
    for t in range(12, 20):
        od, pool, zpool = nla_decode(q[:, t], k[:, t], v[:, t], pool, zpool, [1], act_bf16=False)
        np.testing.assert_allclose(od[0], o[0, t], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(pool[1], S[0], rtol=1e-12)
    np.testing.assert_allclose(zpool[1], z[0], rtol=1e-12)


def test_spec_states_are_prefix_states():
    rng = np.random.default_rng(5)
    q, k, v = _rand(rng, 2, 3, 2, 1, 4, 4)  # two requests (as batch), three drafts
    pool, zpool = np.zeros((8, 2, 4, 4)), np.zeros((8, 2, 4))
    o, pool2, zpool2 = nla_spec_decode(q, k, v, pool, zpool, [0, 1], [[2, 3, 4], [5, 6, 7]], act_bf16=False)
    for n, dst in enumerate([[2, 3, 4], [5, 6, 7]]):
        for i in range(3):
            on, Sn, zn = nla_prefill(q[n:n + 1, :i + 1], k[n:n + 1, :i + 1], v[n:n + 1, :i + 1], act_bf16=False)
            np.testing.assert_allclose(pool2[dst[i]], Sn[0], rtol=1e-12)
            np.testing.assert_allclose(zpool2[dst[i]], zn[0], rtol=1e-12)
            np.testing.assert_allclose(o[n, i], on[0, i], rtol=1e-12, atol=1e-13)
