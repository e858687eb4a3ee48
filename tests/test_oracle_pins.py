"""Pins for the fp64 oracle, each against something other than the oracle itself.

Source: "Inference for linear attention and hybrid architectures",
section "Two ways to write the same computation" (recurrences, chunked form,
short convolution) and section "Checking on a real model" (segmented prefill
and stepwise decode agree with one-shot prefill).

What pins what:
* brute-force O(T^2) sums and explicit transition-matrix products on tiny
  inputs pin the recurrences (a dropped term, a wrong sign, a misplaced gate or
  a transposed operand changes them);
* alpha = 1 reduces gated linear attention to the textbook unnormalised causal
  linear attention tril(Q K^T) V;
* beta = 0 reduces Gated DeltaNet to pure decay;
* with unit keys, k_t S_t = alpha_t (1 - beta_t) k_t S_{t-1} + beta_t v_t;
* the independent chunked form agrees with the recurrence for several C,
  including C = 1 and C = T;
* the page's worked example (seed 0) reproduces allclose(atol=1e-5) == True;
* the convolution reduces to torch's conv1d, the bf16 rounding to torch's cast.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import GDN, GLA
from oracle.chunked import chunked

from gated_deltanet_02_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, B, T, H, dk, dv, s0=True):
    q = rng.standard_normal((B, T, H, dk)) / np.sqrt(dk)
    k = rng.standard_normal((B, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    alpha = 1.0 / (1.0 + np.exp(-(rng.standard_normal((B, T, H)) + 2.0)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    S0 = 0.3 * rng.standard_normal((B, H, dk, dv)) if s0 else None
    return q, k, v, alpha, beta, S0


# ---------------------------------------------------------------------------
# brute force
# ---------------------------------------------------------------------------

def _gla_bruteforce(q, k, v, alpha, S0):
    """o_t = sum_{s<=t} (prod_{r=s+1..t} alpha_r)(q_t.k_s) v_s + (prod_{r<=t} alpha_r) q_t S0."""
    T = q.shape[0]
    o = np.zeros((T, v.shape[1]))
    for t in range(T):
        for s in range(t + 1):
            o[t] += np.prod(alpha[s + 1:t + 1]) * (q[t] @ k[s]) * v[s]
        o[t] += np.prod(alpha[:t + 1]) * (q[t] @ S0)
    S_T = np.prod(alpha) * S0 + sum(np.prod(alpha[s + 1:]) * np.outer(k[s], v[s])
                                    for s in range(T))
    return o, S_T


def _gdn_transitions(q, k, v, alpha, beta, S0):
    """S_t = M_t S_{t-1} + beta_t k_t^T v_t with the explicit d x d matrix
    M_t = alpha_t (I - beta_t k_t^T k_t); the closed form is built from products
    of the M's, o_t = q_t S_t."""
    T, dk = k.shape
    M = [alpha[t] * (np.eye(dk) - beta[t] * np.outer(k[t], k[t])) for t in range(T)]
    o = np.zeros((T, v.shape[1]))
    for t in range(T):
        P = np.eye(dk)
        St = np.zeros((dk, v.shape[1]))
        for s in range(t, -1, -1):  # P = M_t ... M_{s+1}
            St += P @ (beta[s] * np.outer(k[s], v[s]))
            P = P @ M[s]
        St += P @ S0  # P = M_t ... M_1
        o[t] = q[t] @ St
    return o, St


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gla_matches_bruteforce(seed):
    rng = np.random.default_rng(seed)
    q, k, v, alpha, _, S0 = _rand(rng, 2, 17, 3, 8, 5)
    o, S = oracle.recurrence(GLA, q, k, v, alpha, S0=S0)
    for b in range(2):
        for h in range(3):
            ob, Sb = _gla_bruteforce(q[b, :, h], k[b, :, h], v[b, :, h], alpha[b, :, h], S0[b, h])
            np.testing.assert_allclose(o[b, :, h], ob, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(S[b, h], Sb, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1])
def test_gdn_matches_transition_products(seed):
    rng = np.random.default_rng(seed)
    q, k, v, alpha, beta, S0 = _rand(rng, 1, 13, 2, 6, 4)
    o, S = oracle.recurrence(GDN, q, k, v, alpha, beta, S0)
    for h in range(2):
        ob, Sb = _gdn_transitions(q[0, :, h], k[0, :, h], v[0, :, h], alpha[0, :, h],
                                  beta[0, :, h], S0[0, h])
        np.testing.assert_allclose(o[0, :, h], ob, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(S[0, h], Sb, rtol=1e-11, atol=1e-12)


def test_gdn_gate_multiplies_erase_not_write():
    """The write beta k^T v is not decayed: with S0 = 0 and one token,
    S_1 = beta k^T v whatever alpha is (a gate on the write would scale it)."""
    rng = np.random.default_rng(5)
    q, k, v, _, beta, _ = _rand(rng, 1, 1, 1, 4, 3, s0=False)
    for a in (0.3, 0.9):
        alpha = np.full((1, 1, 1), a)
        _, S = oracle.recurrence(GDN, q, k, v, alpha, beta)
        np.testing.assert_allclose(S[0, 0], beta[0, 0, 0] * np.outer(k[0, 0, 0], v[0, 0, 0]),
                                   rtol=1e-14)


# ---------------------------------------------------------------------------
# closed forms and special cases
# ---------------------------------------------------------------------------

def test_alpha_one_is_causal_linear_attention():
    """alpha = 1: o_t = sum_{s<=t} (q_t.k_s) v_s, i.e. O = tril(Q K^T) V."""
    rng = np.random.default_rng(3)
    q, k, v, _, _, _ = _rand(rng, 1, 40, 1, 7, 9, s0=False)
    alpha = np.ones((1, 40, 1))
    o, S = oracle.recurrence(GLA, q, k, v, alpha)
    Q, K, V = q[0, :, 0], k[0, :, 0], v[0, :, 0]
    np.testing.assert_allclose(o[0, :, 0], np.tril(Q @ K.T) @ V, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S[0, 0], K.T @ V, rtol=1e-12, atol=1e-12)


def test_gdn_beta_zero_is_pure_decay():
    rng = np.random.default_rng(4)
    q, k, v, alpha, _, S0 = _rand(rng, 1, 30, 2, 8, 8)
    beta = np.zeros_like(alpha)
    o, S = oracle.recurrence(GDN, q, k, v, alpha, beta, S0)
    gamma = np.cumprod(alpha, axis=1)
    for h in range(2):
        expect = gamma[0, :, h, None] * (q[0, :, h] @ S0[0, h])
        np.testing.assert_allclose(o[0, :, h], expect, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(S[0, h], gamma[0, -1, h] * S0[0, h], rtol=1e-12)


def test_gdn_unit_key_erase_invariant():
    """Erase along k_t, then write: with |k_t| = 1,
    k_t S_t = alpha_t (1 - beta_t) k_t S_{t-1} + beta_t v_t; beta = 1 stores v_t exactly."""
    rng = np.random.default_rng(6)
    q, k, v, alpha, beta, S0 = _rand(rng, 1, 12, 1, 8, 5)
    beta[0, 5, 0] = 1.0
    _, _, states = oracle.recurrence(GDN, q, k, v, alpha, beta, S0, return_states=True)
    prev = S0[0, 0]
    for t in range(12):
        kt = k[0, t, 0]
        lhs = kt @ states[0, t, 0]
        rhs = alpha[0, t, 0] * (1 - beta[0, t, 0]) * (kt @ prev) + beta[0, t, 0] * v[0, t, 0]
        np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
        prev = states[0, t, 0]
    np.testing.assert_allclose(k[0, 5, 0] @ states[0, 5, 0], v[0, 5, 0], rtol=1e-12, atol=1e-12)


def test_gate_outside_domain_is_rejected():
    rng = np.random.default_rng(7)
    q, k, v, alpha, beta, _ = _rand(rng, 1, 4, 1, 4, 4, s0=False)
    for bad in (0.0, -0.5, 1.5, np.nan):
        a = alpha.copy()
        a[0, 2, 0] = bad
        with pytest.raises(ValueError):
            oracle.recurrence(GDN, q, k, v, a, beta)


# ---------------------------------------------------------------------------
# the chunked form (independent path) equals the recurrence
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("variant", [GLA, GDN])
@pytest.mark.parametrize("C", [1, 16, 64, 150])
def test_chunked_equals_recurrence(variant, C):
    rng = np.random.default_rng(10 + C)
    q, k, v, alpha, beta, S0 = _rand(rng, 1, 150, 2, 16, 12)
    o1, S1 = oracle.recurrence(variant, q, k, v, alpha, beta if variant == GDN else None, S0)
    o2, S2 = chunked(variant, q, k, v, alpha, beta if variant == GDN else None, S0, C=C)
    scale_o = np.abs(o1).max()
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12 * scale_o * 10)
    np.testing.assert_allclose(S2, S1, rtol=0, atol=1e-12 * np.abs(S1).max() * 10)


def test_whole_sequence_chunk_is_one_triangular_solve():
    """C = T: the delta-rule values are one forward substitution (I + A) U = rhs;
    solving that system with numpy's general solver gives the same outputs."""
    rng = np.random.default_rng(11)
    T = 24
    q, k, v, alpha, beta, S0 = _rand(rng, 1, T, 1, 6, 5)
    Q, K, V, a, b, S = q[0, :, 0], k[0, :, 0], v[0, :, 0], alpha[0, :, 0], beta[0, :, 0], S0[0, 0]
    g = np.cumsum(np.log(a))
    gam = np.exp(g)
    A = np.zeros((T, T))
    for i in range(T):
        for j in range(i):
            A[i, j] = b[i] * np.exp(g[i] - g[j]) * (K[i] @ K[j])
    U = np.linalg.solve(np.eye(T) + A, b[:, None] * V - (b * gam)[:, None] * (K @ S))
    D = np.tril(np.exp(g[:, None] - g[None, :]))
    O = gam[:, None] * (Q @ S) + ((Q @ K.T) * D) @ U
    o1, _ = oracle.recurrence(GDN, q, k, v, alpha, beta, S0)
    np.testing.assert_allclose(O, o1[0, :, 0], rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------------------
# the page's worked example and segment invariants
# ---------------------------------------------------------------------------

def test_worked_example_recurrent_equals_chunked():
    with open(os.path.join(GOLDEN, "worked_example_gla.json")) as f:
        gold = json.load(f)
    ex = inputs.worked_example()
    q, k, v, alpha = (ex[n].double().numpy() for n in ("q", "k", "v", "alpha"))
    assert q.shape == (1, gold["T"], 1, gold["DK"])
    o1, S1 = oracle.recurrence(GLA, q, k, v, alpha)
    o2, S2 = chunked(GLA, q, k, v, alpha, C=gold["C"])
    assert np.allclose(o1, o2, atol=gold["atol"]) == gold["outputs_allclose"]
    assert np.allclose(S1, S2, atol=gold["atol"]) == gold["final_state_allclose"]
    # the state has DK x DV numbers; the KV cache of the same length would have T x (DK + DV)
    assert S1[0, 0].size == gold["state_numbers"]
    assert gold["T"] * (gold["DK"] + gold["DV"]) == gold["kv_numbers"]


@pytest.mark.parametrize("variant", [GLA, GDN])
def test_segmented_prefill_equals_one_shot(variant):
    """Handing S_T and the conv cache of one segment to the next equals one pass
    (section "Checking on a real model": three-segment prefill)."""
    rng = np.random.default_rng(20 + variant)
    q, k, v, alpha, beta, S0 = _rand(rng, 2, 45, 2, 8, 8)
    Cch = 2 * (8 + 8 + 8)
    w = rng.standard_normal((Cch, 4)) / 2
    be = beta if variant == GDN else None
    o_all, S_all, c_all = oracle.layer_prefill(variant, q, k, v, alpha, be, S0, w, None, True)
    S, cache, outs = S0, None, []
    for s, e in ((0, 20), (20, 22), (22, 45)):  # the middle one is shorter than the conv window
        o_seg, S, cache = oracle.layer_prefill(variant, q[:, s:e], k[:, s:e], v[:, s:e],
                                               alpha[:, s:e], None if be is None else be[:, s:e],
                                               S, w, cache, True)
        outs.append(o_seg)
    np.testing.assert_allclose(np.concatenate(outs, axis=1), o_all, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S, S_all, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(cache, c_all, rtol=0, atol=0)


def test_decode_steps_equal_prefill():
    """Prefill of the first 10 tokens then token-by-token decode from a pool
    slot gives the outputs of one prefill of all 16 tokens."""
    rng = np.random.default_rng(30)
    q, k, v, alpha, beta, S0 = _rand(rng, 1, 16, 2, 8, 8)
    Cch = 2 * 24
    w = rng.standard_normal((Cch, 4)) / 2
    o_all, S_all, c_all = oracle.layer_prefill(GDN, q, k, v, alpha, beta, S0, w, None, True,
                                               act_bf16=False)
    o_pre, S, cache = oracle.layer_prefill(GDN, q[:, :10], k[:, :10], v[:, :10], alpha[:, :10],
                                           beta[:, :10], S0, w, None, True, act_bf16=False)
    pool = np.zeros((4,) + S.shape[1:])
    conv_pool = np.zeros((4, 3, Cch))
    pool[2], conv_pool[2] = S[0], cache[0]
    for t in range(10, 16):
        o_t, pool, conv_pool = oracle.decode(GDN, q[:, t], k[:, t], v[:, t], alpha[:, t],
                                             beta[:, t], pool, [2], w, conv_pool, True,
                                             act_bf16=False)
        np.testing.assert_allclose(o_t[0], o_all[0, t], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(pool[2], S_all[0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(conv_pool[2], c_all[0], rtol=0, atol=0)
    assert not pool[[0, 1, 3]].any()


def test_spec_decode_states_are_prefix_states():
    """The state kept for draft position i is the state after i+1 tokens;
    the source slot is left as it was."""
    rng = np.random.default_rng(31)
    q, k, v, alpha, beta, S0 = _rand(rng, 1, 4, 2, 8, 8)
    pool = np.zeros((6, 2, 8, 8))
    pool[1] = S0[0]
    o, pool2, _ = oracle.spec_decode(GDN, q, k, v, alpha, beta, pool, [1], [[5, 0, 3, 2]],
                                     act_bf16=False)
    _, _, states = oracle.recurrence(GDN, q, k, v, alpha, beta, S0, return_states=True)
    for i, slot in enumerate([5, 0, 3, 2]):
        np.testing.assert_array_equal(pool2[slot], states[0, i])
    np.testing.assert_array_equal(pool2[1], S0[0])
    assert not pool2[4].any()


# ---------------------------------------------------------------------------
# front end pieces against library routines
# ---------------------------------------------------------------------------

def test_causal_conv_matches_torch_conv1d():
    rng = np.random.default_rng(40)
    B, T, Cch = 2, 11, 6
    x = rng.standard_normal((B, T, Cch))
    w = rng.standard_normal((Cch, 4))
    cache = rng.standard_normal((B, 3, Cch))
    y, cout = oracle.causal_conv(x, w, cache)
    hist = torch.from_numpy(np.concatenate([cache, x], axis=1)).permute(0, 2, 1)  # [B,Cch,T+3]
    ref = torch.nn.functional.conv1d(hist, torch.from_numpy(w)[:, None, :], groups=Cch)
    np.testing.assert_allclose(y, ref.permute(0, 2, 1).numpy(), rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(cout, np.concatenate([cache, x], axis=1)[:, -3:])
    # fresh sequence: zero history, i.e. left padding of 3
    y0, _ = oracle.causal_conv(x, w, None)
    ref0 = torch.nn.functional.conv1d(torch.from_numpy(x).permute(0, 2, 1),
                                      torch.from_numpy(w)[:, None, :], padding=3, groups=Cch)
    np.testing.assert_allclose(y0, ref0[..., :T].permute(0, 2, 1).numpy(), rtol=1e-13, atol=1e-13)


def test_conv_cache_short_segment_mixes_history():
    """T < 3: the new cache keeps the newest old inputs, then the new ones."""
    x = np.arange(1, 3, dtype=np.float64).reshape(1, 2, 1)  # x_0 = 1, x_1 = 2
    cache = np.array([[[10.0], [20.0], [30.0]]])
    _, cout = oracle.causal_conv(x, np.ones((1, 4)), cache)
    np.testing.assert_array_equal(cout[0, :, 0], [30.0, 1.0, 2.0])


def test_l2norm_and_bf16_rounding():
    rng = np.random.default_rng(41)
    x = rng.standard_normal((5, 16)) * 3
    y = oracle.l2norm_rows(x)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1) /
                               np.sqrt((x ** 2).sum(-1) + oracle.L2_EPS), rtol=1e-14)
    f32 = rng.standard_normal(4000).astype(np.float32) * 100
    expect = torch.from_numpy(f32).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(oracle.round_bf16(f32.astype(np.float64)), expect)


# ---------------------------------------------------------------------------
# the single-precision front end (bf16 activations): the same definitions
# evaluated in float, checked against the double-precision ones
# ---------------------------------------------------------------------------

U32 = 2.0 ** -24  # unit roundoff of float


def _bf16_exact(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).double().numpy()


def test_single_precision_conv_is_double_conv_rounded():
    rng = np.random.default_rng(42)
    B, T, Cch = 2, 37, 24
    x = _bf16_exact(rng.standard_normal((B, T, Cch)))
    w = rng.standard_normal((Cch, 4)).astype(np.float32).astype(np.float64)
    cache = _bf16_exact(rng.standard_normal((B, 3, Cch)))
    y32, c32 = oracle.causal_conv(x, w, cache, single=True)
    y64, c64 = oracle.causal_conv(x, w, cache)
    np.testing.assert_array_equal(c32, c64)
    hist = np.concatenate([cache, x], axis=1)
    absp = sum(np.abs(w[:, j]) * np.abs(hist[:, j:j + T]) for j in range(4))
    # 1 rounded product and 3 fused multiply-adds: at most 4 units of roundoff of sum |w x|
    assert (np.abs(y32 - y64) <= 4 * U32 * absp).all()
    assert (y32 == y32.astype(np.float32)).all()  # float values
    # small integers: every product and partial sum is exact in float
    xi = rng.integers(-8, 9, (1, 9, 5)).astype(np.float64)
    wi = rng.integers(-8, 9, (5, 4)).astype(np.float64)
    np.testing.assert_array_equal(oracle.causal_conv(xi, wi, single=True)[0], oracle.causal_conv(xi, wi)[0])


def test_single_precision_conv_fuses_the_later_taps():
    """A fused multiply-add rounds the exact w x + acc once, so a result that
    fits a float comes out exact even when the product alone does not:
    1 * (-1) + (1 + 2^-12)^2 = 2^-11 + 2^-24, while the rounded product
    (a tie, to even: 1 + 2^-11) would leave 2^-11.  The same holds for every
    later tap; the first tap is a plain rounded product."""
    e = 1.0 + 2.0 ** -12
    exact = 2.0 ** -11 + 2.0 ** -24
    for j in (1, 2, 3):
        x = np.zeros((1, 4, 1))
        w = np.zeros((1, 4))
        # output at t = 3 reads x_0 .. x_3 with taps 0 .. 3; tap 0 gives -1, tap j gives e^2
        x[0, 0, 0], w[0, 0] = -1.0, 1.0
        x[0, j, 0], w[0, j] = e, e
        y32 = oracle.causal_conv(x, w, single=True)[0]
        assert y32[0, 3, 0] == exact, j
    # the first tap alone is the rounded product: (1 + 2^-12)^2 -> 1 + 2^-11
    x = np.zeros((1, 4, 1)); w = np.zeros((1, 4))
    x[0, 0, 0], w[0, 0] = e, e
    assert oracle.causal_conv(x, w, single=True)[0][0, 3, 0] == 1.0 + 2.0 ** -11


def test_single_precision_l2norm_is_double_l2norm_rounded():
    rng = np.random.default_rng(43)
    for d in (16, 32, 64, 128):
        x = rng.standard_normal((7, d)).astype(np.float32).astype(np.float64) * 3
        y32 = oracle.l2norm_rows(x, single=True)
        y64 = oracle.l2norm_rows(x)
        assert (np.abs(y32 - y64) <= (np.log2(d) + 6) * U32 * np.abs(y64).max(axis=-1, keepdims=True)).all()


def test_single_precision_sum_of_squares_keeps_small_terms():
    """Pairwise summation: 127 squares of 2^-26 beside one square of 1 are not
    lost (added one by one to 1 in float, each would round away), so the
    normalised 1 comes out below 1 / sqrt(1 + eps)."""
    x = np.full((1, 128), 2.0 ** -13)
    x[0, 0] = 1.0
    y = oracle.l2norm_rows(x, single=True)
    swallowed = np.float32(1.0) / np.sqrt(np.float32(1.0) + np.float32(oracle.L2_EPS))
    assert y[0, 0] < swallowed
    np.testing.assert_allclose(y, oracle.l2norm_rows(x), rtol=4 * U32)


def test_single_precision_front_end_rounds_like_double_except_at_ties():
    """Conv, L2 norm and the rounding to bf16: the bf16 values agree with the
    double-precision front end except where the exact value lies within float
    rounding of a bf16 rounding boundary (there either neighbour is right)."""
    B, H, T, d = 2, 3, 50, 128
    ex = inputs.gdn_prefill(B, H, T, d, seed=44)
    q, k, v, w = (ex[n].double().numpy() for n in ("q", "k", "v", "conv_w"))
    q32, k32, v32, _ = oracle.frontend(q, k, v, w, None, True, act_bf16=True)
    q64, k64, v64, _ = oracle.frontend(q, k, v, w, None, True, act_bf16=False)  # unrounded, double
    for a32, a64 in ((q32, q64), (k32, k64), (v32, v64)):
        r64 = oracle.round_bf16(a64)
        diff = a32 != r64
        assert diff.mean() < 1e-3
        # a differing element sits next to the midpoint of its two bf16
        # neighbours, within float rounding of the terms that produced it (a
        # small result of a cancelling conv carries the absolute error of its
        # larger terms)
        lo, hi = np.minimum(a32, r64)[diff], np.maximum(a32, r64)[diff]
        mid = (lo + hi) / 2
        assert (np.abs(a64[diff] - mid) <= 1e-5 * np.abs(a64[diff]) + 1e-6 * np.abs(a64).max()).all()


# ---------------------------------------------------------------------------
# grouped q / k heads (the SSD form: state 128, head dim 64, shared B and C)
# ---------------------------------------------------------------------------

def test_grouped_heads_match_bruteforce_per_head():
    """Four heads, two q / k heads: head h is the brute-force gated linear
    attention on q / k head h // 2, with a rectangular (d_k = 8, d_v = 5) state."""
    rng = np.random.default_rng(9)
    q, k, _, _, _, _ = _rand(rng, 1, 15, 2, 8, 5)
    _, _, v, alpha, _, S0 = _rand(rng, 1, 15, 4, 8, 5)
    o, S = oracle.recurrence(GLA, q, k, v, alpha, S0=S0)
    for h in range(4):
        ob, Sb = _gla_bruteforce(q[0, :, h // 2], k[0, :, h // 2], v[0, :, h], alpha[0, :, h], S0[0, h])
        np.testing.assert_allclose(o[0, :, h], ob, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(S[0, h], Sb, rtol=1e-12, atol=1e-12)


def test_heads_of_one_group_agree_and_groups_differ():
    """With the same v and alpha for every head, the heads that share a q / k
    head give identical outputs and heads of different groups do not: this
    fixes which heads form a group (consecutive ones)."""
    rng = np.random.default_rng(10)
    q, k, v1, a1, _, _ = _rand(rng, 1, 12, 3, 6, 4, s0=False)
    v = np.repeat(v1[:, :, :1], 6, axis=2)
    alpha = np.repeat(a1[:, :, :1], 6, axis=2)
    o, _ = oracle.recurrence(GLA, q, k, v, alpha)
    for g in range(3):
        np.testing.assert_array_equal(o[0, :, 2 * g], o[0, :, 2 * g + 1])
    assert not np.allclose(o[0, :, 1], o[0, :, 2])
    assert not np.allclose(o[0, :, 3], o[0, :, 4])
