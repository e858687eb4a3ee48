"""GPU parity of the hot path on the degenerate cases the pages fix.

"Inference for linear attention and hybrid architectures", section "Two ways
to write the same computation":

* alpha = 1 removes the decay: gated linear attention becomes unnormalised
  causal linear attention, O = tril(Q K^T) V (+ Q S0), and the row / column
  decay factors of the chunked kernels are all 1;
* the delta rule erases the old content along k_t before writing the new one:
  beta = 0 leaves pure decay (o_t = gamma_t q_t S0, S_T = gamma_T S0) and
  beta = 1 with a unit key stores v_t exactly along k_t (k_t S_t = v_t);
* a gate outside (0, 1] (zero, NaN, above one) is a precondition violation:
  the unit raises GLINATTN_DEV_BAD_GATE and writes nothing, while every other
  unit of the same launch is computed as usual.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_02_gb300 import GDN, GLA, glinattn_decode, glinattn_prefill, inputs
from gated_deltanet_02_gb300.glinattn import DEV_BAD_GATE

from helpers import TOL_O_BF16, TOL_S_BF16, NT, f64, relerr, to

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _prefill(g, variant, conv, S0=None, o=None, S_T=None):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, S, c = glinattn_prefill(g["q"], g["k"], g["v"], g["alpha"], g.get("beta"), S0, variant=variant,
                               conv_w=g.get("conv_w") if conv else None, qk_l2norm=conv,
                               out_dtype=torch.float32, dev_status=status, o=o, S_T=S_T)
    torch.cuda.synchronize()
    return o, S, c, int(status.item())


def _oracle(ex, variant, conv, S0=None):
    return oracle.layer_prefill(variant, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]),
                                f64(ex.get("beta")) if variant == GDN else None, S0,
                                f64(ex.get("conv_w")) if conv else None, None, conv, nthreads=NT)


# ---------------------------------------------------------------- alpha = 1 --

@pytest.mark.parametrize("T", [64, 200])
def test_gla_prefill_alpha_one_is_causal_linear_attention(T):
    """alpha = 1: every decay factor is 1 and o = tril(Q K^T) V + Q S0."""
    ex = inputs.gla_prefill(2, 3, T, 128, seed=50 + T, s0_std=0.05)
    ex["alpha"] = torch.ones_like(ex["alpha"])
    o, S, _, st = _prefill(to(ex, DEV), GLA, False, S0=ex["S0"].to(DEV))
    assert st == 0
    o_ref, S_ref, _ = _oracle(ex, GLA, False, S0=f64(ex["S0"]))
    assert relerr(o, o_ref) <= TOL_O_BF16 and relerr(S, S_ref) <= TOL_S_BF16
    # the textbook form, per (batch, head)
    q, k, v, S0 = f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["S0"])
    for b in range(2):
        for h in range(3):
            Q, K, V = q[b, :, h], k[b, :, h], v[b, :, h]
            closed = np.tril(Q @ K.T) @ V + Q @ S0[b, h]
            assert relerr(o[b, :, h], closed) <= TOL_O_BF16, (b, h)
            assert relerr(S[b, h], S0[b, h] + K.T @ V) <= TOL_S_BF16, (b, h)


def test_gdn_prefill_alpha_one():
    ex = inputs.gdn_prefill(2, 2, 200, 128, seed=61)
    ex["alpha"] = torch.ones_like(ex["alpha"])
    o, S, c, st = _prefill(to(ex, DEV), GDN, True, S0=ex["S0"].to(DEV))
    assert st == 0
    o_ref, S_ref, c_ref = _oracle(ex, GDN, True, S0=f64(ex["S0"]))
    assert relerr(o, o_ref) <= TOL_O_BF16 and relerr(S, S_ref) <= TOL_S_BF16
    assert np.array_equal(f64(c), c_ref)


# ------------------------------------------------------------- beta = 0, 1 --

def test_gdn_prefill_beta_zero_is_pure_decay():
    """beta = 0: nothing is erased or written; o_t = gamma_t q'_t S0 and
    S_T = gamma_T S0 (q' the front end's output)."""
    B, H, T, d = 1, 2, 200, 128
    ex = inputs.gdn_prefill(B, H, T, d, seed=62, s0_std=0.05)
    ex["beta"] = torch.zeros_like(ex["beta"])
    o, S, _, st = _prefill(to(ex, DEV), GDN, True, S0=ex["S0"].to(DEV))
    assert st == 0
    o_ref, S_ref, _ = _oracle(ex, GDN, True, S0=f64(ex["S0"]))
    assert relerr(o, o_ref) <= TOL_O_BF16 and relerr(S, S_ref) <= TOL_S_BF16
    qf, _, _, _ = oracle.frontend(f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["conv_w"]), None, True)
    gam = np.cumprod(f64(ex["alpha"]), axis=1)  # [B, T, H]
    S0 = f64(ex["S0"])
    for h in range(H):
        decay_o = gam[0, :, h, None] * (qf[0, :, h] @ S0[0, h])
        assert relerr(o[0, :, h], decay_o) <= TOL_O_BF16, h
        assert relerr(S[0, h], gam[0, -1, h] * S0[0, h]) <= TOL_S_BF16, h


def test_gdn_prefill_beta_one_stores_v_along_k():
    """beta = 1 with unit keys: after the last token, k'_T S_T = v'_T."""
    B, H, T, d = 1, 2, 130, 128
    ex = inputs.gdn_prefill(B, H, T, d, seed=63)
    ex["beta"] = torch.ones_like(ex["beta"])
    o, S, _, st = _prefill(to(ex, DEV), GDN, True, S0=ex["S0"].to(DEV))
    assert st == 0
    o_ref, S_ref, _ = _oracle(ex, GDN, True, S0=f64(ex["S0"]))
    assert relerr(o, o_ref) <= TOL_O_BF16 and relerr(S, S_ref) <= TOL_S_BF16
    _, kf, vf, _ = oracle.frontend(f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["conv_w"]), None, True)
    Sg = f64(S)
    for h in range(H):
        kt, vt = kf[0, -1, h], vf[0, -1, h]
        # k' S_t - v' = (|k'|^2 - 1)(v' - alpha k' S_{t-1}); |k'|^2 - 1 is only the
        # bf16 rounding of the normalised key, so the read-back is v' to ~1e-2
        assert np.abs(kt @ Sg[0, h] - vt).max() <= 1e-2 * np.abs(vt).max(), h


@pytest.mark.parametrize("variant,alpha_one,beta", [(GLA, True, None), (GDN, True, None),
                                                    (GDN, False, 0.0), (GDN, False, 1.0)])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_degenerate_gates(variant, alpha_one, beta, d):
    ex = inputs.gdn_decode(12, 3, d, 40, seed=70 + d, variant_gdn=variant == GDN)
    if alpha_one:
        ex["alpha"] = torch.ones_like(ex["alpha"])
    if beta is not None:
        ex["beta"] = torch.full_like(ex["beta"], beta)
    conv = variant == GDN
    g = to(ex, DEV)
    pool, cpool = g["pool"].clone(), g["conv_pool"].clone() if conv else None
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = glinattn_decode(g["q"], g["k"], g["v"], g["alpha"], g["beta"], pool, g["slot_ids"], variant=variant,
                        conv_w=g["conv_w"] if conv else None, conv_pool=cpool, qk_l2norm=conv,
                        out_dtype=torch.float32, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref, pool_ref, _ = oracle.decode(variant, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]),
                                       f64(ex["beta"]), f64(ex["pool"]), ex["slot_ids"].tolist(),
                                       f64(ex["conv_w"]) if conv else None,
                                       f64(ex["conv_pool"]) if conv else None, conv)
    sl = ex["slot_ids"].long()
    assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(pool[sl.to(DEV)], pool_ref[sl.numpy()]) <= TOL_S_BF16
    if beta == 0.0:  # pure decay of the slot's state
        a = f64(ex["alpha"])
        want = a[:, :, None, None] * f64(ex["pool"])[sl.numpy()]
        assert relerr(pool[sl.to(DEV)], want) <= TOL_S_BF16


# ----------------------------------------------------------------- bad gate --

@pytest.mark.parametrize("bad", [0.0, float("nan"), 1.5])
@pytest.mark.parametrize("variant", [GLA, GDN])
def test_prefill_bad_gate_flags_and_skips_one_unit(variant, bad):
    """One gate of unit (b=1, h=1) is invalid: that unit writes nothing (its o,
    S_T and conv cache keep their sentinel values), the launch raises
    GLINATTN_DEV_BAD_GATE, and every other unit matches the oracle.  T = 200
    keeps gated linear attention on the unsplit kernel."""
    B, H, T, d = 2, 3, 200, 128
    conv = variant == GDN
    ex = (inputs.gdn_prefill if conv else inputs.gla_prefill)(B, H, T, d, seed=80)
    ex["alpha"] = ex["alpha"].clone()
    ex["alpha"][1, 77, 1] = bad
    g = to(ex, DEV)
    o = torch.full((B, T, H, d), 7.0, dtype=torch.float32, device=DEV)
    S_T = torch.full((B, H, d, d), -3.0, dtype=torch.float32, device=DEV)
    S0 = g.get("S0")
    o, S, c, st = _prefill(g, variant, conv, S0=S0, o=o, S_T=S_T)
    assert st == DEV_BAD_GATE
    assert bool((o[1, :, 1] == 7.0).all()) and bool((S[1, 1] == -3.0).all())
    for b in range(B):
        for h in range(H):
            if (b, h) == (1, 1):
                continue
            sub = {k: (v[b:b + 1, :, h:h + 1] if k in ("q", "k", "v", "alpha", "beta") and v is not None else v)
                   for k, v in ex.items()}
            if conv:
                sub["conv_w"] = ex["conv_w"].view(3, H, d, 4)[:, h].reshape(3 * d, 4)
            S0h = None if ex.get("S0") is None else f64(ex["S0"][b:b + 1, h:h + 1])
            o_ref, S_ref, c_ref = _oracle(sub, variant, conv, S0=S0h)
            assert relerr(o[b:b + 1, :, h:h + 1], o_ref) <= TOL_O_BF16, (b, h)
            assert relerr(S[b:b + 1, h:h + 1], S_ref) <= TOL_S_BF16, (b, h)
