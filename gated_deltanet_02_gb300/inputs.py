"""Seeded synthetic inputs for the linear-attention layer.

This module draws random numbers and nothing else: it holds none of the
layer's arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it.  Every tensor comes from a ``torch.Generator`` seeded by the
caller, on the device the caller names.

Workloads (the distributions are those of the configurations this library is
measured on; "N(m, s)" means mean m, standard deviation s):

* ``worked_example``  -- gated linear attention, one head, T=64, d=16, fp32:
  q, k ~ N(0,1)/4, v ~ N(0,1), alpha = sigmoid(N(0,1) + 3), drawn in that order
  from seed 0 (the worked example of "Inference for linear attention and
  hybrid architectures", section "Two ways to write the same computation").
* ``gla_prefill``     -- q, k ~ N(0,1)/sqrt(d), v ~ N(0,1) in bf16; alpha =
  sigmoid(N(0,1) + 3) fp32 per token and head; zero start state.
* ``gdn_prefill``     -- raw q, k with every row scaled to unit L2 norm and
  v ~ N(0,1), in bf16; beta = sigmoid(N(0,1)); alpha = sigmoid(N(0,1) + 3);
  conv weights N(0,1)/2 over the [q | k | v] channels; S0 ~ N(0, 0.01).
* ``gdn_decode``      -- N requests x H heads, one token each; a pool of P
  fp32 states ~ N(0, 0.01) and bf16 conv caches ~ N(0, 1); slot ids = the
  first N entries of a random permutation of the P slots.
* ``spec_drafts``     -- D draft tokens per request and an accepted prefix
  length drawn uniformly from 0..D.
* ``ssd_prefill`` / ``ssd_decode`` -- the SSD form of Mamba2 as gated linear
  attention: G groups of q / k heads (C and B) of size d_k = 128 (the state
  size) shared by H heads of value size d_v = 64 (the head dim); q, k ~
  N(0,1)/sqrt(d_k), v ~ N(0,1) in bf16, alpha = sigmoid(N(0,1) + 3).
* ``selective_scan_inputs`` -- Mamba's selective scan: x ~ N(0,1), delta ~
  N(-2,1), B, C ~ N(0,1), A = -exp(U(0,1)), h0 ~ N(0, 0.1) when asked.
* ``nla_prefill`` / ``nla_decode`` -- normalised kernelised linear attention:
  raw q, k, v ~ N(0,1) (the feature map is applied inside the layer); a start
  state ~ N(0, 0.05) and a positive start normaliser |N(0,1)| * 8 when asked.
"""
from __future__ import annotations

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, g, device, scale=1.0, dtype=torch.float32):
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(dtype)


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    """Scale each last-axis row to unit Euclidean length (input recipe)."""
    return x / x.norm(dim=-1, keepdim=True)


def worked_example(device="cpu"):
    """Seed 0, T=64, DK=DV=16, drawn in the page's order; shapes [1,T,1,d]."""
    T, DK, DV = 64, 16, 16
    g = _gen(0, device)
    q = torch.randn(T, DK, generator=g, device=device) / 4
    k = torch.randn(T, DK, generator=g, device=device) / 4
    v = torch.randn(T, DV, generator=g, device=device)
    alpha = torch.sigmoid(torch.randn(T, generator=g, device=device) + 3)
    return dict(q=q[None, :, None], k=k[None, :, None], v=v[None, :, None],
                alpha=alpha[None, :, None], chunk=16)


def gla_prefill(B, H, T, d, seed=0, device="cpu", dtype=torch.bfloat16, s0_std=0.0):
    g = _gen(seed, device)
    q = _randn((B, T, H, d), g, device, d ** -0.5, dtype)
    k = _randn((B, T, H, d), g, device, d ** -0.5, dtype)
    v = _randn((B, T, H, d), g, device, 1.0, dtype)
    alpha = torch.sigmoid(_randn((B, T, H), g, device) + 3.0)
    S0 = _randn((B, H, d, d), g, device, s0_std) if s0_std > 0 else None
    return dict(q=q, k=k, v=v, alpha=alpha, beta=None, S0=S0)


def gdn_prefill(B, H, T, d, seed=0, device="cpu", dtype=torch.bfloat16, s0_std=0.01,
                conv=True):
    g = _gen(seed, device)
    q = _unit_rows(_randn((B, T, H, d), g, device)).to(dtype)
    k = _unit_rows(_randn((B, T, H, d), g, device)).to(dtype)
    v = _randn((B, T, H, d), g, device, 1.0, dtype)
    beta = torch.sigmoid(_randn((B, T, H), g, device))
    alpha = torch.sigmoid(_randn((B, T, H), g, device) + 3.0)
    conv_w = _randn((3 * H * d, 4), g, device, 0.5) if conv else None
    S0 = _randn((B, H, d, d), g, device, s0_std) if s0_std > 0 else None
    return dict(q=q, k=k, v=v, alpha=alpha, beta=beta, S0=S0, conv_w=conv_w)


def gdn_decode(N, H, d, P, seed=0, device="cpu", dtype=torch.bfloat16, conv=True,
               variant_gdn=True):
    g = _gen(seed, device)
    pool = _randn((P, H, d, d), g, device, 0.01)
    conv_pool = _randn((P, 3, 3 * H * d), g, device, 1.0, dtype) if conv else None
    perm = torch.randperm(P, generator=g, device=device)
    slot_ids = perm[:N].to(torch.int32)
    if variant_gdn:
        q = _unit_rows(_randn((N, H, d), g, device)).to(dtype)
        k = _unit_rows(_randn((N, H, d), g, device)).to(dtype)
    else:
        q = _randn((N, H, d), g, device, d ** -0.5, dtype)
        k = _randn((N, H, d), g, device, d ** -0.5, dtype)
    v = _randn((N, H, d), g, device, 1.0, dtype)
    beta = torch.sigmoid(_randn((N, H), g, device)) if variant_gdn else None
    alpha = torch.sigmoid(_randn((N, H), g, device) + 3.0)
    conv_w = _randn((3 * H * d, 4), g, device, 0.5) if conv else None
    return dict(q=q, k=k, v=v, alpha=alpha, beta=beta, pool=pool, conv_pool=conv_pool,
                slot_ids=slot_ids, conv_w=conv_w)


def spec_drafts(N, D, H, d, seed=0, device="cpu", dtype=torch.bfloat16):
    """Draft-token inputs [N,D,H,*] and accepted prefix lengths a in 0..D."""
    g = _gen(seed, device)
    q = _unit_rows(_randn((N, D, H, d), g, device)).to(dtype)
    k = _unit_rows(_randn((N, D, H, d), g, device)).to(dtype)
    v = _randn((N, D, H, d), g, device, 1.0, dtype)
    beta = torch.sigmoid(_randn((N, D, H), g, device))
    alpha = torch.sigmoid(_randn((N, D, H), g, device) + 3.0)
    accept = torch.randint(0, D + 1, (N,), generator=g, device=device, dtype=torch.int32)
    return dict(q=q, k=k, v=v, alpha=alpha, beta=beta, accept=accept)


def ssd_prefill(B, H, G, T, dk=128, dv=64, seed=0, device="cpu", dtype=torch.bfloat16, s0_std=0.0):
    g = _gen(seed, device)
    q = _randn((B, T, G, dk), g, device, dk ** -0.5, dtype)
    k = _randn((B, T, G, dk), g, device, dk ** -0.5, dtype)
    v = _randn((B, T, H, dv), g, device, 1.0, dtype)
    alpha = torch.sigmoid(_randn((B, T, H), g, device) + 3.0)
    S0 = _randn((B, H, dk, dv), g, device, s0_std) if s0_std > 0 else None
    return dict(q=q, k=k, v=v, alpha=alpha, beta=None, S0=S0)


def ssd_decode(N, H, G, P, dk=128, dv=64, seed=0, device="cpu", dtype=torch.bfloat16, D=None):
    """One token (D=None) or D draft tokens per request, and a pool of P states."""
    g = _gen(seed, device)
    pool = _randn((P, H, dk, dv), g, device, 0.01)
    perm = torch.randperm(P, generator=g, device=device)
    slot_ids = perm[:N].to(torch.int32)
    lead = (N,) if D is None else (N, D)
    q = _randn(lead + (G, dk), g, device, dk ** -0.5, dtype)
    k = _randn(lead + (G, dk), g, device, dk ** -0.5, dtype)
    v = _randn(lead + (H, dv), g, device, 1.0, dtype)
    alpha = torch.sigmoid(_randn(lead + (H,), g, device) + 3.0)
    return dict(q=q, k=k, v=v, alpha=alpha, beta=None, pool=pool, slot_ids=slot_ids, perm=perm)


def nla_prefill(B, H, T, d, Hq=None, seed=0, device="cpu", dtype=torch.bfloat16, start=False, dv=None):
    g = _gen(seed, device)
    Hq = H if Hq is None else Hq
    dv = d if dv is None else dv
    q = _randn((B, T, Hq, d), g, device, 1.0, dtype)
    k = _randn((B, T, Hq, d), g, device, 1.0, dtype)
    v = _randn((B, T, H, dv), g, device, 1.0, dtype)
    S0 = _randn((B, H, d, dv), g, device, 0.05) if start else None
    z0 = _randn((B, H, d), g, device).abs() * 8.0 if start else None
    return dict(q=q, k=k, v=v, alpha=None, beta=None, S0=S0, z0=z0)


def nla_decode(N, H, d, P, Hq=None, seed=0, device="cpu", dtype=torch.bfloat16, D=None):
    """One token (D=None) or D draft tokens per request; pools of P states and
    positive normalisers."""
    g = _gen(seed, device)
    Hq = H if Hq is None else Hq
    pool = _randn((P, H, d, d), g, device, 0.05)
    zpool = _randn((P, H, d), g, device).abs() * 8.0
    perm = torch.randperm(P, generator=g, device=device)
    lead = (N,) if D is None else (N, D)
    q = _randn(lead + (Hq, d), g, device, 1.0, dtype)
    k = _randn(lead + (Hq, d), g, device, 1.0, dtype)
    v = _randn(lead + (H, d), g, device, 1.0, dtype)
    return dict(q=q, k=k, v=v, pool=pool, zpool=zpool, slot_ids=perm[:N].to(torch.int32), perm=perm)


def selective_scan_inputs(B, T, D, N, seed=0, device="cpu", dtype=torch.float32, start=False):
    """Mamba's selective scan: x ~ N(0,1), delta ~ N(-2,1) (softplus(delta)
    mostly in 0.05..0.5), B, C ~ N(0,1), A = -exp(U(0,1)) per channel and state
    index (the stable construction of the page's block); h0 ~ N(0, 0.1)."""
    g = _gen(seed, device)
    x = _randn((B, T, D), g, device, 1.0, dtype)
    delta = (_randn((B, T, D), g, device) - 2.0).to(dtype)
    Bm = _randn((B, T, N), g, device, 1.0, dtype)
    Cm = _randn((B, T, N), g, device, 1.0, dtype)
    A = -torch.exp(torch.rand((D, N), generator=g, device=device))
    h0 = _randn((B, D, N), g, device, 0.1) if start else None
    return dict(x=x, delta=delta, Bm=Bm, Cm=Cm, A=A, h0=h0)


def segment_lengths(T: int, fractions=(0.20, 0.35)):
    """Split T into segments of floor(f*T) tokens for each fraction, and the rest."""
    out = [int(T * f) for f in fractions]
    out.append(T - sum(out))
    return out
