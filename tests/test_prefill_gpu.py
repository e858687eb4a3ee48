"""GPU parity of prefill against the oracle.

"Inference for linear attention and hybrid architectures", section "Two ways
to write the same computation": the chunked form equals the recurrence, and a
prompt prefilled in segments (the state handed from one segment to the next)
equals one prefill; section "Checking on a real model" checks the same on a
real model with a three-segment prefill.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_02_gb300 import GDN, GLA, glinattn_prefill, inputs
from gated_deltanet_02_gb300.glinattn import prefill_workspace_size
from oracle.chunked import chunked

from helpers import TOL_F32, TOL_O_BF16, TOL_S_BF16, NT, f64, relerr, to

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _gpu_prefill(g, variant, conv, S0=None, conv_in=None, out_dtype=torch.float32):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, S, c = glinattn_prefill(g["q"], g["k"], g["v"], g["alpha"], g.get("beta"), S0,
                               variant=variant, conv_w=g.get("conv_w") if conv else None,
                               conv_in=conv_in, qk_l2norm=conv, out_dtype=out_dtype,
                               dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return o, S, c


def _oracle_prefill(ex, variant, conv, S0=None, conv_in=None, sl=slice(None), heads=slice(None)):
    def cut(t):
        return None if t is None else f64(t[:, sl, heads] if t.dim() >= 3 else t)
    q, k, v = cut(ex["q"]), cut(ex["k"]), cut(ex["v"])
    a = cut(ex["alpha"])
    b = cut(ex.get("beta")) if variant == GDN else None
    return oracle.layer_prefill(variant, q, k, v, a, b, S0, f64(ex.get("conv_w")) if conv else None,
                                conv_in, conv, nthreads=NT)


def test_worked_example_fp32():
    """T=64, d=16, fp32: the GPU matches the oracle to 1e-5 and, like the
    page's chunked form, agrees with the recurrence under allclose(atol=1e-5)."""
    ex = inputs.worked_example()
    g = to(ex, DEV)
    o, S, _ = _gpu_prefill(g, GLA, False)
    o_ref, S_ref = oracle.recurrence(GLA, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]))
    assert relerr(o, o_ref) <= TOL_F32 and relerr(S, S_ref) <= TOL_F32
    o_c, S_c = chunked(GLA, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]), C=ex["chunk"])
    assert np.allclose(f64(o), o_c, atol=1e-5) and np.allclose(f64(S), S_c, atol=1e-5)


@pytest.mark.parametrize("T", [1, 63, 64, 200, 300])
def test_gla_bf16_small(T):
    ex = inputs.gla_prefill(2, 3, T, 128, seed=T, s0_std=0.05)
    g = to(ex, DEV)
    o, S, _ = _gpu_prefill(g, GLA, False, S0=g["S0"])
    o_ref, S_ref, _ = _oracle_prefill(ex, GLA, False, S0=f64(ex["S0"]))
    assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(S, S_ref) <= TOL_S_BF16


@pytest.mark.parametrize("T", [2, 64, 130, 257])
def test_gdn_bf16_conv_small(T):
    ex = inputs.gdn_prefill(2, 2, T, 128, seed=T)
    g = to(ex, DEV)
    o, S, c = _gpu_prefill(g, GDN, True, S0=g["S0"])
    o_ref, S_ref, c_ref = _oracle_prefill(ex, GDN, True, S0=f64(ex["S0"]))
    assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(S, S_ref) <= TOL_S_BF16
    assert np.array_equal(f64(c), c_ref)


@pytest.mark.parametrize("d", [16, 32, 64])
def test_other_head_sizes(d):
    ex = inputs.gdn_prefill(1, 2, 77, d, seed=d)
    g = to(ex, DEV)
    o, S, c = _gpu_prefill(g, GDN, True, S0=g["S0"])
    o_ref, S_ref, c_ref = _oracle_prefill(ex, GDN, True, S0=f64(ex["S0"]))
    assert relerr(o, o_ref) <= TOL_O_BF16 and relerr(S, S_ref) <= TOL_S_BF16
    assert np.array_equal(f64(c), c_ref)


@pytest.mark.parametrize("variant", [GLA, GDN])
def test_segmented_equals_one_shot(variant):
    """Three ragged segments carrying S and the conv cache equal one call."""
    T = 333
    ex = (inputs.gdn_prefill if variant == GDN else inputs.gla_prefill)(1, 2, T, 128, seed=21)
    g = to(ex, DEV)
    conv = variant == GDN
    o_all, S_all, c_all = _gpu_prefill(g, variant, conv, S0=g.get("S0"))
    S, c, outs = g.get("S0"), None, []
    for s, e in ((0, 70), (70, 72), (72, T)):
        seg = {k: (v[:, s:e].contiguous() if k in ("q", "k", "v", "alpha", "beta") and v is not None
                   else v) for k, v in g.items()}
        o, S, c = _gpu_prefill(seg, variant, conv, S0=S, conv_in=c)
        outs.append(o)
    o_seg = torch.cat(outs, dim=1)
    o_ref, S_ref, c_ref = _oracle_prefill(ex, variant, conv, S0=f64(ex.get("S0")))
    assert relerr(o_seg, o_ref) <= TOL_O_BF16 and relerr(S, S_ref) <= TOL_S_BF16
    assert relerr(o_seg, f64(o_all)) <= TOL_O_BF16 and relerr(S, f64(S_all)) <= TOL_S_BF16
    if conv:
        assert torch.equal(c, c_all)
        assert np.array_equal(f64(c), c_ref)


def test_zero_length_segment_hands_state_on():
    ex = inputs.gdn_prefill(2, 2, 0, 128, seed=3)
    g = to(ex, DEV)
    cin = torch.randn(2, 3, 2 * 3 * 128, device=DEV).to(torch.bfloat16)
    o, S, c = _gpu_prefill(g, GDN, True, S0=g["S0"], conv_in=cin)
    assert o.numel() == 0
    assert torch.equal(S, g["S0"]) and torch.equal(c, cin)


def test_bf16_output():
    ex = inputs.gla_prefill(1, 2, 150, 128, seed=5)
    g = to(ex, DEV)
    o, _, _ = _gpu_prefill(g, GLA, False, out_dtype=torch.bfloat16)
    o_ref, _, _ = _oracle_prefill(ex, GLA, False)
    err = np.abs(f64(o) - o_ref)
    assert (err <= np.abs(o_ref) * 2.0 ** -8 + TOL_O_BF16 * np.abs(o_ref).max()).all()


def _full_all_units(ex, variant, conv):
    """Run the full workload on the GPU and check every (b, h) unit in full
    against the oracle (run over the whole batch on all host cores)."""
    g = to(ex, DEV)
    o, S, c = _gpu_prefill(g, variant, conv, S0=g.get("S0"), out_dtype=torch.float32)
    del g
    cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in ex.items()}
    S0 = None if cpu.get("S0") is None else f64(cpu["S0"])
    o_ref, S_ref, c_ref = oracle.layer_prefill(
        variant, f64(cpu["q"]), f64(cpu["k"]), f64(cpu["v"]), f64(cpu["alpha"]),
        f64(cpu.get("beta")) if variant == GDN else None, S0, f64(cpu.get("conv_w")) if conv else None,
        None, conv, nthreads=NT)
    o64, S64 = f64(o), f64(S)
    B, H = S64.shape[:2]
    for b in range(B):
        for h in range(H):
            assert relerr(o64[b, :, h], o_ref[b, :, h]) <= TOL_O_BF16, (b, h)
            assert relerr(S64[b, h], S_ref[b, h]) <= TOL_S_BF16, (b, h)
    if conv:
        assert np.array_equal(f64(c), c_ref)


def test_gla_prefill_full_size_all_units():
    """B=4, H=16, T=4096, d=128, bf16: all 64 (batch, head) units in full."""
    ex = inputs.gla_prefill(4, 16, 4096, 128, seed=0, device=DEV)
    _full_all_units(ex, GLA, False)


def test_gdn_prefill_full_size_all_units():
    """B=2, H=16, T=8192, d=128, conv + L2 norm, S0 ~ N(0, 0.01): all 32 units."""
    ex = inputs.gdn_prefill(2, 16, 8192, 128, seed=0, device=DEV)
    _full_all_units(ex, GDN, True)


@pytest.mark.parametrize("variant", [GLA, GDN])
def test_strong_decay_pairwise_path(variant):
    """alpha ~ U(0.05, 0.2): a chunk's total decay is far below 2^-100, so the
    decay mask cannot be factored into row and column factors and every
    D_ij = 2^(g_i - g_j) is formed pairwise."""
    T = 200
    ex = (inputs.gdn_prefill if variant == GDN else inputs.gla_prefill)(1, 2, T, 128, seed=31)
    gen = torch.Generator().manual_seed(7)
    ex["alpha"] = (0.05 + 0.15 * torch.rand(ex["alpha"].shape, generator=gen)).to(ex["alpha"].dtype)
    g = to(ex, DEV)
    conv = variant == GDN
    o, S, _ = _gpu_prefill(g, variant, conv, S0=g.get("S0"))
    o_ref, S_ref, _ = _oracle_prefill(ex, variant, conv, S0=f64(ex.get("S0")))
    assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(S, S_ref) <= TOL_S_BF16


@pytest.mark.parametrize("variant", [GLA, GDN])
def test_more_units_than_sms(variant):
    """B=3, H=40: 240 GLA CTAs and 480 GDN scan CTAs, more than one wave."""
    ex = (inputs.gdn_prefill if variant == GDN else inputs.gla_prefill)(3, 40, 130, 128, seed=41)
    conv = variant == GDN
    heads = [(0, 0), (1, 17), (2, 39)]
    g = to(ex, DEV)
    o, S, _ = _gpu_prefill(g, variant, conv, S0=g.get("S0"))
    H, d = 40, 128
    for b, h in heads:
        sub = {k: (v[b:b + 1, :, h:h + 1] if k in ("q", "k", "v", "alpha", "beta") and v is not None
                   else v) for k, v in ex.items()}
        if conv:
            sub["conv_w"] = ex["conv_w"].view(3, H, d, 4)[:, h].reshape(3 * d, 4)
        S0 = None if ex.get("S0") is None else f64(ex["S0"][b:b + 1, h:h + 1])
        o_ref, S_ref, _ = _oracle_prefill(sub, variant, conv, S0=S0)
        assert relerr(o[b:b + 1, :, h:h + 1], o_ref) <= TOL_O_BF16, (b, h)
        assert relerr(S[b:b + 1, h:h + 1], S_ref) <= TOL_S_BF16, (b, h)


# ------------------------------------------------------- random shapes ---------
def _shapes(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        out.append((int(rng.integers(1, 4)), int(rng.integers(1, 6)), int(rng.integers(1, 700)),
                    bool(rng.integers(0, 2)), bool(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("B,H,T,with_s0,bf16_out", _shapes(8, 2024))
@pytest.mark.parametrize("variant", [GLA, GDN])
def test_random_shapes_match_oracle(variant, B, H, T, with_s0, bf16_out):
    """Seeded random batch, head count and length (ragged last chunks, one to
    five heads, start state or none, bf16 or fp32 outputs) for both forms at
    d = 128, against the oracle."""
    conv = variant == GDN
    maker = inputs.gdn_prefill if conv else inputs.gla_prefill
    ex = maker(B, H, T, 128, seed=B * 1000 + H * 100 + T, **({} if conv else {"s0_std": 0.05}))
    g = to(ex, DEV)
    S0 = g.get("S0") if with_s0 else None
    o, S, c = _gpu_prefill(g, variant, conv, S0=S0, out_dtype=torch.bfloat16 if bf16_out else torch.float32)
    o_ref, S_ref, c_ref = _oracle_prefill(ex, variant, conv, S0=f64(ex["S0"]) if with_s0 else None)
    if bf16_out:
        err = np.abs(f64(o) - o_ref)
        assert (err <= np.abs(o_ref) * 2.0 ** -8 + TOL_O_BF16 * np.abs(o_ref).max()).all()
    else:
        assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(S, S_ref) <= TOL_S_BF16
    if conv:
        assert np.array_equal(f64(c), c_ref)


# ------------------------------------------------ prepared activations ---------
def _prepared_qk(ws, B, H, T):
    """q', k' as the chunked Gated DeltaNet kernels leave them in the
    workspace: bf16 rows [B*H, Tp, 128] (Tp = T rounded up to the 64-token
    chunk), q' first, k' at the next 256-byte boundary."""
    Tp = (T + 63) // 64 * 64
    n = B * H * Tp * 128 * 2
    kq = ws[:n].view(torch.bfloat16).view(B, H, Tp, 128)[:, :, :T]
    off = (n + 255) // 256 * 256
    kk = ws[off:off + n].view(torch.bfloat16).view(B, H, Tp, 128)[:, :, :T]
    return f64(kq).transpose(0, 2, 1, 3), f64(kk).transpose(0, 2, 1, 3)


@pytest.mark.parametrize("B,H,T,with_conv_in", [(3, 3, 418, False), (2, 4, 1000, True), (1, 2, 4096, False)])
def test_prepared_activations_bit_exact(B, H, T, with_conv_in):
    """The bf16 q' and k' the tensor-core passes read (conv, L2 norm, rounding)
    equal the oracle's front end bit for bit: the rounding to bf16 is a
    decision both sides take in single precision, every product and sum
    rounded on its own."""
    ex = inputs.gdn_prefill(B, H, T, 128, seed=31 * T + H)
    g = to(ex, DEV)
    conv_in = None
    if with_conv_in:
        gen = torch.Generator().manual_seed(T)
        conv_in = torch.randn((B, 3, 3 * H * 128), generator=gen).to(torch.bfloat16)
    ws = torch.zeros(int(prefill_workspace_size(B, T, H, 128)), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    glinattn_prefill(g["q"], g["k"], g["v"], g["alpha"], g["beta"], None, variant=GDN, conv_w=g["conv_w"],
                     conv_in=None if conv_in is None else conv_in.to(DEV), qk_l2norm=True,
                     out_dtype=torch.float32, workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    qp, kp = _prepared_qk(ws, B, H, T)
    qf, kf, _, _ = oracle.frontend(f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["conv_w"]),
                                   f64(conv_in), True, True)
    assert np.array_equal(qp, qf), int((qp != qf).sum())
    assert np.array_equal(kp, kf), int((kp != kf).sum())
