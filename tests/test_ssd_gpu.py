"""GPU parity of the SSD form: gated linear attention with a 128 x 64 state
(state size 128, head dim 64) and q / k heads shared by groups of heads.

"Inference for linear attention and hybrid architectures", section "Two ways
to write the same computation", lists the SSD form of Mamba2 among the gated
linear attention recurrences S_t = alpha_t S_{t-1} + k_t^T v_t; the Mamba2
layer of "Long context, fast inference, smart decoding, and life beyond
attention", section "Mamba and hybrid SSMs, the real packages", has state size
128 and head dim 64.  Prefill, decode, speculative decode, replay and
checkpoints all run on this shape.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_02_gb300 import (GLA, glinattn_decode, glinattn_prefill, glinattn_replay,
                                     glinattn_spec_decode, inputs)

from helpers import TOL_F32, TOL_O_BF16, TOL_S_BF16, NT, f64, relerr, to

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _prefill(g, S0=None, out_dtype=torch.float32, **kw):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = glinattn_prefill(g["q"], g["k"], g["v"], g["alpha"], None, S0, variant=GLA, out_dtype=out_dtype,
                           dev_status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out


@pytest.mark.parametrize("T", [1, 63, 200, 300])
@pytest.mark.parametrize("G", [1, 2, 4])
def test_ssd_prefill_bf16(T, G):
    """The chunked tensor-core kernel, one CTA per (batch, head)."""
    ex = inputs.ssd_prefill(2, 4, G, T, seed=T + G, s0_std=0.05)
    g = to(ex, DEV)
    o, S, _ = _prefill(g, g["S0"])
    o_ref, S_ref = oracle.recurrence(GLA, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]),
                                     S0=f64(ex["S0"]), nthreads=NT)
    assert o.shape == (2, T, 4, 64) and S.shape == (2, 4, 128, 64)
    assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(S, S_ref) <= TOL_S_BF16


def test_grouped_gla_with_square_heads():
    """Grouped q / k heads with d_v = 128 (two CTAs per head)."""
    ex = inputs.ssd_prefill(1, 4, 2, 150, dv=128, seed=3, s0_std=0.05)
    g = to(ex, DEV)
    o, S, _ = _prefill(g, g["S0"])
    o_ref, S_ref = oracle.recurrence(GLA, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]),
                                     S0=f64(ex["S0"]), nthreads=NT)
    assert relerr(o, o_ref) <= TOL_O_BF16 and relerr(S, S_ref) <= TOL_S_BF16


@pytest.mark.parametrize("G", [1, 3])
def test_ssd_prefill_fp32_token_serial(G):
    ex = inputs.ssd_prefill(2, 3, G, 45, seed=G, dtype=torch.float32, s0_std=0.05)
    g = to(ex, DEV)
    o, S, _ = _prefill(g, g["S0"])
    o_ref, S_ref = oracle.recurrence(GLA, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]),
                                     S0=f64(ex["S0"]))
    assert relerr(o, o_ref) <= TOL_F32 and relerr(S, S_ref) <= TOL_F32


def test_ssd_segments_and_checkpoints():
    """Three ragged segments chain exactly, and the state emitted every 64
    tokens is the state after those tokens."""
    T = 333
    ex = inputs.ssd_prefill(1, 4, 2, T, seed=21)
    g = to(ex, DEV)
    o_all, S_all, _, Sb, _ = _prefill(g, None, state_every=64)
    _, _, states = oracle.recurrence(GLA, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]),
                                     return_states=True, nthreads=NT)
    for j in range(T // 64):
        assert relerr(Sb[:, j], states[:, 64 * (j + 1) - 1]) <= TOL_S_BF16, j
    S, outs = None, []
    for s, e in ((0, 70), (70, 72), (72, T)):
        seg = {key: (val[:, s:e].contiguous() if key in ("q", "k", "v", "alpha") else val)
               for key, val in g.items()}
        o, S, _ = _prefill(seg, S)
        outs.append(o)
    o_seg = torch.cat(outs, dim=1)
    assert relerr(o_seg, f64(o_all)) <= TOL_O_BF16 and relerr(S, f64(S_all)) <= TOL_S_BF16
    assert relerr(S, states[:, -1]) <= TOL_S_BF16


def test_ssd_prefill_full_size_sampled():
    """B=2, T=4096, 32 heads of head dim 64 sharing one q / k head (one group),
    state size 128: the Mamba2 layer shape; units (0, 0) and (1, 31) in full."""
    ex = inputs.ssd_prefill(2, 32, 1, 4096, seed=0, device=DEV)
    o, S, _ = _prefill(ex)
    for b, h in ((0, 0), (1, 31)):
        o_ref, S_ref = oracle.recurrence(GLA, f64(ex["q"][b:b + 1]), f64(ex["k"][b:b + 1]),
                                         f64(ex["v"][b:b + 1, :, h:h + 1]), f64(ex["alpha"][b:b + 1, :, h:h + 1]))
        assert relerr(o[b:b + 1, :, h:h + 1], o_ref) <= TOL_O_BF16, (b, h)
        assert relerr(S[b:b + 1, h:h + 1], S_ref) <= TOL_S_BF16, (b, h)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_ssd_decode(dtype):
    N, H, G, P = 12, 4, 2, 30
    dx = inputs.ssd_decode(N, H, G, P, seed=5, dtype=dtype)
    g = to(dx, DEV)
    pool = g["pool"].clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = glinattn_decode(g["q"], g["k"], g["v"], g["alpha"], None, pool, g["slot_ids"], variant=GLA,
                        out_dtype=torch.float32, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref, pool_ref, _ = oracle.decode(GLA, f64(dx["q"]), f64(dx["k"]), f64(dx["v"]), f64(dx["alpha"]), None,
                                       f64(dx["pool"]), dx["slot_ids"].tolist(),
                                       act_bf16=dtype == torch.bfloat16)
    tol_o, tol_s = (TOL_O_BF16, TOL_S_BF16) if dtype == torch.bfloat16 else (TOL_F32, TOL_F32)
    sl = dx["slot_ids"].long()
    assert relerr(o, o_ref) <= tol_o
    assert relerr(pool[sl.to(DEV)], pool_ref[sl.numpy()]) <= tol_s
    untouched = torch.ones(P, dtype=torch.bool)
    untouched[sl] = False
    assert torch.equal(pool.cpu()[untouched], dx["pool"][untouched])


def test_ssd_spec_decode_and_replay():
    """Per-draft states match the oracle; a verify-only round plus a replay of
    the accepted drafts lands on the same states bit for bit."""
    N, D, H, G = 6, 4, 4, 1
    P = N * (1 + D)
    dx = inputs.ssd_decode(N, H, G, P, seed=8, D=D)
    g = to(dx, DEV)
    perm = dx["perm"]
    src = perm[:N].to(torch.int32)
    dst = perm[N:N + N * D].to(torch.int32).reshape(N, D)
    pool = g["pool"].clone()
    o = glinattn_spec_decode(g["q"], g["k"], g["v"], g["alpha"], None, pool, src.to(DEV), dst.to(DEV),
                             variant=GLA, out_dtype=torch.float32)
    o_ref, pool_ref, _ = oracle.spec_decode(GLA, f64(dx["q"]), f64(dx["k"]), f64(dx["v"]), f64(dx["alpha"]),
                                            None, f64(dx["pool"]), src.tolist(), dst.tolist())
    torch.cuda.synchronize()
    dl = dst.long()
    assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(pool[dl.to(DEV)], pool_ref[dl.numpy()]) <= TOL_S_BF16
    pool2 = g["pool"].clone()
    o2 = glinattn_spec_decode(g["q"], g["k"], g["v"], g["alpha"], None, pool2, src.to(DEV), None,
                              variant=GLA, out_dtype=torch.float32)
    accept = torch.tensor([0, 4, 1, 2, 3, 4], dtype=torch.int32)
    glinattn_replay(g["k"], g["v"], g["alpha"], None, pool2, src.to(DEV), accept.to(DEV), q=g["q"],
                    variant=GLA)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)
    for n, a in enumerate(accept.tolist()):
        want = dx["pool"][int(src[n])] if a == 0 else pool[int(dst[n, a - 1])].cpu()
        assert torch.equal(pool2[int(src[n])].cpu(), want), (n, a)
    assert np.isfinite(f64(pool2)).all()
