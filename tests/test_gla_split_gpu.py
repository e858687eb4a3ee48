"""GPU parity of the sequence-split gated linear attention prefill (few
(batch, head) units: the sequence is cut into pieces of whole chunks that run
side by side, their start states composed from each piece's local end state and
gate product).  "Inference for linear attention and hybrid architectures",
section "Two ways to write the same computation": only the state passes
between chunks.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_02_gb300 import GLA, glinattn_prefill, inputs
from gated_deltanet_02_gb300 import glinattn as G
from gated_deltanet_02_gb300.glinattn import DEV_BAD_GATE

from helpers import TOL_O_BF16, TOL_S_BF16, NT, f64, relerr, to

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("B,H,G_,T,dv", [(1, 2, 2, 1024, 128), (1, 8, 1, 2048, 64), (2, 3, 3, 768, 128)])
def test_split_prefill_matches_oracle(B, H, G_, T, dv):
    ex = inputs.ssd_prefill(B, H, G_, T, dv=dv, seed=T + H, s0_std=0.05)
    g = to(ex, DEV)
    assert G.prefill_workspace_size(B, T, H, 128, variant=GLA) >= 0
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, S, _ = glinattn_prefill(g["q"], g["k"], g["v"], g["alpha"], None, g["S0"], variant=GLA,
                               out_dtype=torch.float32, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref, S_ref = oracle.recurrence(GLA, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]),
                                     S0=f64(ex["S0"]), nthreads=NT)
    assert relerr(o, o_ref) <= TOL_O_BF16 and relerr(S, S_ref) <= TOL_S_BF16


def _abi_prefill(g, with_workspace, o, S, status, alpha=None):
    B, T, Hq, dk = g["q"].shape
    H, dv = g["v"].shape[2], g["v"].shape[3]
    a = G.PrefillArgs(variant=G.GLA, in_dtype=G.BF16, out_dtype=G.F32, batch=B, seqlen=T, heads=H, dk=dk, dv=dv,
                      q=_ptr(g["q"]), k=_ptr(g["k"]), v=_ptr(g["v"]), alpha=_ptr(g["alpha"] if alpha is None else alpha),
                      S0=_ptr(g["S0"]), S_T=_ptr(S), o=_ptr(o), dev_status=_ptr(status), qk_heads=Hq)
    need = G.library().glinattn_prefill_workspace_size(ctypes.byref(a))
    ws = None
    if with_workspace and need:
        ws = torch.empty(need, dtype=torch.uint8, device=DEV)
        a.workspace, a.workspace_bytes = _ptr(ws), need
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    assert G.library().glinattn_prefill(ctypes.byref(a), stream) == 0
    torch.cuda.synchronize()
    return need


def test_split_equals_unsplit():
    """Without the scratch the same call runs unsplit: the two agree to fp32
    rounding of the state composition."""
    ex = inputs.ssd_prefill(1, 4, 2, 1024, dv=128, seed=5, s0_std=0.05)
    g = to(ex, DEV)
    outs = []
    for ws in (True, False):
        o = torch.empty(1, 1024, 4, 128, device=DEV)
        S = torch.empty(1, 4, 128, 128, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        need = _abi_prefill(g, ws, o, S, status)
        assert int(status.item()) == 0
        outs.append((o, S))
    assert need > 0  # this shape takes the split
    assert relerr(outs[0][0], f64(outs[1][0])) <= 1e-5 and relerr(outs[0][1], f64(outs[1][1])) <= 1e-5


def test_split_bad_gate_skips_every_piece():
    """An invalid gate in the first piece: the unit raises the flag and none of
    its pieces, nor its final state, is written; the other unit is computed."""
    ex = inputs.ssd_prefill(1, 2, 2, 1024, dv=128, seed=6)
    g = to(ex, DEV)
    alpha = g["alpha"].clone()
    alpha[0, 10, 1] = 0.0  # head 1, token 10
    o = torch.full((1, 1024, 2, 128), 7.0, device=DEV)
    S = torch.full((1, 2, 128, 128), 7.0, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    need = _abi_prefill(g, True, o, S, status, alpha=alpha)
    assert need > 0
    assert int(status.item()) & DEV_BAD_GATE
    assert bool((o[0, :, 1] == 7.0).all()) and bool((S[0, 1] == 7.0).all())
    o_ref, S_ref = oracle.recurrence(GLA, f64(ex["q"][:, :, :1]), f64(ex["k"][:, :, :1]), f64(ex["v"][:, :, :1]),
                                     f64(ex["alpha"][:, :, :1]))
    assert relerr(o[:, :, :1], o_ref) <= TOL_O_BF16 and relerr(S[:, :1], S_ref) <= TOL_S_BF16
