"""The prefill entry point that allocates nothing.

glinattn_prefill_static_scratch serves callers whose device memory is all
planned by their own pools (no spare buffer for scratch, no cudaMalloc from a
library): it runs the same kernels with their scratch in a fixed device array.
This file is collected last so that a run stopping at the first failure has
already run every other test.  Through the C ABI it checks, against the oracle
at the parity tolerances and bit for bit against glinattn_prefill given a
workspace of its own, a call that fills the array almost to its 32 MiB limit
and then two smaller calls in a row (so the small calls run over the large
call's leftovers), the normalised linear attention and the split gated linear
attention scratch, and that a call needing more than the array holds is
refused before anything is launched.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_02_gb300 import glinattn as G
from gated_deltanet_02_gb300 import inputs
from oracle.normalized import nla_prefill

from helpers import TOL_O_BF16, TOL_S_BF16, NT, f64, relerr

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
UNSUPPORTED = 2
LIMIT = 32 << 20


def _entry():
    fn = G.library().glinattn_prefill_static_scratch
    fn.argtypes = [ctypes.POINTER(G.PrefillArgs), ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)


def _args(ex, variant, o, S, conv_out=None, z=None, status=None):
    B, T, H, d = ex["q"].shape
    return G.PrefillArgs(variant=variant, in_dtype=G.BF16, out_dtype=G.F32,
                         qk_l2norm=int(variant == G.GDN), batch=B, seqlen=T, heads=H, dk=d, dv=d,
                         q=_ptr(ex["q"]), k=_ptr(ex["k"]), v=_ptr(ex["v"]), alpha=_ptr(ex.get("alpha")),
                         beta=_ptr(ex.get("beta")), S0=_ptr(ex.get("S0")), S_T=_ptr(S), o=_ptr(o),
                         conv_w=_ptr(ex.get("conv_w")), conv_out=_ptr(conv_out), dev_status=_ptr(status),
                         z0=_ptr(ex.get("z0")), z_T=_ptr(z))


def _run_static(ex, variant):
    """One call of the static entry point; returns (o, S_T, conv_out or z_T)."""
    B, T, H, d = ex["q"].shape
    o = torch.empty(B, T, H, d, dtype=torch.float32, device=DEV)
    S = torch.empty(B, H, d, d, dtype=torch.float32, device=DEV)
    third = (torch.empty(B, 3, 3 * H * d, dtype=torch.bfloat16, device=DEV) if variant == G.GDN
             else torch.empty(B, H, d, dtype=torch.float32, device=DEV) if variant == G.NLA else None)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    a = _args(ex, variant, o, S, conv_out=third if variant == G.GDN else None,
              z=third if variant == G.NLA else None, status=status)
    assert 0 < G.library().glinattn_prefill_workspace_size(ctypes.byref(a)) <= LIMIT
    assert _entry()(ctypes.byref(a), _stream()) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return o, S, third


def _run_workspace(ex, variant):
    """The same call through glinattn_prefill with a workspace of its own."""
    B, T, H, d = ex["q"].shape
    need = G.prefill_workspace_size(B, T, H, d, variant=variant)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=DEV)
    if variant == G.NLA:
        o, S, _, z = G.glinattn_prefill(ex["q"], ex["k"], ex["v"], None, None, ex.get("S0"), variant=G.NLA,
                                        z0=ex.get("z0"), out_dtype=torch.float32, workspace=ws)
        third = z
    else:
        o, S, third = G.glinattn_prefill(ex["q"], ex["k"], ex["v"], ex["alpha"], ex.get("beta"), ex.get("S0"),
                                         variant=variant, conv_w=ex.get("conv_w"),
                                         qk_l2norm=variant == G.GDN, out_dtype=torch.float32, workspace=ws)
    torch.cuda.synchronize()
    return o, S, third


def _oracle_gdn(ex):
    c = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in ex.items()}
    return oracle.layer_prefill(G.GDN, f64(c["q"]), f64(c["k"]), f64(c["v"]), f64(c["alpha"]), f64(c["beta"]),
                                f64(c["S0"]), f64(c["conv_w"]), None, True, nthreads=NT)


def _check_gdn(ex, got):
    o, S, conv = got
    o_ref, S_ref, c_ref = _oracle_gdn(ex)
    assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(S, S_ref) <= TOL_S_BF16
    assert np.array_equal(f64(conv), c_ref)
    ref = _run_workspace(ex, G.GDN)
    for x, y in zip(got, ref):
        assert torch.equal(x, y)


def _largest_gdn_T(B, H, d):
    """The longest segment (a whole number of chunks) whose scratch fits the array."""
    T = 64
    while G.prefill_workspace_size(B, T + 64, H, d) <= LIMIT:
        T += 64
    return T


def test_static_scratch_near_limit_then_twice():
    # a call filling the array almost to its limit leaves non-zero data in it;
    # two smaller calls in a row on different inputs then run over those
    # leftovers (and over each other's) and must still match the oracle and a
    # call with a fresh workspace bit for bit
    B, H, d = 1, 4, 128
    T = _largest_gdn_T(B, H, d)
    need = G.prefill_workspace_size(B, T, H, d)
    assert 0.98 * LIMIT < need <= LIMIT
    ex = inputs.gdn_prefill(B, H, T, d, seed=11, device=DEV)
    _check_gdn(ex, _run_static(ex, G.GDN))
    for seed in (1, 2):
        ex = inputs.gdn_prefill(2, 4, 300, d, seed=seed, device=DEV)
        _check_gdn(ex, _run_static(ex, G.GDN))


def test_static_scratch_refuses_oversized_calls():
    # 2 x 16 heads x 8192 tokens needs about 330 MB of scratch: refused on the host
    B, T, H, d = 2, 8192, 16, 128
    need = G.prefill_workspace_size(B, T, H, d)
    assert need > LIMIT
    fake = 0x10000  # aligned, never dereferenced: the size check comes first
    a = G.PrefillArgs(variant=G.GDN, in_dtype=G.BF16, out_dtype=G.F32, batch=B, seqlen=T,
                      heads=H, dk=d, dv=d, q=fake, k=fake, v=fake, alpha=fake, beta=fake,
                      S_T=fake, o=fake)
    assert _entry()(ctypes.byref(a), None) == UNSUPPORTED


def test_static_scratch_runs_normalised_linear_attention():
    """The chunked normalised linear attention takes its scratch (features,
    chunk sums, normalisers at chunk starts) from the same array."""
    ex = inputs.nla_prefill(1, 2, 300, 128, seed=4, device=DEV, start=True)
    got = _run_static(ex, G.NLA)
    c = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in ex.items()}
    o_ref, S_ref, z_ref = nla_prefill(f64(c["q"]), f64(c["k"]), f64(c["v"]), f64(c["S0"]), f64(c["z0"]))
    assert relerr(got[0], o_ref) <= TOL_O_BF16
    assert relerr(got[1], S_ref) <= TOL_S_BF16 and relerr(got[2], z_ref) <= TOL_S_BF16
    for x, y in zip(got, _run_workspace(ex, G.NLA)):
        assert torch.equal(x, y)


def test_static_scratch_runs_split_gated_linear_attention():
    """Few (batch, head) units: gated linear attention splits the sequence into
    pieces and keeps the pieces' states in the scratch array."""
    B, H, T, d = 1, 2, 4096, 128
    ex = inputs.gla_prefill(B, H, T, d, seed=12, device=DEV, s0_std=0.05)
    assert G.prefill_workspace_size(B, T, H, d, variant=G.GLA) > 0  # the split path
    o, S, _ = _run_static(ex, G.GLA)
    c = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in ex.items()}
    o_ref, S_ref, _ = oracle.layer_prefill(G.GLA, f64(c["q"]), f64(c["k"]), f64(c["v"]), f64(c["alpha"]), None,
                                           f64(c["S0"]), nthreads=NT)
    assert relerr(o, o_ref) <= TOL_O_BF16 and relerr(S, S_ref) <= TOL_S_BF16
    o2, S2, _ = _run_workspace(ex, G.GLA)
    assert torch.equal(o, o2) and torch.equal(S, S2)
