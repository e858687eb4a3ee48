"""The prefill entry point that allocates nothing.

glinattn_prefill_static_scratch serves callers whose device memory is all
planned by their own pools (no spare buffer for scratch, no cudaMalloc from a
library): it runs the same kernels with their scratch in a fixed device array.
This file is collected last so that a run stopping at the first failure has
already run every other test.  It checks, through the C ABI, that two calls in
a row give what glinattn_prefill gives on the same inputs, and that a call
needing more than the array holds is refused before anything is launched.
"""
import ctypes

import pytest
import torch

from gated_deltanet_02_gb300 import glinattn as G
from gated_deltanet_02_gb300 import inputs

from helpers import TOL_O_BF16, TOL_S_BF16, relerr

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
UNSUPPORTED = 2


def _entry():
    fn = G.library().glinattn_prefill_static_scratch
    fn.argtypes = [ctypes.POINTER(G.PrefillArgs), ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _run_static(ex):
    B, T, H, d = ex["q"].shape
    o = torch.empty(B, T, H, d, dtype=torch.float32, device=DEV)
    S = torch.empty(B, H, d, d, dtype=torch.float32, device=DEV)
    conv_out = torch.empty(B, 3, 3 * H * d, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    a = G.PrefillArgs(variant=G.GDN, in_dtype=G.BF16, out_dtype=G.F32, qk_l2norm=1, batch=B,
                      seqlen=T, heads=H, dk=d, dv=d, q=_ptr(ex["q"]), k=_ptr(ex["k"]),
                      v=_ptr(ex["v"]), alpha=_ptr(ex["alpha"]), beta=_ptr(ex["beta"]),
                      S0=_ptr(ex["S0"]), S_T=_ptr(S), o=_ptr(o), conv_w=_ptr(ex["conv_w"]),
                      conv_out=_ptr(conv_out), dev_status=_ptr(status))
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    assert _entry()(ctypes.byref(a), stream) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return o, S, conv_out


def test_static_scratch_matches_workspace_entry_point_twice():
    # two calls in a row on different inputs: the second must not see the
    # first one's leftovers in the shared array
    for seed in (1, 2):
        ex = inputs.gdn_prefill(2, 4, 300, 128, seed=seed, device=DEV)
        need = G.prefill_workspace_size(2, 300, 4, 128)
        assert 0 < need <= 32 << 20
        o, S, c = _run_static(ex)
        o_ref, S_ref, c_ref = G.glinattn_prefill(
            ex["q"], ex["k"], ex["v"], ex["alpha"], ex["beta"], ex["S0"], variant=G.GDN,
            conv_w=ex["conv_w"], qk_l2norm=True, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert relerr(o, o_ref.double().cpu().numpy()) <= TOL_O_BF16
        assert relerr(S, S_ref.double().cpu().numpy()) <= TOL_S_BF16
        assert torch.equal(c, c_ref)


def test_static_scratch_refuses_oversized_calls():
    # 2 x 16 heads x 8192 tokens needs about 330 MB of scratch: refused on the host
    B, T, H, d = 2, 8192, 16, 128
    need = G.prefill_workspace_size(B, T, H, d)
    assert need > 32 << 20
    fake = 0x10000  # aligned, never dereferenced: the size check comes first
    a = G.PrefillArgs(variant=G.GDN, in_dtype=G.BF16, out_dtype=G.F32, batch=B, seqlen=T,
                      heads=H, dk=d, dv=d, q=fake, k=fake, v=fake, alpha=fake, beta=fake,
                      S_T=fake, o=fake)
    assert _entry()(ctypes.byref(a), None) == UNSUPPORTED


def test_static_scratch_runs_normalised_linear_attention():
    """The chunked normalised linear attention takes its scratch (features,
    chunk sums, the fp32 numerator) from the same array."""
    B, T, H, d = 1, 300, 2, 128
    ex = inputs.nla_prefill(B, H, T, d, seed=4, device=DEV, start=True)
    o = torch.empty(B, T, H, d, dtype=torch.bfloat16, device=DEV)
    S = torch.empty(B, H, d, d, dtype=torch.float32, device=DEV)
    z = torch.empty(B, H, d, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    a = G.PrefillArgs(variant=G.NLA, in_dtype=G.BF16, out_dtype=G.BF16, batch=B, seqlen=T, heads=H, dk=d,
                      dv=d, q=_ptr(ex["q"]), k=_ptr(ex["k"]), v=_ptr(ex["v"]), S0=_ptr(ex["S0"]), S_T=_ptr(S),
                      o=_ptr(o), dev_status=_ptr(status), z0=_ptr(ex["z0"]), z_T=_ptr(z))
    assert 0 < G.library().glinattn_prefill_workspace_size(ctypes.byref(a)) <= 32 << 20
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    assert _entry()(ctypes.byref(a), stream) == 0
    o_ref, S_ref, _, z_ref = G.glinattn_prefill(ex["q"], ex["k"], ex["v"], None, None, ex["S0"], variant=G.NLA,
                                                z0=ex["z0"], out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(o, o_ref) and torch.equal(S, S_ref) and torch.equal(z, z_ref)
