"""Long-context Gated DeltaNet at full size on the GPU: B=1, H=32, T=32768
prefilled as segments of 20% / 35% / 45% carrying state and conv cache, then
64 requests doing speculative decode of 4 draft tokens with one state per draft
position, rolled back to an accepted prefix length 0..4.

"Inference for linear attention and hybrid architectures": section "Two ways
to write the same computation" (segmented prefill hands the state on),
section "Prefix caching has to be redone" (each request continues from its
own copy of the state), section "Speculative decoding and PD disaggregation"
(one state per draft position; rollback is a choice of state).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_02_gb300 import GDN, glinattn_prefill, glinattn_spec_decode, inputs

from helpers import TOL_O_BF16, TOL_S_BF16, NT, f64, relerr

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
B, H, T, D_HEAD = 1, 32, 32768, 128
N_REQ, DRAFT = 64, 4


@pytest.fixture(scope="module")
def prefilled():
    ex = inputs.gdn_prefill(B, H, T, D_HEAD, seed=5, device=DEV, s0_std=0.0)
    segs = inputs.segment_lengths(T)
    assert segs == [6553, 11468, 14747]
    S, conv, outs, s0 = None, None, [], 0
    for L in segs:
        sl = slice(s0, s0 + L)
        o, S, conv = glinattn_prefill(ex["q"][:, sl].contiguous(), ex["k"][:, sl].contiguous(),
                                      ex["v"][:, sl].contiguous(), ex["alpha"][:, sl].contiguous(),
                                      ex["beta"][:, sl].contiguous(), S, variant=GDN,
                                      conv_w=ex["conv_w"], conv_in=conv, qk_l2norm=True,
                                      out_dtype=torch.float32)
        outs.append(o)
        s0 += L
    torch.cuda.synchronize()
    return ex, torch.cat(outs, dim=1), S, conv


def test_segmented_long_prefill_matches_oracle(prefilled):
    """Every one of the 32 heads of the three-segment prefill against the
    oracle's one-shot prefill (all host cores)."""
    ex, o, S, conv = prefilled
    cpu = {k: ex[k].cpu() for k in ("q", "k", "v", "alpha", "beta", "conv_w")}
    o_ref, S_ref, c_ref = oracle.layer_prefill(GDN, *(f64(cpu[k]) for k in ("q", "k", "v", "alpha", "beta")),
                                               None, f64(cpu["conv_w"]), None, True, nthreads=NT)
    o64, S64 = f64(o), f64(S)
    for h in range(H):
        assert relerr(o64[:, :, h], o_ref[:, :, h]) <= TOL_O_BF16, h
        assert relerr(S64[:, h], S_ref[:, h]) <= TOL_S_BF16, h
    assert np.array_equal(f64(conv), c_ref)


def test_segmented_equals_one_shot_long(prefilled):
    ex, o_seg, S_seg, conv_seg = prefilled
    o1, S1, c1 = glinattn_prefill(ex["q"], ex["k"], ex["v"], ex["alpha"], ex["beta"], None,
                                  variant=GDN, conv_w=ex["conv_w"], qk_l2norm=True,
                                  out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert relerr(o_seg, f64(o1)) <= TOL_O_BF16
    assert relerr(S_seg, f64(S1)) <= TOL_S_BF16
    assert torch.equal(conv_seg, c1)


def test_spec_decode_rollback_long_context(prefilled):
    ex, _, S, conv = prefilled
    P = N_REQ * (1 + DRAFT)
    pool = torch.empty(P, H, D_HEAD, D_HEAD, dtype=torch.float32, device=DEV)
    cpool = torch.empty(P, 3, 3 * H * D_HEAD, dtype=torch.bfloat16, device=DEV)
    src = torch.arange(N_REQ, dtype=torch.int32, device=DEV)
    dst = (N_REQ + torch.arange(N_REQ * DRAFT, dtype=torch.int32, device=DEV)).view(N_REQ, DRAFT)
    pool[:N_REQ] = S[0]          # every request continues from its own copy
    cpool[:N_REQ] = conv[0]
    dr = inputs.spec_drafts(N_REQ, DRAFT, H, D_HEAD, seed=9, device=DEV)
    src_before = pool[:N_REQ].clone()
    o = glinattn_spec_decode(dr["q"], dr["k"], dr["v"], dr["alpha"], dr["beta"], pool, src, dst,
                             variant=GDN, conv_w=ex["conv_w"], conv_pool=cpool, qk_l2norm=True,
                             out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(pool[:N_REQ], src_before)
    accept = dr["accept"].tolist()
    # rollback: the kept state of request n is src (a = 0) or dst[n, a-1]
    kept = [int(src[n]) if a == 0 else int(dst[n, a - 1]) for n, a in enumerate(accept)]
    # the oracle for every request, all heads, from the prefilled state
    for n in range(N_REQ):
        mini_pool = f64(S)  # slot 0: the request's copy of the prefilled state
        o_ref, pool_ref, cpool_ref = oracle.spec_decode(
            GDN, f64(dr["q"][n:n + 1]), f64(dr["k"][n:n + 1]), f64(dr["v"][n:n + 1]),
            f64(dr["alpha"][n:n + 1]), f64(dr["beta"][n:n + 1]), np.concatenate(
                [mini_pool, np.zeros((DRAFT,) + mini_pool.shape[1:])]), [0], [[1, 2, 3, 4]],
            f64(ex["conv_w"]), np.concatenate([f64(conv), np.zeros((DRAFT,) + tuple(conv.shape[1:]))]),
            True)
        assert relerr(o[n:n + 1], o_ref) <= TOL_O_BF16, n
        for i in range(DRAFT):
            assert relerr(pool[int(dst[n, i])], pool_ref[1 + i]) <= TOL_S_BF16, (n, i)
            assert np.array_equal(f64(cpool[int(dst[n, i])]), cpool_ref[1 + i]), (n, i)
        a = accept[n]
        want = f64(S)[0] if a == 0 else pool_ref[a]
        assert relerr(pool[kept[n]], want) <= TOL_S_BF16, n
