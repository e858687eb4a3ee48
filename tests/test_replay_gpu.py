"""GPU parity of replay rollback: verify-only speculative decode followed by a
replay of the accepted drafts.

"Inference for linear attention and hybrid architectures", section
"Speculative decoding and PD disaggregation": a state cannot be rolled back,
so either one state is kept per draft position, or the draft steps are
recorded and replayed from a chosen position.  Both must leave the request at
the state after its accepted drafts; here the replayed state is compared with
the per-draft state bit for bit (both run the decode step's arithmetic) and
with the oracle.  The verify-only outputs of the 128 x 128 gated forms come
from the chunked form over the drafts (one read of the start state), so they
match the per-draft outputs to fp32 rounding and the oracle to the outputs'
tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_02_gb300 import GDN, GLA, glinattn_replay, glinattn_spec_decode, inputs
from gated_deltanet_02_gb300.glinattn import DEV_BAD_COUNT, DEV_BAD_GATE, DEV_BAD_SLOT

from helpers import TOL_F32, TOL_O_BF16, TOL_S_BF16, f64, relerr

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _setup(N, D, H, d, P, seed, dtype, variant):
    base = inputs.gdn_decode(N, H, d, P, seed=seed, dtype=dtype, variant_gdn=variant == GDN)
    dr = inputs.spec_drafts(N, D, H, d, seed=seed + 100, dtype=dtype)
    if variant == GLA:
        dr["beta"] = None
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(seed))
    src = perm[:N].to(torch.int32)
    dst = perm[N:N + N * D].to(torch.int32).reshape(N, D)
    return base, dr, src, dst


def _dev(t):
    return None if t is None else t.to(DEV)


@pytest.mark.parametrize("d,D,dtype,variant", [
    (64, 4, torch.bfloat16, GDN),
    (128, 4, torch.bfloat16, GDN),
    (128, 4, torch.float32, GDN),
    (64, 3, torch.float32, GDN),
    (128, 4, torch.bfloat16, GLA),
    (128, 10, torch.bfloat16, GDN),   # drafts past the d = 128 kernel's per-unit table
])
def test_verify_then_replay_equals_per_draft_state(d, D, dtype, variant):
    N, H, P = 8, 3, 8 + 8 * 10
    conv = variant == GDN
    base, dr, src, dst = _setup(N, D, H, d, P, 17 + d + D, dtype, variant)
    g = {k: _dev(v) for k, v in dr.items()}
    w = _dev(base["conv_w"]) if conv else None
    # per-draft states
    pool_a, cpool_a = _dev(base["pool"]), _dev(base["conv_pool"])
    o_a = glinattn_spec_decode(g["q"], g["k"], g["v"], g["alpha"], g["beta"], pool_a, _dev(src), _dev(dst),
                               variant=variant, conv_w=w, conv_pool=cpool_a if conv else None,
                               qk_l2norm=conv, out_dtype=torch.float32)
    # verify only: same outputs, nothing written
    pool_b, cpool_b = _dev(base["pool"]), _dev(base["conv_pool"])
    o_b = glinattn_spec_decode(g["q"], g["k"], g["v"], g["alpha"], g["beta"], pool_b, _dev(src), None,
                               variant=variant, conv_w=w, conv_pool=cpool_b if conv else None,
                               qk_l2norm=conv, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert relerr(o_b, f64(o_a)) <= TOL_F32
    assert torch.equal(pool_b.cpu(), base["pool"]) and torch.equal(cpool_b.cpu(), base["conv_pool"])
    # replay the accepted drafts in place: every length 0..D occurs
    accept = (torch.arange(N, dtype=torch.int32) * 7 + 3) % (D + 1)
    accept[0], accept[1] = 0, D
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    glinattn_replay(g["k"], g["v"], g["alpha"], g["beta"], pool_b, _dev(src), _dev(accept), q=g["q"],
                    variant=variant, conv_w=w, conv_pool=cpool_b if conv else None, qk_l2norm=conv,
                    dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    pool_a, pool_b = pool_a.cpu(), pool_b.cpu()
    cpool_a, cpool_b = cpool_a.cpu(), cpool_b.cpu()
    for n, a in enumerate(accept.tolist()):
        s = int(src[n])
        want = base["pool"][s] if a == 0 else pool_a[int(dst[n, a - 1])]
        assert torch.equal(pool_b[s], want), (n, a)
        if conv:
            cwant = base["conv_pool"][s] if a == 0 else cpool_a[int(dst[n, a - 1])]
            assert torch.equal(cpool_b[s], cwant), (n, a)
    others = torch.ones(P, dtype=torch.bool)
    others[src.long()] = False
    assert torch.equal(pool_b[others], base["pool"][others])
    # and the oracle's state after the accepted drafts
    o_ref, pool_ref, _ = oracle.spec_decode(variant, f64(dr["q"]), f64(dr["k"]), f64(dr["v"]), f64(dr["alpha"]),
                                            f64(dr["beta"]), f64(base["pool"]), src.tolist(), dst.tolist(),
                                            f64(base["conv_w"]) if conv else None,
                                            f64(base["conv_pool"]) if conv else None, conv,
                                            act_bf16=dtype == torch.bfloat16)
    assert relerr(o_b, o_ref) <= (TOL_O_BF16 if dtype == torch.bfloat16 else TOL_F32)
    tol = TOL_S_BF16 if dtype == torch.bfloat16 else TOL_F32
    for n, a in enumerate(accept.tolist()):
        if a:
            assert relerr(pool_b[int(src[n])], pool_ref[int(dst[n, a - 1])]) <= tol, (n, a)


@pytest.mark.parametrize("d", [64, 128])
def test_replay_bad_length_is_flagged_and_skipped(d):
    N, D, H, P = 6, 4, 2, 40
    base, dr, src, dst = _setup(N, D, H, d, P, 5, torch.bfloat16, GDN)
    g = {k: _dev(v) for k, v in dr.items()}
    pool, cpool = _dev(base["pool"]), _dev(base["conv_pool"])
    accept = torch.tensor([2, 5, -1, 0, 4, 1], dtype=torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    glinattn_replay(g["k"], g["v"], g["alpha"], g["beta"], pool, _dev(src), _dev(accept), q=g["q"],
                    variant=GDN, conv_w=_dev(base["conv_w"]), conv_pool=cpool, qk_l2norm=True,
                    dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & DEV_BAD_COUNT
    pool, cpool = pool.cpu(), cpool.cpu()
    for n in (1, 2, 3):  # bad lengths and the empty replay: untouched
        s = int(src[n])
        assert torch.equal(pool[s], base["pool"][s]) and torch.equal(cpool[s], base["conv_pool"][s])
    _, pool_ref, cpool_ref = oracle.spec_decode(GDN, f64(dr["q"]), f64(dr["k"]), f64(dr["v"]),
                                                f64(dr["alpha"]), f64(dr["beta"]), f64(base["pool"]),
                                                src.tolist(), dst.tolist(), f64(base["conv_w"]),
                                                f64(base["conv_pool"]), True)
    for n in (0, 4, 5):
        s, a = int(src[n]), int(accept[n])
        assert relerr(pool[s], pool_ref[int(dst[n, a - 1])]) <= TOL_S_BF16
        assert np.array_equal(f64(cpool[s]), cpool_ref[int(dst[n, a - 1])])


@pytest.mark.parametrize("variant", [GDN, GLA])
@pytest.mark.parametrize("D", [1, 5, 16])
def test_verify_only_outputs_match_oracle(variant, D):
    """Verify-only outputs at d = 128 for 1, 5 and 16 drafts (the chunked form
    handles up to 16) against the oracle and the per-draft outputs."""
    N, H, d = 5, 4, 128
    P = N * (1 + D)
    conv = variant == GDN
    base, dr, src, dst = _setup(N, D, H, d, P, 60 + D, torch.bfloat16, variant)
    g = {k: _dev(v) for k, v in dr.items()}
    w = _dev(base["conv_w"]) if conv else None
    pool, cpool = _dev(base["pool"]), _dev(base["conv_pool"])
    o_v = glinattn_spec_decode(g["q"], g["k"], g["v"], g["alpha"], g["beta"], pool, _dev(src), None,
                               variant=variant, conv_w=w, conv_pool=cpool if conv else None, qk_l2norm=conv,
                               out_dtype=torch.float32)
    o_s = glinattn_spec_decode(g["q"], g["k"], g["v"], g["alpha"], g["beta"], pool, _dev(src), _dev(dst),
                               variant=variant, conv_w=w, conv_pool=cpool if conv else None, qk_l2norm=conv,
                               out_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, _, _ = oracle.spec_decode(variant, f64(dr["q"]), f64(dr["k"]), f64(dr["v"]), f64(dr["alpha"]),
                                     f64(dr["beta"]), f64(base["pool"]), src.tolist(), dst.tolist(),
                                     f64(base["conv_w"]) if conv else None,
                                     f64(base["conv_pool"]) if conv else None, conv)
    assert relerr(o_v, o_ref) <= TOL_O_BF16
    assert relerr(o_v, f64(o_s)) <= TOL_F32


def test_verify_only_bad_slot_and_gate_are_flagged_and_skipped():
    N, D, H, d, P = 4, 4, 2, 128, 24
    base, dr, src, dst = _setup(N, D, H, d, P, 71, torch.bfloat16, GDN)
    dr["alpha"][2, 1, 0] = 0.0        # request 2: a gate outside (0, 1]
    src[1] = P + 3                     # request 1: a slot past the pool
    g = {k: _dev(v) for k, v in dr.items()}
    pool, cpool = _dev(base["pool"]), _dev(base["conv_pool"])
    o = torch.full((N, D, H, d), 7.0, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    glinattn_spec_decode(g["q"], g["k"], g["v"], g["alpha"], g["beta"], pool, _dev(src), None, variant=GDN,
                         conv_w=_dev(base["conv_w"]), conv_pool=cpool, qk_l2norm=True, o=o, out_dtype=torch.float32,
                         dev_status=status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st & DEV_BAD_SLOT and st & DEV_BAD_GATE
    assert bool((o[1] == 7.0).all()) and bool((o[2, :, 0] == 7.0).all())
    assert torch.equal(pool.cpu(), base["pool"])
    good = [0, 3]
    sub = {k: (v[good] if v is not None else None) for k, v in dr.items()}
    o_ref, _, _ = oracle.spec_decode(GDN, f64(sub["q"]), f64(sub["k"]), f64(sub["v"]), f64(sub["alpha"]),
                                     f64(sub["beta"]), f64(base["pool"]), src[good].tolist(), dst[good].tolist(),
                                     f64(base["conv_w"]), f64(base["conv_pool"]), True)
    assert relerr(o[good], o_ref) <= TOL_O_BF16
