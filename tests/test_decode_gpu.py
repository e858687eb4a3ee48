"""GPU parity of recurrent decode and speculative decode against the oracle.

"Inference for linear attention and hybrid architectures": section "Two ways
to write the same computation" (decode = one read and one rank-one update of
the state per token) and section "Speculative decoding and PD disaggregation"
(slot-indexed state pool; one state kept per draft position for rollback).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_02_gb300 import GDN, GLA, glinattn_decode, glinattn_spec_decode, inputs
from gated_deltanet_02_gb300.glinattn import DEV_BAD_GATE, DEV_BAD_SLOT

from helpers import TOL_F32, TOL_O_BF16, TOL_S_BF16, f64, relerr, to

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _run_decode(ex, variant, conv, l2, out_dtype=torch.float32):
    g = to(ex, DEV)
    pool, cpool = g["pool"].clone(), (g["conv_pool"].clone() if conv else None)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = glinattn_decode(g["q"], g["k"], g["v"], g["alpha"], g["beta"], pool, g["slot_ids"],
                        variant=variant, conv_w=g["conv_w"] if conv else None, conv_pool=cpool,
                        qk_l2norm=l2, out_dtype=out_dtype, dev_status=status)
    torch.cuda.synchronize()
    return o, pool, cpool, int(status.item())


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("variant", [GLA, GDN])
def test_decode_matches_oracle_bf16(d, variant):
    ex = inputs.gdn_decode(12, 3, d, 40, seed=d + variant, variant_gdn=variant == GDN)
    conv = variant == GDN
    o, pool, cpool, st = _run_decode(ex, variant, conv, conv)
    assert st == 0
    o_ref, pool_ref, cpool_ref = oracle.decode(
        variant, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]), f64(ex["beta"]),
        f64(ex["pool"]), ex["slot_ids"].tolist(), f64(ex["conv_w"]) if conv else None,
        f64(ex["conv_pool"]) if conv else None, conv)
    slots = ex["slot_ids"].long()
    assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(pool[slots.to(DEV)], pool_ref[slots.numpy()]) <= TOL_S_BF16
    # untouched slots are byte-identical
    untouched = torch.ones(ex["pool"].shape[0], dtype=torch.bool)
    untouched[slots] = False
    assert torch.equal(pool.cpu()[untouched], ex["pool"][untouched])
    if conv:  # conv caches hold raw inputs: exact
        assert np.array_equal(f64(cpool), cpool_ref)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_fp32_inputs_tight(d):
    ex = inputs.gdn_decode(6, 2, d, 10, seed=3, dtype=torch.float32)
    o, pool, cpool, st = _run_decode(ex, GDN, True, True)
    o_ref, pool_ref, cpool_ref = oracle.decode(
        GDN, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]), f64(ex["beta"]),
        f64(ex["pool"]), ex["slot_ids"].tolist(), f64(ex["conv_w"]), f64(ex["conv_pool"]), True,
        act_bf16=False)
    assert relerr(o, o_ref) <= TOL_F32
    assert relerr(pool, pool_ref) <= TOL_F32
    assert np.array_equal(f64(cpool), cpool_ref)


def test_decode_full_size_all_requests():
    """256 requests x 16 heads, d = 128, 512-slot pool: all 4096 states updated in
    one launch; every request is checked against the oracle and every
    untouched slot is byte-identical."""
    N, H, d, P = 256, 16, 128, 512
    ex = inputs.gdn_decode(N, H, d, P, seed=0, device=DEV)
    o, pool, cpool, st = _run_decode(ex, GDN, True, True)
    assert st == 0
    slots = ex["slot_ids"].long()
    untouched = torch.ones(P, dtype=torch.bool, device=DEV)
    untouched[slots] = False
    assert torch.equal(pool[untouched], ex["pool"][untouched])
    assert torch.equal(cpool[untouched], ex["conv_pool"][untouched])
    # the oracle on a pool holding only the touched slots, in request order
    o_ref, pool_ref, cpool_ref = oracle.decode(
        GDN, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]), f64(ex["beta"]),
        f64(ex["pool"][slots]), list(range(N)), f64(ex["conv_w"]), f64(ex["conv_pool"][slots]), True)
    o64, p64 = f64(o), f64(pool[slots])
    for n in range(N):
        assert relerr(o64[n], o_ref[n]) <= TOL_O_BF16, n
        assert relerr(p64[n], pool_ref[n]) <= TOL_S_BF16, n
    assert np.array_equal(f64(cpool[slots]), cpool_ref)


def test_decode_bf16_output():
    ex = inputs.gdn_decode(8, 2, 128, 16, seed=4)
    o, _, _, _ = _run_decode(ex, GDN, True, True, out_dtype=torch.bfloat16)
    o_ref, _, _ = oracle.decode(GDN, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]),
                                f64(ex["beta"]), f64(ex["pool"]), ex["slot_ids"].tolist(),
                                f64(ex["conv_w"]), f64(ex["conv_pool"]), True)
    # a bf16 output carries up to half an ulp (2^-9 relative) on top of the fp32 error
    err = np.abs(f64(o) - o_ref)
    assert (err <= np.abs(o_ref) * 2.0 ** -8 + TOL_O_BF16 * np.abs(o_ref).max()).all()


def test_bad_slot_and_gate_are_flagged_and_skipped():
    ex = inputs.gdn_decode(4, 2, 64, 8, seed=5)
    ex["slot_ids"] = ex["slot_ids"].clone()
    ex["slot_ids"][1] = 8  # out of range
    ex["alpha"] = ex["alpha"].clone()
    ex["alpha"][2, 1] = 0.0  # gate outside (0, 1]
    o, pool, cpool, st = _run_decode(ex, GDN, True, True)
    assert st == DEV_BAD_SLOT | DEV_BAD_GATE
    # request 2 / head 1 skipped: its slot is unchanged; request 0 / head 0 updated
    s2 = int(ex["slot_ids"][2])
    assert torch.equal(pool[s2, 1].cpu(), ex["pool"][s2, 1])
    s0 = int(ex["slot_ids"][0])
    assert not torch.equal(pool[s0, 0].cpu(), ex["pool"][s0, 0])


def test_decode128_bad_slot_and_gate_are_flagged_and_skipped():
    ex = inputs.gdn_decode(6, 3, 128, 12, seed=21)
    ex["slot_ids"] = ex["slot_ids"].clone()
    ex["slot_ids"][1] = 12  # out of range
    ex["alpha"] = ex["alpha"].clone()
    ex["alpha"][2, 1] = 1.5  # gate outside (0, 1]
    o, pool, cpool, st = _run_decode(ex, GDN, True, True)
    assert st == DEV_BAD_SLOT | DEV_BAD_GATE
    s2 = int(ex["slot_ids"][2])
    assert torch.equal(pool[s2, 1].cpu(), ex["pool"][s2, 1])
    hd = [c for part in range(3) for c in range(part * 3 * 128 + 128, part * 3 * 128 + 256)]
    assert torch.equal(cpool[s2][:, hd].cpu(), ex["conv_pool"][s2][:, hd])
    # every other unit is updated as the oracle says
    good = [0, 3, 4, 5]
    sl = ex["slot_ids"][good].long()
    o_ref, pool_ref, cpool_ref = oracle.decode(
        GDN, f64(ex["q"][good]), f64(ex["k"][good]), f64(ex["v"][good]), f64(ex["alpha"][good]),
        f64(ex["beta"][good]), f64(ex["pool"][sl]), list(range(len(good))), f64(ex["conv_w"]),
        f64(ex["conv_pool"][sl]), True)
    assert relerr(o[good], o_ref) <= TOL_O_BF16
    assert relerr(pool[sl.to(DEV)], pool_ref) <= TOL_S_BF16
    assert np.array_equal(f64(cpool[sl.to(DEV)]), cpool_ref)
    # request 2: heads 0 and 2 are updated (the oracle run gets a valid gate for head 1)
    a2 = ex["alpha"][2:3].clone()
    a2[0, 1] = 0.5
    s2t = torch.tensor([s2])
    _, p2_ref, _ = oracle.decode(
        GDN, f64(ex["q"][2:3]), f64(ex["k"][2:3]), f64(ex["v"][2:3]), f64(a2), f64(ex["beta"][2:3]),
        f64(ex["pool"][s2t]), [0], f64(ex["conv_w"]), f64(ex["conv_pool"][s2t]), True)
    for h in (0, 2):
        assert relerr(pool[s2, h], p2_ref[0, h]) <= TOL_S_BF16


def test_decode128_many_units_per_cluster():
    """3 requests x 600 heads: each persistent cluster walks several units in
    turn, and the head (hence the conv weights) changes every 3 units."""
    N, H, d, P = 3, 600, 128, 4
    ex = inputs.gdn_decode(N, H, d, P, seed=13)
    o, pool, cpool, st = _run_decode(ex, GDN, True, True, out_dtype=torch.bfloat16)
    assert st == 0
    o_ref, pool_ref, cpool_ref = oracle.decode(
        GDN, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]), f64(ex["beta"]),
        f64(ex["pool"]), ex["slot_ids"].tolist(), f64(ex["conv_w"]), f64(ex["conv_pool"]), True)
    err = np.abs(f64(o) - o_ref)
    assert (err <= np.abs(o_ref) * 2.0 ** -8 + TOL_O_BF16 * np.abs(o_ref).max()).all()
    sl = ex["slot_ids"].long()
    assert relerr(pool[sl.to(DEV)], pool_ref[sl.numpy()]) <= TOL_S_BF16
    assert np.array_equal(f64(cpool), cpool_ref)


def _spec_setup(N, D, H, d, P, seed):
    base = inputs.gdn_decode(N, H, d, P, seed=seed)
    dr = inputs.spec_drafts(N, D, H, d, seed=seed + 100)
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(seed))
    src = perm[:N].to(torch.int32)
    dst = perm[N:N + N * D].to(torch.int32).reshape(N, D)
    return base, dr, src, dst


@pytest.mark.parametrize("D,P", [(4, 64), (10, 80)])
def test_spec_decode_matches_oracle_and_repeated_decode(D, P):
    """D = 10 drafts also covers steps whose gates and slots are read past the
    per-unit table of the d = 128 kernel."""
    N, H, d = 6, 3, 128
    base, dr, src, dst = _spec_setup(N, D, H, d, P, 7)
    pool, cpool = base["pool"].to(DEV), base["conv_pool"].to(DEV)
    g = to(dr, DEV)
    w = base["conv_w"].to(DEV)
    o = glinattn_spec_decode(g["q"], g["k"], g["v"], g["alpha"], g["beta"], pool, src.to(DEV),
                             dst.to(DEV), variant=GDN, conv_w=w, conv_pool=cpool, qk_l2norm=True,
                             out_dtype=torch.float32)
    torch.cuda.synchronize()
    # oracle
    o_ref, pool_ref, cpool_ref = oracle.spec_decode(
        GDN, f64(dr["q"]), f64(dr["k"]), f64(dr["v"]), f64(dr["alpha"]), f64(dr["beta"]),
        f64(base["pool"]), src.tolist(), dst.tolist(), f64(base["conv_w"]), f64(base["conv_pool"]),
        True)
    assert relerr(o, o_ref) <= TOL_O_BF16
    dl = dst.long()
    assert relerr(pool[dl.to(DEV)], pool_ref[dl.numpy()]) <= TOL_S_BF16
    assert np.array_equal(f64(cpool[dl.to(DEV)]), cpool_ref[dl.numpy()])
    # the source slots are only read
    assert torch.equal(pool[src.long().to(DEV)].cpu(), base["pool"][src.long()])
    # bit-identical to D repeated decode steps on a copy of the source states
    pool2, cpool2 = base["pool"].to(DEV), base["conv_pool"].to(DEV)
    for i in range(D):
        oi = glinattn_decode(g["q"][:, i].contiguous(), g["k"][:, i].contiguous(),
                             g["v"][:, i].contiguous(), g["alpha"][:, i].contiguous(),
                             g["beta"][:, i].contiguous(), pool2, src.to(DEV), variant=GDN,
                             conv_w=w, conv_pool=cpool2, qk_l2norm=True, out_dtype=torch.float32)
        assert torch.equal(oi, o[:, i])
        assert torch.equal(pool2[src.long().to(DEV)], pool[dl[:, i].to(DEV)])
        assert torch.equal(cpool2[src.long().to(DEV)], cpool[dl[:, i].to(DEV)])


def test_spec_rollback_selects_accepted_prefix_state():
    """Rolling back to accepted length a picks src (a = 0) or dst[a-1]; the
    picked state equals the oracle state after a draft tokens."""
    N, D, H, d, P = 8, 4, 2, 64, 64
    base, dr, src, dst = _spec_setup(N, D, H, d, P, 11)
    pool = base["pool"].to(DEV)
    g = to(dr, DEV)
    glinattn_spec_decode(g["q"], g["k"], g["v"], g["alpha"], g["beta"], pool, src.to(DEV),
                         dst.to(DEV), variant=GDN, qk_l2norm=True)
    torch.cuda.synchronize()
    accept = dr["accept"].tolist()
    chosen = [int(src[n]) if a == 0 else int(dst[n, a - 1]) for n, a in enumerate(accept)]
    _, pool_ref, _ = oracle.spec_decode(GDN, f64(dr["q"]), f64(dr["k"]), f64(dr["v"]),
                                        f64(dr["alpha"]), f64(dr["beta"]), f64(base["pool"]),
                                        src.tolist(), dst.tolist(), None, None, True)
    for n, s in enumerate(chosen):
        assert relerr(pool[s], pool_ref[s]) <= TOL_S_BF16
