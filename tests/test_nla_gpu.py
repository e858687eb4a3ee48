"""GPU parity of normalised kernelised linear attention against the oracle.

"Long context, fast inference, smart decoding, and life beyond attention",
section "Linear attention: removing softmax entirely": phi = elu + 1 on q and
k, a running state S and normaliser z, o = phi(q) S / (phi(q) . z + 1e-6).
Prefill (chunked and token-serial), segments handing (S, z) on, decode,
speculative decode and replay are checked.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_02_gb300 import (NLA, glinattn_decode, glinattn_prefill, glinattn_replay,
                                     glinattn_spec_decode, inputs)
from oracle.normalized import nla_decode, nla_prefill, nla_spec_decode

from helpers import TOL_F32, TOL_O_BF16, TOL_S_BF16, f64, relerr, to

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _prefill(g, S0=None, z0=None, out_dtype=torch.float32):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, S, _, z = glinattn_prefill(g["q"], g["k"], g["v"], None, None, S0, variant=NLA, z0=z0,
                                  out_dtype=out_dtype, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return o, S, z


def _ref(ex, start=True):
    return nla_prefill(f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["S0"]) if start else None,
                       f64(ex["z0"]) if start else None, act_bf16=ex["q"].dtype == torch.bfloat16)


@pytest.mark.parametrize("d,Hq", [(16, 2), (64, 2), (128, 2), (128, 1)])
def test_nla_prefill_fp32(d, Hq):
    ex = inputs.nla_prefill(2, 2, 77, d, Hq=Hq, seed=d + Hq, dtype=torch.float32, start=True)
    g = to(ex, DEV)
    o, S, z = _prefill(g, g["S0"], g["z0"])
    o_ref, S_ref, z_ref = _ref(ex)
    assert relerr(o, o_ref) <= TOL_F32 and relerr(S, S_ref) <= TOL_F32 and relerr(z, z_ref) <= TOL_F32


@pytest.mark.parametrize("T", [1, 63, 64, 200, 300])
def test_nla_prefill_bf16(T):
    ex = inputs.nla_prefill(2, 3, T, 128, seed=T, start=T % 2 == 0)
    g = to(ex, DEV)
    start = T % 2 == 0
    o, S, z = _prefill(g, g["S0"], g["z0"])
    o_ref, S_ref, z_ref = _ref(ex, start)
    assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(S, S_ref) <= TOL_S_BF16 and relerr(z, z_ref) <= TOL_S_BF16


def test_nla_segments_hand_state_and_normaliser_on():
    T = 333
    ex = inputs.nla_prefill(1, 2, T, 128, seed=4)
    g = to(ex, DEV)
    S, z, outs = None, None, []
    for s, e in ((0, 70), (70, 72), (72, T)):
        seg = {key: (val[:, s:e].contiguous() if key in ("q", "k", "v") else val) for key, val in g.items()}
        o, S, z = _prefill(seg, S, z)
        outs.append(o)
    o_ref, S_ref, z_ref = _ref(ex, start=False)
    assert relerr(torch.cat(outs, 1), o_ref) <= TOL_O_BF16
    assert relerr(S, S_ref) <= TOL_S_BF16 and relerr(z, z_ref) <= TOL_S_BF16


@pytest.mark.parametrize("d,dtype", [(64, torch.bfloat16), (128, torch.bfloat16), (128, torch.float32)])
def test_nla_decode(d, dtype):
    N, H, P = 10, 3, 24
    dx = inputs.nla_decode(N, H, d, P, seed=d, dtype=dtype)
    g = to(dx, DEV)
    pool, zpool = g["pool"].clone(), g["zpool"].clone()
    o = glinattn_decode(g["q"], g["k"], g["v"], None, None, pool, g["slot_ids"], variant=NLA, z_pool=zpool,
                        out_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, pool_ref, zpool_ref = nla_decode(f64(dx["q"]), f64(dx["k"]), f64(dx["v"]), f64(dx["pool"]),
                                            f64(dx["zpool"]), dx["slot_ids"].tolist(),
                                            act_bf16=dtype == torch.bfloat16)
    tol_o, tol_s = (TOL_O_BF16, TOL_S_BF16) if dtype == torch.bfloat16 else (TOL_F32, TOL_F32)
    sl = dx["slot_ids"].long()
    assert relerr(o, o_ref) <= tol_o
    assert relerr(pool[sl.to(DEV)], pool_ref[sl.numpy()]) <= tol_s
    assert relerr(zpool[sl.to(DEV)], zpool_ref[sl.numpy()]) <= tol_s
    untouched = torch.ones(P, dtype=torch.bool)
    untouched[sl] = False
    assert torch.equal(zpool.cpu()[untouched], dx["zpool"][untouched])


@pytest.mark.parametrize("d", [64, 128])
def test_nla_spec_decode_and_replay(d):
    N, D, H = 5, 4, 2
    P = N * (1 + D)
    dx = inputs.nla_decode(N, H, d, P, seed=11 + d, D=D)
    g = to(dx, DEV)
    src = dx["perm"][:N].to(torch.int32)
    dst = dx["perm"][N:N + N * D].to(torch.int32).reshape(N, D)
    pool, zpool = g["pool"].clone(), g["zpool"].clone()
    o = glinattn_spec_decode(g["q"], g["k"], g["v"], None, None, pool, src.to(DEV), dst.to(DEV), variant=NLA,
                             z_pool=zpool, out_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, pool_ref, zpool_ref = nla_spec_decode(f64(dx["q"]), f64(dx["k"]), f64(dx["v"]), f64(dx["pool"]),
                                                 f64(dx["zpool"]), src.tolist(), dst.tolist())
    dl = dst.long()
    assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(pool[dl.to(DEV)], pool_ref[dl.numpy()]) <= TOL_S_BF16
    assert relerr(zpool[dl.to(DEV)], zpool_ref[dl.numpy()]) <= TOL_S_BF16
    # verify only + replay lands on the per-draft states bit for bit
    pool2, zpool2 = g["pool"].clone(), g["zpool"].clone()
    o2 = glinattn_spec_decode(g["q"], g["k"], g["v"], None, None, pool2, src.to(DEV), None, variant=NLA,
                              z_pool=zpool2, out_dtype=torch.float32)
    accept = torch.tensor([0, 4, 1, 3, 2], dtype=torch.int32)
    glinattn_replay(g["k"], g["v"], None, None, pool2, src.to(DEV), accept.to(DEV), q=g["q"], variant=NLA,
                    z_pool=zpool2)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)
    for n, a in enumerate(accept.tolist()):
        s = int(src[n])
        want_S = g["pool"][s] if a == 0 else pool[int(dst[n, a - 1])]
        want_z = g["zpool"][s] if a == 0 else zpool[int(dst[n, a - 1])]
        assert torch.equal(pool2[s], want_S) and torch.equal(zpool2[s], want_z), (n, a)


def test_nla_chunked_grouped_head_dim_64():
    """Chunked path with two q / k heads for four heads of value size 64."""
    ex = inputs.nla_prefill(2, 4, 150, 128, Hq=2, dv=64, seed=31, start=True)
    g = to(ex, DEV)
    o, S, z = _prefill(g, g["S0"], g["z0"])
    o_ref, S_ref, z_ref = _ref(ex)
    assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(S, S_ref) <= TOL_S_BF16 and relerr(z, z_ref) <= TOL_S_BF16


def test_nla_bf16_output_and_normaliser_in_place():
    """bf16 outputs (one rounding of the normalised value), z_T over z0."""
    ex = inputs.nla_prefill(1, 2, 190, 128, seed=32, start=True)
    g = to(ex, DEV)
    z = g["z0"].clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, S, _, z_out = glinattn_prefill(g["q"], g["k"], g["v"], None, None, g["S0"], variant=NLA, z0=z, z_T=z,
                                      out_dtype=torch.bfloat16, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and z_out.data_ptr() == z.data_ptr()
    o_ref, S_ref, z_ref = _ref(ex)
    err = np.abs(f64(o) - o_ref)
    assert (err <= np.abs(o_ref) * 2.0 ** -8 + TOL_O_BF16 * np.abs(o_ref).max()).all()
    assert relerr(z, z_ref) <= TOL_S_BF16


def test_nla_full_size_sampled():
    """B=4, H=16, T=4096, d=128 (the gated linear attention prefill shape);
    units (0, 0) and (3, 15) in full."""
    ex = inputs.nla_prefill(4, 16, 4096, 128, seed=0, device=DEV)
    o, S, z = _prefill(ex)
    for b, h in ((0, 0), (3, 15)):
        sub = {key: ex[key][b:b + 1, :, h:h + 1] for key in ("q", "k", "v")}
        o_ref, S_ref, z_ref = nla_prefill(f64(sub["q"]), f64(sub["k"]), f64(sub["v"]))
        assert relerr(o[b:b + 1, :, h:h + 1], o_ref) <= TOL_O_BF16, (b, h)
        assert relerr(S[b:b + 1, h:h + 1], S_ref) <= TOL_S_BF16, (b, h)
        assert relerr(z[b:b + 1, h:h + 1], z_ref) <= TOL_S_BF16, (b, h)


def test_nla_zero_length_segment_hands_state_and_normaliser_on():
    ex = inputs.nla_prefill(2, 2, 0, 64, seed=40, dtype=torch.float32, start=True)
    g = to(ex, DEV)
    o, S, z = _prefill(g, g["S0"], g["z0"])
    assert o.numel() == 0
    assert torch.equal(S, g["S0"]) and torch.equal(z, g["z0"])


def test_nla_decode_bad_slot_is_flagged_and_skipped():
    from gated_deltanet_02_gb300.glinattn import DEV_BAD_SLOT
    dx = inputs.nla_decode(3, 2, 64, 6, seed=41)
    g = to(dx, DEV)
    pool, zpool = g["pool"].clone(), g["zpool"].clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    glinattn_decode(g["q"], g["k"], g["v"], None, None, pool, torch.tensor([1, 9, 4], dtype=torch.int32,
                    device=DEV), variant=NLA, z_pool=zpool, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & DEV_BAD_SLOT
    for s in (0, 2, 3, 5):
        assert torch.equal(pool[s], g["pool"][s]) and torch.equal(zpool[s], g["zpool"][s])
    assert not torch.equal(zpool[1], g["zpool"][1])
