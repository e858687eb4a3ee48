"""Seeded random shapes for decode, speculative decode, verify + replay, the
SSD form, normalised linear attention and the selective scan, against the
oracle; and the decode front end bit for bit.

"Inference for linear attention and hybrid architectures": section "Two ways
to write the same computation" (decode is one read and one rank-one update of
the state per token) and section "Speculative decoding and PD disaggregation"
(slot-indexed pool; one state per draft position, or the drafts replayed from
the chosen position); "Long context, fast inference, smart decoding, and life
beyond attention", chapter "05 · State-space models" (the selective scan) and
section "Linear attention: removing softmax entirely" (the normalised form).  Shapes are drawn from a fixed seed: request counts
that do and do not fill the persistent grid, one to six heads, the head sizes
the kernels support, both forms, with and without the conv / L2 front end.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_02_gb300 import (GDN, GLA, NLA, glinattn_decode, glinattn_prefill, glinattn_replay,
                                     glinattn_selective_scan, glinattn_spec_decode, inputs)
from oracle.normalized import nla_prefill
from oracle.selective_scan import selective_scan

from helpers import NT, TOL_F32, TOL_O_BF16, TOL_S_BF16, f64, relerr, to

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _draw(n, seed, draw):
    rng = np.random.default_rng(seed)
    return [draw(rng) for _ in range(n)]


def _d(t):
    return None if t is None else t.to(DEV)


def _check_o(o, o_ref):
    if o.dtype == torch.bfloat16:
        err = np.abs(f64(o) - o_ref)
        assert (err <= np.abs(o_ref) * 2.0 ** -8 + TOL_O_BF16 * np.abs(o_ref).max()).all()
    else:
        assert relerr(o, o_ref) <= TOL_O_BF16


# ------------------------------------------------------------------ decode ------
_DECODE = _draw(8, 77, lambda r: (int(r.integers(1, 301)), int(r.integers(1, 7)), int(r.choice([16, 32, 64, 128])),
                                  int(r.choice([GLA, GDN])), bool(r.integers(0, 2))))


@pytest.mark.parametrize("N,H,d,variant,bf16_out", _DECODE)
def test_random_decode_matches_oracle(N, H, d, variant, bf16_out):
    P = N + 1 + (N * 7) % 13
    gdn = variant == GDN
    ex = inputs.gdn_decode(N, H, d, P, seed=N * 31 + H * 7 + d, variant_gdn=gdn)
    pool = ex["pool"].to(DEV)
    cpool = ex["conv_pool"].to(DEV) if gdn else None
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = glinattn_decode(ex["q"].to(DEV), ex["k"].to(DEV), ex["v"].to(DEV), ex["alpha"].to(DEV),
                        _d(ex["beta"]), pool, ex["slot_ids"].to(DEV), variant=variant,
                        conv_w=ex["conv_w"].to(DEV) if gdn else None, conv_pool=cpool, qk_l2norm=gdn,
                        out_dtype=torch.bfloat16 if bf16_out else torch.float32, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref, pool_ref, cpool_ref = oracle.decode(
        variant, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]), f64(ex["beta"]) if gdn else None,
        f64(ex["pool"]), ex["slot_ids"].tolist(), f64(ex["conv_w"]) if gdn else None,
        f64(ex["conv_pool"]) if gdn else None, gdn)
    _check_o(o, o_ref)
    sl = ex["slot_ids"].long()
    assert relerr(pool[sl.to(DEV)], pool_ref[sl.numpy()]) <= TOL_S_BF16
    untouched = torch.ones(P, dtype=torch.bool)
    untouched[sl] = False
    assert torch.equal(pool.cpu()[untouched], ex["pool"][untouched])
    if gdn:
        assert np.array_equal(f64(cpool), cpool_ref)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_front_end_bit_exact(d):
    """From a zero state with beta = 1 the delta-rule step writes k'^T v'
    (S = alpha (0 - ...) + beta k'^T v'), and a product of two bf16 values is
    exact in fp32: the written state reveals the kernel's bf16 k' and v', which
    equal the oracle's front end (conv with its cache, L2 norm, rounding)
    bit for bit."""
    N, H, P = 96, 3, 128
    ex = inputs.gdn_decode(N, H, d, P, seed=d + 5)
    ex["beta"] = torch.ones_like(ex["beta"])
    sl = ex["slot_ids"].long()
    ex["pool"][sl] = 0.0
    pool, cpool = ex["pool"].to(DEV), ex["conv_pool"].to(DEV)
    glinattn_decode(ex["q"].to(DEV), ex["k"].to(DEV), ex["v"].to(DEV), ex["alpha"].to(DEV), ex["beta"].to(DEV),
                    pool, ex["slot_ids"].to(DEV), variant=GDN, conv_w=ex["conv_w"].to(DEV), conv_pool=cpool,
                    qk_l2norm=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    _, kf, vf, _ = oracle.frontend(f64(ex["q"])[:, None], f64(ex["k"])[:, None], f64(ex["v"])[:, None],
                                   f64(ex["conv_w"]), f64(ex["conv_pool"])[sl.numpy()], True, True)
    want = np.einsum("nhi,nhj->nhij", kf[:, 0], vf[:, 0])
    got = f64(pool)[sl.numpy()]
    assert np.array_equal(got, want), int((got != want).sum())


# --------------------------------------------------------- speculative decode ----
_SPEC = _draw(6, 78, lambda r: (int(r.integers(1, 41)), int(r.integers(1, 13)), int(r.integers(1, 5)),
                                int(r.choice([64, 128])), int(r.choice([GLA, GDN]))))


@pytest.mark.parametrize("N,D,H,d,variant", _SPEC)
def test_random_spec_decode_matches_oracle(N, D, H, d, variant):
    gdn = variant == GDN
    P = N * (D + 1) + 3
    seed = N * 13 + D * 5 + H + d
    base = inputs.gdn_decode(N, H, d, P, seed=seed, variant_gdn=gdn)
    dr = inputs.spec_drafts(N, D, H, d, seed=seed + 100)
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(seed))
    src = perm[:N].to(torch.int32)
    dst = perm[N:N + N * D].to(torch.int32).reshape(N, D)
    pool, cpool = base["pool"].to(DEV), base["conv_pool"].to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = glinattn_spec_decode(dr["q"].to(DEV), dr["k"].to(DEV), dr["v"].to(DEV), dr["alpha"].to(DEV),
                             dr["beta"].to(DEV) if gdn else None, pool, src.to(DEV), dst.to(DEV), variant=variant,
                             conv_w=base["conv_w"].to(DEV) if gdn else None, conv_pool=cpool if gdn else None,
                             qk_l2norm=gdn, out_dtype=torch.float32, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref, pool_ref, cpool_ref = oracle.spec_decode(
        variant, f64(dr["q"]), f64(dr["k"]), f64(dr["v"]), f64(dr["alpha"]), f64(dr["beta"]) if gdn else None,
        f64(base["pool"]), src.tolist(), dst.tolist(), f64(base["conv_w"]) if gdn else None,
        f64(base["conv_pool"]) if gdn else None, gdn)
    assert relerr(o, o_ref) <= TOL_O_BF16
    dl = dst.long()
    assert relerr(pool[dl.to(DEV)], pool_ref[dl.numpy()]) <= TOL_S_BF16
    assert torch.equal(pool[src.long().to(DEV)].cpu(), base["pool"][src.long()])
    if gdn:
        assert np.array_equal(f64(cpool[dl.to(DEV)]), cpool_ref[dl.numpy()])


# ---------------------------------------------------------- verify + replay ------
_VERIFY = _draw(6, 79, lambda r: (int(r.integers(1, 41)), int(r.integers(1, 17)), int(r.integers(1, 5)),
                                  int(r.choice([GLA, GDN]))))


@pytest.mark.parametrize("N,D,H,variant", _VERIFY)
def test_random_verify_then_replay_matches_oracle(N, D, H, variant):
    """d = 128: the verify outputs come from the chunked form over the drafts
    (up to 16); the replay applies a random accepted prefix 0..D in place."""
    d = 128
    gdn = variant == GDN
    P = N * (D + 1) + 2
    seed = N * 17 + D * 3 + H
    base = inputs.gdn_decode(N, H, d, P, seed=seed, variant_gdn=gdn)
    dr = inputs.spec_drafts(N, D, H, d, seed=seed + 100)
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(seed))
    src = perm[:N].to(torch.int32)
    dst = perm[N:N + N * D].to(torch.int32).reshape(N, D)
    accept = torch.from_numpy(np.random.default_rng(seed).integers(0, D + 1, N).astype(np.int32))
    g = {k: (None if v is None else v.to(DEV)) for k, v in dr.items()}
    beta = g["beta"] if gdn else None
    w = base["conv_w"].to(DEV) if gdn else None
    pool, cpool = base["pool"].to(DEV), base["conv_pool"].to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = glinattn_spec_decode(g["q"], g["k"], g["v"], g["alpha"], beta, pool, src.to(DEV), None, variant=variant,
                             conv_w=w, conv_pool=cpool if gdn else None, qk_l2norm=gdn, out_dtype=torch.float32,
                             dev_status=status)
    glinattn_replay(g["k"], g["v"], g["alpha"], beta, pool, src.to(DEV), accept.to(DEV), q=g["q"], variant=variant,
                    conv_w=w, conv_pool=cpool if gdn else None, qk_l2norm=gdn, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref, pool_ref, cpool_ref = oracle.spec_decode(
        variant, f64(dr["q"]), f64(dr["k"]), f64(dr["v"]), f64(dr["alpha"]), f64(dr["beta"]) if gdn else None,
        f64(base["pool"]), src.tolist(), dst.tolist(), f64(base["conv_w"]) if gdn else None,
        f64(base["conv_pool"]) if gdn else None, gdn)
    assert relerr(o, o_ref) <= TOL_O_BF16
    pool, cpool = pool.cpu(), cpool.cpu()
    for n, a in enumerate(accept.tolist()):
        s = int(src[n])
        if a == 0:
            assert torch.equal(pool[s], base["pool"][s]), n
            continue
        assert relerr(pool[s], pool_ref[int(dst[n, a - 1])]) <= TOL_S_BF16, (n, a)
        if gdn:
            assert np.array_equal(f64(cpool[s]), cpool_ref[int(dst[n, a - 1])]), (n, a)
    others = torch.ones(P, dtype=torch.bool)
    others[src.long()] = False
    assert torch.equal(pool[others], base["pool"][others])


# ------------------------------------------------------------------ SSD form ----
_SSD = _draw(5, 80, lambda r: (int(r.integers(1, 4)), int(r.choice([1, 2, 4])), int(r.integers(1, 3)),
                               int(r.integers(1, 600))))


@pytest.mark.parametrize("B,G,per_group,T", _SSD)
def test_random_ssd_prefill_matches_oracle(B, G, per_group, T):
    """128 x 64 states, q / k heads shared by groups of heads."""
    H = G * per_group
    ex = inputs.ssd_prefill(B, H, G, T, seed=B * 100 + H * 10 + T, s0_std=0.05)
    g = to(ex, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, S, _ = glinattn_prefill(g["q"], g["k"], g["v"], g["alpha"], None, g["S0"], variant=GLA,
                               out_dtype=torch.float32, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref, S_ref = oracle.recurrence(GLA, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]),
                                     S0=f64(ex["S0"]), nthreads=NT)
    assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(S, S_ref) <= TOL_S_BF16


# -------------------------------------------------- normalised linear attention ----
_NLA = _draw(5, 81, lambda r: (int(r.integers(1, 4)), int(r.integers(1, 5)), int(r.integers(1, 600)),
                               bool(r.integers(0, 2))))


@pytest.mark.parametrize("B,H,T,start", _NLA)
def test_random_nla_prefill_matches_oracle(B, H, T, start):
    ex = inputs.nla_prefill(B, H, T, 128, seed=B * 100 + H * 10 + T, start=start)
    g = to(ex, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, S, _, z = glinattn_prefill(g["q"], g["k"], g["v"], None, None, g["S0"] if start else None, variant=NLA,
                                  z0=g["z0"] if start else None, out_dtype=torch.float32, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref, S_ref, z_ref = nla_prefill(f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["S0"]) if start else None,
                                      f64(ex["z0"]) if start else None, act_bf16=True)
    assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(S, S_ref) <= TOL_S_BF16 and relerr(z, z_ref) <= TOL_S_BF16


# ------------------------------------------------------------- selective scan ----
_SCAN = _draw(5, 82, lambda r: (int(r.integers(1, 4)), int(r.integers(1, 400)), int(r.integers(1, 700)),
                                int(r.choice([8, 16, 32])), bool(r.integers(0, 2))))


@pytest.mark.parametrize("B,T,D,N,start", _SCAN)
def test_random_selective_scan_matches_oracle(B, T, D, N, start):
    ex = inputs.selective_scan_inputs(B, T, D, N, seed=B * 1000 + T + D + N, start=start)
    g = to(ex, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y, h = glinattn_selective_scan(g["x"], g["delta"], g["Bm"], g["Cm"], g["A"], g["h0"] if start else None,
                                   out_dtype=torch.float32, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    y_ref, h_ref = selective_scan(f64(ex["x"]), f64(ex["delta"]), f64(ex["Bm"]), f64(ex["Cm"]), f64(ex["A"]),
                                  f64(ex["h0"]) if start else None)
    assert relerr(y, y_ref) <= TOL_F32 and relerr(h, h_ref) <= TOL_F32
