"""GPU parity of Gated DeltaNet with grouped q / k heads (several value heads
sharing one q / k head), on the token-serial kernel: prefill, decode and
speculative decode against the oracle, which expands each group to its heads.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_02_gb300 import GDN, glinattn_decode, glinattn_prefill, glinattn_spec_decode

from helpers import TOL_O_BF16, TOL_S_BF16, f64, relerr

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _inputs(lead, H, Hq, d, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    unit = lambda x: x / x.norm(dim=-1, keepdim=True)
    q = unit(torch.randn(*lead, Hq, d, generator=g)).to(dtype)
    k = unit(torch.randn(*lead, Hq, d, generator=g)).to(dtype)
    v = torch.randn(*lead, H, d, generator=g).to(dtype)
    beta = torch.sigmoid(torch.randn(*lead, H, generator=g))
    alpha = torch.sigmoid(torch.randn(*lead, H, generator=g) + 3.0)
    return q, k, v, alpha, beta


def test_grouped_gdn_prefill():
    B, T, H, Hq, d = 2, 100, 4, 2, 128
    q, k, v, alpha, beta = _inputs((B, T), H, Hq, d, seed=1)
    S0 = torch.randn(B, H, d, d, generator=torch.Generator().manual_seed(2)) * 0.01
    o, S, _ = glinattn_prefill(q.to(DEV), k.to(DEV), v.to(DEV), alpha.to(DEV), beta.to(DEV), S0.to(DEV),
                               variant=GDN, qk_l2norm=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, S_ref, _ = oracle.layer_prefill(GDN, f64(q), f64(k), f64(v), f64(alpha), f64(beta), f64(S0), None,
                                           None, True)
    assert relerr(o, o_ref) <= TOL_O_BF16 and relerr(S, S_ref) <= TOL_S_BF16


def test_grouped_gdn_decode_and_spec():
    N, D, H, Hq, d, P = 6, 3, 4, 1, 128, 30
    gen = torch.Generator().manual_seed(3)
    pool = torch.randn(P, H, d, d, generator=gen) * 0.01
    perm = torch.randperm(P, generator=gen)
    slots = perm[:N].to(torch.int32)
    q, k, v, alpha, beta = _inputs((N,), H, Hq, d, seed=4)
    pool_d = pool.to(DEV)
    o = glinattn_decode(q.to(DEV), k.to(DEV), v.to(DEV), alpha.to(DEV), beta.to(DEV), pool_d, slots.to(DEV),
                        variant=GDN, qk_l2norm=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, pool_ref, _ = oracle.decode(GDN, f64(q), f64(k), f64(v), f64(alpha), f64(beta), f64(pool),
                                       slots.tolist(), None, None, True)
    sl = slots.long()
    assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(pool_d[sl.to(DEV)], pool_ref[sl.numpy()]) <= TOL_S_BF16
    # speculative decode from the same start states
    qd, kd, vd, ad, bd = _inputs((N, D), H, Hq, d, seed=5)
    src = perm[:N].to(torch.int32)
    dst = perm[N:N + N * D].to(torch.int32).reshape(N, D)
    pool2 = pool.to(DEV)
    os_ = glinattn_spec_decode(qd.to(DEV), kd.to(DEV), vd.to(DEV), ad.to(DEV), bd.to(DEV), pool2, src.to(DEV),
                               dst.to(DEV), variant=GDN, qk_l2norm=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    os_ref, pool2_ref, _ = oracle.spec_decode(GDN, f64(qd), f64(kd), f64(vd), f64(ad), f64(bd), f64(pool),
                                              src.tolist(), dst.tolist(), None, None, True)
    dl = dst.long()
    assert relerr(os_, os_ref) <= TOL_O_BF16
    assert relerr(pool2[dl.to(DEV)], pool2_ref[dl.numpy()]) <= TOL_S_BF16
    assert np.isfinite(f64(pool2)).all()
