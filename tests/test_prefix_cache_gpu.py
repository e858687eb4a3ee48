"""GPU parity of prefix-cache checkpoints: the states and conv caches a prefill
emits at block boundaries, and whole-slot copies inside the state pool.

"Inference for linear attention and hybrid architectures", section "Prefix
caching has to be redone": a state summarises its whole prefix, so a prefix can
be reused only where a checkpoint (state and conv cache) was saved, and a
request that reuses one continues from its own copy of it (copy on write).  By
definition the checkpoint after t tokens is the state a prefill of those t
tokens ends with; continuing from it equals the one-shot prefill.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_02_gb300 import GDN, GLA, glinattn_decode, glinattn_prefill, glinattn_state_copy, inputs
from gated_deltanet_02_gb300.glinattn import DEV_BAD_SLOT

from helpers import TOL_F32, TOL_O_BF16, TOL_S_BF16, NT, f64, relerr, to

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _oracle_states(ex, variant, conv, conv_in=None):
    """Front end, then the recurrence keeping the state after every token."""
    q, k, v, _ = oracle.frontend(f64(ex["q"]), f64(ex["k"]), f64(ex["v"]),
                                 f64(ex.get("conv_w")) if conv else None, conv_in, conv,
                                 act_bf16=ex["q"].dtype == torch.bfloat16)
    beta = f64(ex["beta"]) if variant == GDN else None
    o, S, states = oracle.recurrence(variant, q, k, v, f64(ex["alpha"]), beta, f64(ex.get("S0")),
                                     return_states=True, nthreads=NT)
    return o, S, states


def _prefill(g, variant, conv, every, conv_in=None, conv_out=None, S0="from_inputs"):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = glinattn_prefill(g["q"], g["k"], g["v"], g["alpha"], g.get("beta"),
                           g.get("S0") if S0 == "from_inputs" else S0, variant=variant,
                           conv_w=g.get("conv_w") if conv else None, conv_in=conv_in,
                           conv_out=conv_out, qk_l2norm=conv, out_dtype=torch.float32,
                           dev_status=status, state_every=every)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out


@pytest.mark.parametrize("variant,T,every", [(GLA, 300, 64), (GLA, 256, 128), (GDN, 300, 64),
                                             (GDN, 257, 128), (GDN, 192, 192)])
def test_block_states_match_oracle(variant, T, every):
    """bf16, d=128 (the chunked tensor-core kernels): S_blocks[:, j] is the
    state after (j + 1) * every tokens; conv_blocks[:, j] the conv cache there."""
    conv = variant == GDN
    ex = (inputs.gdn_prefill if conv else inputs.gla_prefill)(2, 3, T, 128, seed=T + every)
    g = to(ex, DEV)
    o, S, c, Sb, cb = _prefill(g, variant, conv, every)
    assert Sb.shape == (2, T // every, 3, 128, 128)
    _, _, states = _oracle_states(ex, variant, conv)
    for j in range(T // every):
        assert relerr(Sb[:, j], states[:, (j + 1) * every - 1]) <= TOL_S_BF16, j
        if conv:  # raw inputs: exact
            P = (j + 1) * every
            _, _, _, c_ref = oracle.frontend(f64(ex["q"][:, :P]), f64(ex["k"][:, :P]), f64(ex["v"][:, :P]),
                                             f64(ex["conv_w"]), None, True)
            assert np.array_equal(f64(cb[:, j]), c_ref), j
    # emitting checkpoints leaves the layer's own results unchanged, bit for bit
    o2, S2, c2 = glinattn_prefill(g["q"], g["k"], g["v"], g["alpha"], g.get("beta"), g.get("S0"),
                                  variant=variant, conv_w=g.get("conv_w") if conv else None,
                                  qk_l2norm=conv, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(S, S2)
    if conv:
        assert torch.equal(c, c2)


@pytest.mark.parametrize("every", [1, 2, 10])
def test_block_states_fp32_any_length(every):
    """fp32 inputs (the token-serial kernel) take any block length.  A non-zero
    conv history is handed in and conv_out aliases conv_in: blocks that end
    within the first three tokens still see the history as it was."""
    T, H, d = 37, 2, 64
    ex = inputs.gdn_prefill(2, H, T, d, seed=every, dtype=torch.float32)
    g = to(ex, DEV)
    gen = torch.Generator().manual_seed(5)
    cin = torch.randn(2, 3, 3 * H * d, generator=gen)
    cbuf = cin.to(DEV).clone()
    o, S, c, Sb, cb = _prefill(g, GDN, True, every, conv_in=cbuf, conv_out=cbuf)
    o_ref, S_ref, states = _oracle_states(ex, GDN, True, conv_in=f64(cin))
    assert relerr(o, o_ref) <= TOL_F32 and relerr(S, S_ref) <= TOL_F32
    for j in range(T // every):
        P = (j + 1) * every
        assert relerr(Sb[:, j], states[:, P - 1]) <= TOL_F32, j
        _, _, _, c_ref = oracle.frontend(f64(ex["q"][:, :P]), f64(ex["k"][:, :P]), f64(ex["v"][:, :P]),
                                         f64(ex["conv_w"]), f64(cin), True, act_bf16=False)
        assert np.array_equal(f64(cb[:, j]), c_ref), j


def test_block_length_longer_than_segment_emits_nothing():
    ex = inputs.gla_prefill(1, 2, 100, 128, seed=2)
    g = to(ex, DEV)
    o, S, _, Sb, cb = _prefill(g, GLA, False, 128)
    assert Sb.shape[1] == 0 and cb is None
    o_ref, S_ref, _ = oracle.layer_prefill(GLA, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]),
                                           nthreads=NT)
    assert relerr(o, o_ref) <= TOL_O_BF16 and relerr(S, S_ref) <= TOL_S_BF16


@pytest.mark.parametrize("variant", [GLA, GDN])
def test_resume_from_checkpoint_equals_one_shot(variant):
    """Continue from (S_blocks[:, j], conv_blocks[:, j]) over the rest of the
    prompt: the outputs and final state equal the one-shot prefill's."""
    T, every = 320, 64
    conv = variant == GDN
    ex = (inputs.gdn_prefill if conv else inputs.gla_prefill)(2, 2, T, 128, seed=77)
    g = to(ex, DEV)
    o, S, c, Sb, cb = _prefill(g, variant, conv, every)
    o_ref, S_ref, c_ref = oracle.layer_prefill(variant, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]),
                                               f64(ex["alpha"]), f64(ex.get("beta")) if conv else None,
                                               f64(ex.get("S0")), f64(ex.get("conv_w")) if conv else None,
                                               None, conv, nthreads=NT)
    for j in (0, 2, 3):
        P = (j + 1) * every
        rest = {key: (val[:, P:].contiguous() if key in ("q", "k", "v", "alpha", "beta") and val is not None
                      else val) for key, val in g.items()}
        o2, S2, c2 = glinattn_prefill(rest["q"], rest["k"], rest["v"], rest["alpha"], rest.get("beta"),
                                      Sb[:, j].contiguous(), variant=variant,
                                      conv_w=g.get("conv_w") if conv else None,
                                      conv_in=cb[:, j].contiguous() if conv else None, qk_l2norm=conv,
                                      out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert relerr(o2, o_ref[:, P:]) <= TOL_O_BF16, j
        assert relerr(S2, S_ref) <= TOL_S_BF16, j
        assert relerr(o2, f64(o[:, P:])) <= TOL_O_BF16, j
        if conv:
            assert np.array_equal(f64(c2), c_ref) and torch.equal(c2, c)


@pytest.mark.parametrize("conv_dtype", [torch.bfloat16, torch.float32, None])
def test_state_copy_bit_exact(conv_dtype):
    P, H, d = 10, 4, 128
    gen = torch.Generator().manual_seed(11)
    pool = torch.randn(P, H, d, d, generator=gen)
    cpool = None if conv_dtype is None else torch.randn(P, 3, 3 * H * d, generator=gen).to(conv_dtype)
    src, dst = [1, 3, 3, 7], [0, 2, 5, 9]
    want = pool.numpy().copy()
    want[dst] = pool.numpy()[src]
    pool_d = pool.to(DEV)
    cpool_d = None if cpool is None else cpool.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    glinattn_state_copy(pool_d, torch.tensor(src, dtype=torch.int32, device=DEV),
                        torch.tensor(dst, dtype=torch.int32, device=DEV), conv_pool=cpool_d, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(pool_d.cpu().numpy(), want)
    if cpool is not None:
        cwant = cpool.clone()
        cwant[dst] = cpool[src]
        assert torch.equal(cpool_d.cpu(), cwant)


def test_state_copy_bad_slot_is_flagged_and_skipped():
    P, H, d = 6, 2, 64
    pool = torch.randn(P, H, d, d, generator=torch.Generator().manual_seed(3))
    pool_d = pool.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    glinattn_state_copy(pool_d, torch.tensor([1, 9, -1], dtype=torch.int32, device=DEV),
                        torch.tensor([0, 4, 5], dtype=torch.int32, device=DEV), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & DEV_BAD_SLOT
    want = pool.clone()
    want[0] = pool[1]
    assert torch.equal(pool_d.cpu(), want)  # slots 4 and 5 untouched


def test_copy_on_write_decode_leaves_checkpoint_intact():
    """A shared prompt is prefilled once into a checkpoint slot; two requests
    copy it and decode different tokens.  Their outputs equal the oracle's
    decode from the prompt's state, and the checkpoint slot is unchanged."""
    H, d, T, P = 2, 128, 130, 8
    ex = inputs.gdn_prefill(1, H, T, d, seed=13)
    g = to(ex, DEV)
    pool = torch.zeros(P, H, d, d, device=DEV)
    cpool = torch.zeros(P, 3, 3 * H * d, dtype=torch.bfloat16, device=DEV)
    ck = 6
    glinattn_prefill(g["q"], g["k"], g["v"], g["alpha"], g["beta"], g["S0"], variant=GDN,
                     conv_w=g["conv_w"], qk_l2norm=True, out_dtype=torch.float32,
                     S_T=pool[ck:ck + 1], conv_out=cpool[ck:ck + 1])
    slots = torch.tensor([2, 5], dtype=torch.int32, device=DEV)
    glinattn_state_copy(pool, torch.tensor([ck, ck], dtype=torch.int32, device=DEV), slots, conv_pool=cpool)
    saved, csaved = pool[ck].clone(), cpool[ck].clone()
    dx = inputs.gdn_decode(2, H, d, P, seed=14)
    dg = to(dx, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = glinattn_decode(dg["q"], dg["k"], dg["v"], dg["alpha"], dg["beta"], pool, slots, variant=GDN,
                        conv_w=g["conv_w"], conv_pool=cpool, qk_l2norm=True, out_dtype=torch.float32,
                        dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(pool[ck], saved) and torch.equal(cpool[ck], csaved)
    _, S_ref, c_ref = oracle.layer_prefill(GDN, f64(ex["q"]), f64(ex["k"]), f64(ex["v"]), f64(ex["alpha"]),
                                           f64(ex["beta"]), f64(ex["S0"]), f64(ex["conv_w"]), None, True,
                                           nthreads=NT)
    pool_ref = np.zeros((P, H, d, d))
    cpool_ref = np.zeros((P, 3, 3 * H * d))
    pool_ref[[2, 5]] = S_ref[0]
    cpool_ref[[2, 5]] = c_ref[0]
    o_ref, pool_ref, _ = oracle.decode(GDN, f64(dx["q"]), f64(dx["k"]), f64(dx["v"]), f64(dx["alpha"]),
                                       f64(dx["beta"]), pool_ref, [2, 5], f64(ex["conv_w"]), cpool_ref, True)
    assert relerr(o, o_ref) <= TOL_O_BF16
    assert relerr(pool[[2, 5]], pool_ref[[2, 5]]) <= TOL_S_BF16
