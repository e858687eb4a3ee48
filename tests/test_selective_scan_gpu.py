"""GPU parity of Mamba's selective scan against the oracle.

"Long context, fast inference, smart decoding, and life beyond attention",
chapter "05 · State-space models: the architectural alternative": with
dt = softplus(delta), h_t = exp(dt A) h_{t-1} + dt B_t x_t and y_t = h_t C_t,
per channel and state index.  All GPU arithmetic is fp32, so fp32 and bf16
inputs are both held to the fp32 tolerance (bf16 values are exact in the
oracle's fp64).
"""
import numpy as np
import pytest
import torch

from gated_deltanet_02_gb300 import glinattn_selective_scan, glinattn_selective_scan_decode, inputs
from gated_deltanet_02_gb300.glinattn import DEV_BAD_SLOT
from oracle.selective_scan import selective_scan, selective_scan_decode

from helpers import TOL_F32, TOL_O_BF16, f64, relerr, to

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _run(g, h0=None, out_dtype=torch.float32, h_T=None):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y, h = glinattn_selective_scan(g["x"], g["delta"], g["Bm"], g["Cm"], g["A"], h0, out_dtype=out_dtype,
                                   h_T=h_T, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return y, h


def _ref(ex, h0=None):
    return selective_scan(f64(ex["x"]), f64(ex["delta"]), f64(ex["Bm"]), f64(ex["Cm"]), f64(ex["A"]), h0)


@pytest.mark.parametrize("T", [1, 63, 64, 200, 300])
@pytest.mark.parametrize("N", [8, 16, 32])
def test_scan_fp32(T, N):
    """D = 200: a ragged block of channels past the first 128."""
    ex = inputs.selective_scan_inputs(2, T, 200, N, seed=T + N, start=True)
    g = to(ex, DEV)
    y, h = _run(g, g["h0"])
    y_ref, h_ref = _ref(ex, f64(ex["h0"]))
    assert relerr(y, y_ref) <= TOL_F32 and relerr(h, h_ref) <= TOL_F32


@pytest.mark.parametrize("T", [1, 63, 65, 130])
@pytest.mark.parametrize("N", [8, 16, 32])
def test_scan_many_channels(T, N):
    """B = 4 sequences of D = 1000 channels (a ragged last block of channels),
    T ending inside, at and past a 64-token chunk."""
    ex = inputs.selective_scan_inputs(4, T, 1000, N, seed=40 + T + N, start=True)
    g = to(ex, DEV)
    y, h = _run(g, g["h0"])
    y_ref, h_ref = _ref(ex, f64(ex["h0"]))
    assert relerr(y, y_ref) <= TOL_F32 and relerr(h, h_ref) <= TOL_F32


def test_scan_many_channels_bf16_state_in_place():
    ex = inputs.selective_scan_inputs(4, 70, 1024, 16, seed=44, dtype=torch.bfloat16, start=True)
    g = to(ex, DEV)
    h = g["h0"].clone()
    yb, h2 = _run(g, h, out_dtype=torch.bfloat16, h_T=h)
    assert h2.data_ptr() == h.data_ptr()
    y_ref, h_ref = _ref(ex, f64(ex["h0"]))
    err = np.abs(f64(yb) - y_ref)
    assert (err <= np.abs(y_ref) * 2.0 ** -8 + TOL_O_BF16 * np.abs(y_ref).max()).all()
    assert relerr(h, h_ref) <= TOL_F32


def test_scan_bf16_inputs_and_outputs():
    ex = inputs.selective_scan_inputs(2, 150, 256, 16, seed=3, dtype=torch.bfloat16)
    g = to(ex, DEV)
    y, h = _run(g)
    y_ref, h_ref = _ref(ex)
    assert relerr(y, y_ref) <= TOL_F32 and relerr(h, h_ref) <= TOL_F32
    yb, _ = _run(g, out_dtype=torch.bfloat16)
    err = np.abs(f64(yb) - y_ref)
    assert (err <= np.abs(y_ref) * 2.0 ** -8 + TOL_O_BF16 * np.abs(y_ref).max()).all()


def test_scan_segments_chain_and_state_in_place():
    T = 333
    ex = inputs.selective_scan_inputs(1, T, 128, 16, seed=5)
    g = to(ex, DEV)
    h = torch.zeros(1, 128, 16, device=DEV)
    ys = []
    for s, e in ((0, 70), (70, 70), (70, 72), (72, T)):  # includes an empty segment
        seg = {k: (v[:, s:e].contiguous() if k in ("x", "delta", "Bm", "Cm") else v) for k, v in g.items()}
        y, h2 = _run(seg, h, h_T=h)  # h_T over h0
        assert h2.data_ptr() == h.data_ptr()
        ys.append(y)
    y_ref, h_ref = _ref(ex)
    assert relerr(torch.cat(ys, 1), y_ref) <= TOL_F32 and relerr(h, h_ref) <= TOL_F32


def test_scan_full_size_sampled():
    """B=2, T=4096, D=2048 channels (d_model 1024 expanded 2x), N=16 states:
    eight channels checked in full (channels are independent)."""
    ex = inputs.selective_scan_inputs(2, 4096, 2048, 16, seed=0, device=DEV, dtype=torch.bfloat16)
    y, h = _run(ex)
    ds = [0, 127, 128, 700, 1023, 1500, 2046, 2047]
    sub = {k: ex[k][..., ds] for k in ("x", "delta")}
    y_ref, h_ref = selective_scan(f64(sub["x"]), f64(sub["delta"]), f64(ex["Bm"]), f64(ex["Cm"]), f64(ex["A"][ds]))
    assert relerr(y[..., ds], y_ref) <= TOL_F32
    assert relerr(h[:, ds], h_ref) <= TOL_F32


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_scan_decode(dtype):
    R, D, N, P = 12, 300, 16, 30
    ex = inputs.selective_scan_inputs(R, 1, D, N, seed=9, dtype=dtype)
    gen = torch.Generator().manual_seed(9)
    pool = torch.randn(P, D, N, generator=gen) * 0.1
    slots = torch.randperm(P, generator=gen)[:R].to(torch.int32)
    g = to(ex, DEV)
    pool_d = pool.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = glinattn_selective_scan_decode(g["x"][:, 0].contiguous(), g["delta"][:, 0].contiguous(),
                                       g["Bm"][:, 0].contiguous(), g["Cm"][:, 0].contiguous(), g["A"], pool_d,
                                       slots.to(DEV), out_dtype=torch.float32, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    y_ref, pool_ref = selective_scan_decode(f64(ex["x"][:, 0]), f64(ex["delta"][:, 0]), f64(ex["Bm"][:, 0]),
                                            f64(ex["Cm"][:, 0]), f64(ex["A"]), f64(pool), slots.tolist())
    sl = slots.long()
    assert relerr(y, y_ref) <= TOL_F32
    assert relerr(pool_d[sl.to(DEV)], pool_ref[sl.numpy()]) <= TOL_F32
    untouched = torch.ones(P, dtype=torch.bool)
    untouched[sl] = False
    assert torch.equal(pool_d.cpu()[untouched], pool[untouched])


def test_scan_decode_bad_slot_is_flagged_and_skipped():
    R, D, N, P = 3, 64, 8, 5
    ex = inputs.selective_scan_inputs(R, 1, D, N, seed=2)
    g = to(ex, DEV)
    pool = torch.randn(P, D, N, device=DEV)
    before = pool.clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    glinattn_selective_scan_decode(g["x"][:, 0].contiguous(), g["delta"][:, 0].contiguous(),
                                   g["Bm"][:, 0].contiguous(), g["Cm"][:, 0].contiguous(), g["A"], pool,
                                   torch.tensor([1, 7, -2], dtype=torch.int32, device=DEV), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & DEV_BAD_SLOT
    assert torch.equal(pool[[0, 2, 3, 4]], before[[0, 2, 3, 4]])
    assert not torch.equal(pool[1], before[1])


def test_scan_zero_length_segment_copies_the_state():
    ex = inputs.selective_scan_inputs(2, 0, 96, 8, seed=12, start=True)
    g = to(ex, DEV)
    y, h = _run(g, g["h0"])
    assert y.numel() == 0 and torch.equal(h, g["h0"])
    y, h = _run(g)  # no start state: zeros
    assert torch.equal(h, torch.zeros_like(h))
