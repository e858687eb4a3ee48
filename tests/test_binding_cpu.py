"""Host-side checks of the Python binding: shapes, dtypes and argument
combinations are rejected before anything reaches the library (CPU tensors,
no GPU needed)."""
import pytest
import torch

from gated_deltanet_02_gb300 import (GDN, GLA, NLA, glinattn_decode, glinattn_prefill, glinattn_replay,
                                     glinattn_selective_scan, glinattn_selective_scan_decode,
                                     glinattn_spec_decode, glinattn_state_copy)


def _bf(*s):
    return torch.zeros(*s, dtype=torch.bfloat16)


def _f(*s):
    return torch.zeros(*s, dtype=torch.float32)


def test_prefill_shape_and_dtype_checks():
    q, k, v = _bf(1, 8, 2, 16), _bf(1, 8, 2, 16), _bf(1, 8, 2, 16)
    with pytest.raises(ValueError):  # alpha of the wrong length
        glinattn_prefill(q, k, v, _f(1, 7, 2), variant=GLA)
    with pytest.raises(TypeError):   # alpha must be fp32
        glinattn_prefill(q, k, v, _bf(1, 8, 2), variant=GLA)
    with pytest.raises(TypeError):   # k in another dtype than q
        glinattn_prefill(q, k.float(), v, _f(1, 8, 2), variant=GLA)
    with pytest.raises(ValueError):  # S0 shape
        glinattn_prefill(q, k, v, _f(1, 8, 2), None, _f(1, 2, 16, 8), variant=GLA)
    with pytest.raises(ValueError):  # non-contiguous input
        glinattn_prefill(_bf(1, 2, 8, 16).transpose(1, 2), k, v, _f(1, 8, 2), variant=GLA)
    with pytest.raises(ValueError):  # negative block length
        glinattn_prefill(q, k, v, _f(1, 8, 2), variant=GLA, state_every=-1)
    with pytest.raises(ValueError):  # z0 of the wrong shape for the normalised variant
        glinattn_prefill(q, k, v, None, variant=NLA, z0=_f(1, 2, 8))


def test_grouped_heads_shapes():
    q, k = _bf(1, 8, 1, 16), _bf(1, 8, 1, 16)   # one q / k head
    v = _bf(1, 8, 4, 16)                         # four value heads
    with pytest.raises(ValueError):  # alpha is per value head
        glinattn_prefill(q, k, v, _f(1, 8, 1), variant=GLA)
    with pytest.raises(ValueError):  # the state is per value head
        glinattn_prefill(q, k, v, _f(1, 8, 4), None, _f(1, 1, 16, 16), variant=GLA)


def test_decode_spec_replay_checks():
    pool = _f(4, 2, 16, 16)
    q, k, v = _bf(3, 2, 16), _bf(3, 2, 16), _bf(3, 2, 16)
    with pytest.raises(TypeError):   # slot ids must be int32
        glinattn_decode(q, k, v, _f(3, 2), _f(3, 2), pool, torch.zeros(3, dtype=torch.int64))
    with pytest.raises(ValueError):  # the normaliser pool must match the state pool
        glinattn_decode(q, k, v, None, None, pool, torch.zeros(3, dtype=torch.int32), variant=NLA,
                        z_pool=_f(4, 2, 8))
    qd, kd, vd = _bf(3, 2, 2, 16), _bf(3, 2, 2, 16), _bf(3, 2, 2, 16)
    with pytest.raises(ValueError):  # destinations are [N, D]
        glinattn_spec_decode(qd, kd, vd, _f(3, 2, 2), _f(3, 2, 2), pool, torch.zeros(3, dtype=torch.int32),
                             torch.zeros(3, dtype=torch.int32))
    with pytest.raises(ValueError):  # a conv needs the raw q of the drafts
        glinattn_replay(kd, vd, _f(3, 2, 2), _f(3, 2, 2), pool, torch.zeros(3, dtype=torch.int32),
                        torch.zeros(3, dtype=torch.int32), variant=GDN, conv_w=_f(96, 4), conv_pool=_bf(4, 3, 96))


def test_state_copy_and_scan_checks():
    pool = _f(4, 2, 16, 16)
    with pytest.raises(TypeError):
        glinattn_state_copy(pool, torch.zeros(2, dtype=torch.int64), torch.zeros(2, dtype=torch.int32))
    with pytest.raises(ValueError):  # conv pool of the wrong channel count
        glinattn_state_copy(pool, torch.zeros(2, dtype=torch.int32), torch.ones(2, dtype=torch.int32),
                            conv_pool=_bf(4, 3, 95))
    x = _f(1, 8, 32)
    with pytest.raises(ValueError):  # A is [D, N]
        glinattn_selective_scan(x, x, _f(1, 8, 16), _f(1, 8, 16), _f(16, 32))
    with pytest.raises(TypeError):   # delta in another dtype than x
        glinattn_selective_scan(x, x.to(torch.bfloat16), _f(1, 8, 16), _f(1, 8, 16), _f(32, 16))
    with pytest.raises(ValueError):  # pool is [P, D, N]
        glinattn_selective_scan_decode(_f(2, 32), _f(2, 32), _f(2, 16), _f(2, 16), _f(32, 16), _f(4, 32, 8),
                                       torch.zeros(2, dtype=torch.int32))
