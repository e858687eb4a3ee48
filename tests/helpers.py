"""Shared helpers for the GPU parity tests.

Error metric: normwise max relative error, max|x - ref| / max|ref| over the
whole tensor (elementwise relative error is undefined near zero).  Tolerances
for bf16 inputs: outputs 2e-3, final fp32 states 1e-3; fp32 inputs: 1e-5.
"""
import os

import numpy as np
import torch

TOL_O_BF16, TOL_S_BF16, TOL_F32 = 2e-3, 1e-3, 1e-5
# oracle threads: every host core
NT = os.cpu_count() or 1


def relerr(x, ref):
    x = x.double().cpu().numpy() if isinstance(x, torch.Tensor) else np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    den = np.abs(ref).max()
    return float(np.abs(x - ref).max() / den) if den > 0 else float(np.abs(x).max())


def f64(t):
    return None if t is None else t.double().cpu().numpy()


def to(d, dev):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
