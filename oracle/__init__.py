"""Plain fp64 CPU oracle for the state-passing linear-attention layer.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The CUDA product path in
``gated_deltanet_02_gb300`` never imports this package, and this package never
imports that one; both receive the same seeded inputs from
``gated_deltanet_02_gb300.inputs``, which holds none of the method's arithmetic.

Source of every definition: "Inference for linear attention and hybrid
architectures" (ai-infra-handbooks), section "Two ways to write the same
computation" (the recurrences, the short causal convolution and its cache) and
section "Speculative decoding and PD disaggregation" (slot-indexed state pool,
one state per draft position).  The token-by-token recurrence itself lives in
``glinattn_oracle.c`` (plain C, double precision); this module builds it with
gcc on first use and composes the layer from it:

* ``recurrence``   -- the C recurrence, optionally emitting every state;
* ``expand_groups``-- grouped q / k heads (the SSD form's shared B, C) to one per head;
* ``frontend``     -- conv (width 4) -> L2 norm of q, k -> bf16 rounding;
* ``layer_prefill``-- front end + recurrence over a whole segment;
* ``decode``       -- by definition a one-token prefill from a pool slot;
* ``spec_decode``  -- D one-token steps, the state after each kept in its slot.

``oracle.chunked`` holds the second, independent fp64 path (the chunked form).

Inputs are float64 numpy arrays holding exactly the values the GPU receives
(bf16 values are exact in float64).  Outputs are float64.  The recurrences
run in double precision; the front end of bf16 activations (conv, L2 norm,
then the rounding to bf16, which decides a bf16 code) runs in single
precision in the order its definitions read, see ``frontend``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "glinattn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

GLA, GDN = 0, 1
L2_EPS = 1e-6  # front-end normalisation: x / sqrt(sum x^2 + eps)


def build(force: bool = False) -> str:
    """Compile ``glinattn_oracle.c`` into ``_build/liboracle.so`` with gcc."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        # -ffp-contract=off: a product and a sum fuse into one rounding only
        # where the source calls fmaf
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_recurrence.argtypes = [ctypes.c_int] * 6 + [dp] * 8 + [ctypes.c_int]
            lib.oracle_causal_conv.argtypes = [ctypes.c_int] * 3 + [dp] * 5
            lib.oracle_l2norm_rows.argtypes = [ctypes.c_longlong, ctypes.c_int, dp, ctypes.c_double]
            lib.oracle_round_bf16.argtypes = [ctypes.c_longlong, dp]
            lib.oracle_causal_conv_f32.argtypes = [ctypes.c_int] * 3 + [dp] * 5
            lib.oracle_l2norm_rows_f32.argtypes = [ctypes.c_longlong, ctypes.c_int, dp, ctypes.c_double]
            for f in (lib.oracle_recurrence, lib.oracle_causal_conv, lib.oracle_l2norm_rows,
                      lib.oracle_round_bf16, lib.oracle_causal_conv_f32, lib.oracle_l2norm_rows_f32):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(x):
    if x is None:
        return None
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check(rc: int, what: str):
    if rc != 0:
        msg = {-1: "bad argument", -2: "gate alpha outside (0, 1]", -3: "out of memory"}
        raise ValueError(f"oracle {what}: {msg.get(rc, rc)}")


# --------------------------------------------------------------------------
# The recurrence
# --------------------------------------------------------------------------

def expand_groups(x, heads):
    """q or k [..., Hq, d] -> [..., H, d] when groups of H / Hq consecutive heads
    share one q / k head: head h reads head h // (H / Hq).  The linear-attention
    page lists the SSD form of Mamba2 among the gated linear attention
    recurrences (section "Two ways to write the same computation"); its B and C
    (k and q here) are shared by the heads of a group, the convention of the
    Mamba2 layer on the field-notes page (section "Mamba and hybrid SSMs, the
    real packages")."""
    x = _f64(x)
    hq = x.shape[-2]
    if hq <= 0 or heads % hq:
        raise ValueError("q / k heads must divide the number of heads")
    return np.repeat(x, heads // hq, axis=-2)


def recurrence(variant, q, k, v, alpha, beta=None, S0=None, return_states=False, nthreads=1):
    """Token-by-token recurrence over q, k [B,T,H,dk] (or [B,T,Hq,dk] shared
    by groups of heads, see ``expand_groups``), v [B,T,H,dv], alpha/beta
    [B,T,H]; S0 [B,H,dk,dv] or None (zeros).

    Returns (o [B,T,H,dv], S_T [B,H,dk,dv]) and, with ``return_states``, the
    state after every token [B,T,H,dk,dv].
    """
    q, k, v, alpha = _f64(q), _f64(k), _f64(v), _f64(alpha)
    if q.ndim == 4 and v.ndim == 4 and q.shape[2] != v.shape[2]:
        q, k = expand_groups(q, v.shape[2]), expand_groups(k, v.shape[2])
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (B, T, H) or alpha.shape != (B, T, H):
        raise ValueError("shape mismatch")
    if variant == GDN:
        if beta is None:
            raise ValueError("Gated DeltaNet needs beta")
        beta = _f64(beta)
        if beta.shape != (B, T, H):
            raise ValueError("beta shape")
    else:
        beta = None
    S = np.zeros((B, H, dk, dv)) if S0 is None else _f64(S0).copy()
    if S.shape != (B, H, dk, dv):
        raise ValueError("S0 shape")
    o = np.zeros((B, T, H, dv))
    states = np.zeros((B, T, H, dk, dv)) if return_states else None
    rc = _load().oracle_recurrence(variant, B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(alpha), _ptr(beta), _ptr(S), _ptr(o), _ptr(states),
                                   int(nthreads))
    _check(rc, "recurrence")
    return (o, S, states) if return_states else (o, S)


# --------------------------------------------------------------------------
# The front end: short causal convolution, L2 norm, bf16 activations
# --------------------------------------------------------------------------

def causal_conv(x, w, cache_in=None, single=False):
    """Depthwise causal conv, width 4: x [B,T,Cch], w [Cch,4], cache [B,3,Cch].
    Returns (y [B,T,Cch], cache_out [B,3,Cch]).  ``single``: evaluated in
    single precision, taps oldest first, the first product rounded and each
    later tap added by one fused multiply-add (the values then fit a float
    exactly; see ``frontend``)."""
    x, w = _f64(x), _f64(w)
    B, T, Cch = x.shape
    if w.shape != (Cch, 4):
        raise ValueError("conv weight shape")
    cin = None if cache_in is None else _f64(cache_in)
    if cin is not None and cin.shape != (B, 3, Cch):
        raise ValueError("conv cache shape")
    y = np.zeros_like(x)
    cout = np.zeros((B, 3, Cch))
    fn = _load().oracle_causal_conv_f32 if single else _load().oracle_causal_conv
    _check(fn(B, T, Cch, _ptr(x), _ptr(w), _ptr(cin), _ptr(y), _ptr(cout)), "causal_conv")
    return y, cout


def l2norm_rows(x, eps=L2_EPS, single=False):
    """Normalise the last axis: x / sqrt(sum x^2 + eps).  ``single``: in single
    precision, the sum of squares by pairwise summation, then each element
    times 1 / sqrt(s + eps)."""
    x = _f64(x).copy()
    d = x.shape[-1]
    fn = _load().oracle_l2norm_rows_f32 if single else _load().oracle_l2norm_rows
    _check(fn(x.size // d, d, _ptr(x), eps), "l2norm")
    return x


def round_bf16(x):
    """Round to the nearest bfloat16 value (ties to even), returned as float64."""
    x = _f64(x).copy()
    _check(_load().oracle_round_bf16(x.size, _ptr(x)), "round_bf16")
    return x


def frontend(q, k, v, conv_w=None, conv_in=None, qk_l2norm=False, act_bf16=True):
    """The layer's input stage on raw q, k [B,T,H,dk], v [B,T,H,dv].

    Channels are ordered [q | k | v], each head-major (channel = part offset +
    h * d + i), so conv_w is [H*(2dk+dv), 4] and the conv cache is
    [B, 3, H*(2dk+dv)].  Steps: optional conv (with conv_in as the history, or
    zeros), then optional L2 norm of each q and k row per head, then rounding to
    bf16 when activations are bf16.  Returns (q, k, v, conv_out or None).

    With bf16 activations the rounding to bf16 decides an integer (the bf16
    code), so the steps before it are taken in the precision the layer
    computes them in, single precision, in the order the definitions read
    (``causal_conv`` / ``l2norm_rows`` with ``single``); with fp32 activations
    nothing is decided and they stay in double precision.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    conv_out = None
    changed = False
    single = bool(act_bf16)
    if conv_w is not None:
        x = np.concatenate([q.reshape(B, T, H * dk), k.reshape(B, T, H * dk),
                            v.reshape(B, T, H * dv)], axis=-1)
        y, conv_out = causal_conv(x, conv_w, conv_in, single=single)
        q = y[..., :H * dk].reshape(B, T, H, dk)
        k = y[..., H * dk:2 * H * dk].reshape(B, T, H, dk)
        v = y[..., 2 * H * dk:].reshape(B, T, H, dv)
        changed = True
    if qk_l2norm:
        q, k = l2norm_rows(q, single=single), l2norm_rows(k, single=single)
        changed = True
    if act_bf16 and changed:
        q, k, v = round_bf16(q), round_bf16(k), round_bf16(v)
    return q, k, v, conv_out


# --------------------------------------------------------------------------
# Layer-level compositions
# --------------------------------------------------------------------------

def layer_prefill(variant, q, k, v, alpha, beta=None, S0=None, conv_w=None, conv_in=None,
                  qk_l2norm=False, act_bf16=True, nthreads=1):
    """Front end, then the recurrence over the whole segment.  A segment that
    starts from (S0, conv_in) continues a previous one exactly: section "Two
    ways to write the same computation" (the state handed to the next segment).
    Returns (o, S_T, conv_out)."""
    qf, kf, vf, conv_out = frontend(q, k, v, conv_w, conv_in, qk_l2norm, act_bf16)
    o, S = recurrence(variant, qf, kf, vf, alpha, beta, S0, nthreads=nthreads)
    return o, S, conv_out


def decode(variant, q, k, v, alpha, beta, pool, slot_ids, conv_w=None, conv_pool=None,
           qk_l2norm=False, act_bf16=True):
    """One decode step for N requests: q, k [N,H,dk], v [N,H,dv], alpha/beta
    [N,H]; pool [P,H,dk,dv]; slot_ids [N]; conv_pool [P,3,Cch] or None.

    By definition a one-token prefill of each request from its slot's state
    and conv cache.  Returns (o [N,H,dv], pool', conv_pool') where the primed
    pools are updated copies (untouched slots unchanged)."""
    pool = _f64(pool).copy()
    conv_pool = None if conv_pool is None else _f64(conv_pool).copy()
    N, H = np.shape(alpha)
    dv = np.shape(v)[-1]
    o = np.zeros((N, H, dv))
    slots = [int(s) for s in slot_ids]
    if len(set(slots)) != len(slots) or any(s < 0 or s >= pool.shape[0] for s in slots):
        raise ValueError("slot ids must be distinct and inside the pool")
    for n, s in enumerate(slots):
        cin = None if conv_pool is None else conv_pool[s][None]
        on, Sn, cout = layer_prefill(
            variant, np.asarray(q[n])[None, None], np.asarray(k[n])[None, None],
            np.asarray(v[n])[None, None], np.asarray(alpha[n])[None, None],
            None if beta is None else np.asarray(beta[n])[None, None], pool[s][None],
            conv_w, cin, qk_l2norm, act_bf16)
        o[n] = on[0, 0]
        pool[s] = Sn[0]
        if conv_pool is not None:
            conv_pool[s] = cout[0]
    return o, pool, conv_pool


def spec_decode(variant, q, k, v, alpha, beta, pool, src_slot, dst_slots, conv_w=None,
                conv_pool=None, qk_l2norm=False, act_bf16=True):
    """Speculative decode of D draft tokens per request: q, k [N,D,H,dk],
    v [N,D,H,dv], alpha/beta [N,D,H]; the state (and conv cache) after draft i
    goes to slot dst_slots[n][i]; the source slot is left as it was: section
    "Speculative decoding and PD disaggregation" (one state per draft
    position).  Returns (o [N,D,H,dv], pool', conv_pool')."""
    pool = _f64(pool).copy()
    conv_pool = None if conv_pool is None else _f64(conv_pool).copy()
    N, D, H = np.shape(alpha)
    dv = np.shape(v)[-1]
    o = np.zeros((N, D, H, dv))
    for n in range(N):
        S = pool[int(src_slot[n])][None].copy()
        cache = None if conv_pool is None else conv_pool[int(src_slot[n])][None].copy()
        for i in range(D):
            on, S, cache = layer_prefill(
                variant, np.asarray(q[n, i])[None, None], np.asarray(k[n, i])[None, None],
                np.asarray(v[n, i])[None, None], np.asarray(alpha[n, i])[None, None],
                None if beta is None else np.asarray(beta[n, i])[None, None], S,
                conv_w, cache, qk_l2norm, act_bf16)
            o[n, i] = on[0, 0]
            pool[int(dst_slots[n][i])] = S[0]
            if conv_pool is not None:
                conv_pool[int(dst_slots[n][i])] = cache[0]
    return o, pool, conv_pool
