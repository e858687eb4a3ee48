"""Thin Python binding of the glinattn C ABI (``include/glinattn.h``).

Argument marshalling only: every step of the layer runs in the CUDA kernels of
``libglinattn.so``.  PyTorch supplies device memory and streams.  There is no
CPU fallback: if the library cannot be built or loaded, every call raises.

The entry points keep the C names:

* ``glinattn_prefill``     -- chunked prefill of a segment (state hand-over in/out)
* ``glinattn_decode``      -- one recurrent step per request, state pool by slot id
* ``glinattn_spec_decode`` -- D draft steps, one state per draft position
* ``glinattn_replay``      -- apply the accepted drafts to the pool in place
* ``glinattn_state_copy``  -- whole-slot copies inside a state pool (copy on write)
* ``glinattn_selective_scan`` / ``glinattn_selective_scan_decode`` -- Mamba's
  selective scan (chunked prefill; one step from a slot-indexed pool)
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import build as _build

GLA, GDN, NLA = 0, 1, 2
F32, BF16 = 0, 1

DEV_BAD_SLOT = 0x1
DEV_BAD_GATE = 0x2
DEV_WAIT_TIMEOUT = 0x4
DEV_BAD_COUNT = 0x8

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration", 3: "CUDA error",
           4: "device reported an error status", 5: "device wait timed out"}


class GlinattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {_STATUS.get(status, status)} (status {status})")
        self.status = status


_vp = ctypes.c_void_p
_i32 = ctypes.c_int32


class PrefillArgs(ctypes.Structure):
    _fields_ = [("variant", _i32), ("in_dtype", _i32), ("out_dtype", _i32), ("qk_l2norm", _i32),
                ("batch", _i32), ("seqlen", _i32), ("heads", _i32), ("dk", _i32), ("dv", _i32),
                ("state_every", _i32),
                ("q", _vp), ("k", _vp), ("v", _vp), ("alpha", _vp), ("beta", _vp), ("S0", _vp),
                ("S_T", _vp), ("o", _vp), ("conv_w", _vp), ("conv_in", _vp), ("conv_out", _vp),
                ("dev_status", _vp), ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
                ("S_blocks", _vp), ("conv_blocks", _vp), ("qk_heads", _i32), ("z0", _vp), ("z_T", _vp)]


class DecodeArgs(ctypes.Structure):
    _fields_ = [("variant", _i32), ("in_dtype", _i32), ("out_dtype", _i32), ("qk_l2norm", _i32),
                ("num_req", _i32), ("heads", _i32), ("dk", _i32), ("dv", _i32),
                ("pool_slots", _i32), ("qk_heads", _i32),
                ("q", _vp), ("k", _vp), ("v", _vp), ("alpha", _vp), ("beta", _vp),
                ("state_pool", _vp), ("slot_ids", _vp), ("o", _vp), ("conv_w", _vp),
                ("conv_pool", _vp), ("dev_status", _vp), ("z_pool", _vp)]


class SpecArgs(ctypes.Structure):
    _fields_ = [("variant", _i32), ("in_dtype", _i32), ("out_dtype", _i32), ("qk_l2norm", _i32),
                ("num_req", _i32), ("draft_len", _i32), ("heads", _i32), ("dk", _i32),
                ("dv", _i32), ("pool_slots", _i32),
                ("q", _vp), ("k", _vp), ("v", _vp), ("alpha", _vp), ("beta", _vp),
                ("state_pool", _vp), ("src_slots", _vp), ("dst_slots", _vp), ("o", _vp),
                ("conv_w", _vp), ("conv_pool", _vp), ("dev_status", _vp), ("qk_heads", _i32),
                ("z_pool", _vp)]


class ReplayArgs(ctypes.Structure):
    _fields_ = [("variant", _i32), ("in_dtype", _i32), ("qk_l2norm", _i32), ("num_req", _i32),
                ("draft_len", _i32), ("heads", _i32), ("dk", _i32), ("dv", _i32), ("pool_slots", _i32),
                ("qk_heads", _i32),
                ("q", _vp), ("k", _vp), ("v", _vp), ("alpha", _vp), ("beta", _vp),
                ("state_pool", _vp), ("slot_ids", _vp), ("accept", _vp), ("conv_w", _vp),
                ("conv_pool", _vp), ("dev_status", _vp), ("z_pool", _vp)]


class ScanArgs(ctypes.Structure):
    _fields_ = [("in_dtype", _i32), ("out_dtype", _i32), ("batch", _i32), ("seqlen", _i32),
                ("channels", _i32), ("state", _i32), ("x", _vp), ("delta", _vp), ("Bm", _vp), ("Cm", _vp),
                ("A", _vp), ("h0", _vp), ("h_T", _vp), ("y", _vp), ("workspace", _vp),
                ("workspace_bytes", ctypes.c_size_t), ("dev_status", _vp)]


class ScanDecodeArgs(ctypes.Structure):
    _fields_ = [("in_dtype", _i32), ("out_dtype", _i32), ("num_req", _i32), ("channels", _i32),
                ("state", _i32), ("pool_slots", _i32), ("x", _vp), ("delta", _vp), ("Bm", _vp), ("Cm", _vp),
                ("A", _vp), ("state_pool", _vp), ("slot_ids", _vp), ("y", _vp), ("dev_status", _vp)]


class CopyArgs(ctypes.Structure):
    _fields_ = [("n", _i32), ("pool_slots", _i32), ("heads", _i32), ("dk", _i32), ("dv", _i32),
                ("in_dtype", _i32), ("state_pool", _vp), ("conv_pool", _vp), ("src_slots", _vp),
                ("dst_slots", _vp), ("dev_status", _vp)]


_lock = threading.Lock()
_lib = None


def library() -> ctypes.CDLL:
    """Load ``libglinattn.so`` (building it first when its sources are newer)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            lib = ctypes.CDLL(path)
            for name, argt in (("glinattn_prefill", PrefillArgs), ("glinattn_decode", DecodeArgs),
                               ("glinattn_spec_decode", SpecArgs), ("glinattn_replay", ReplayArgs),
                               ("glinattn_state_copy", CopyArgs), ("glinattn_selective_scan", ScanArgs),
                               ("glinattn_selective_scan_decode", ScanDecodeArgs)):
                f = getattr(lib, name)
                f.argtypes = [ctypes.POINTER(argt), _vp]
                f.restype = ctypes.c_int
            lib.glinattn_status_string.argtypes = [ctypes.c_int]
            lib.glinattn_status_string.restype = ctypes.c_char_p
            lib.glinattn_version.restype = ctypes.c_int
            lib.glinattn_state_bytes.argtypes = [ctypes.c_int] * 3
            lib.glinattn_state_bytes.restype = ctypes.c_size_t
            lib.glinattn_prefill_workspace_size.argtypes = [ctypes.POINTER(PrefillArgs)]
            lib.glinattn_prefill_workspace_size.restype = ctypes.c_size_t
            lib.glinattn_selective_scan_workspace_size.argtypes = [ctypes.POINTER(ScanArgs)]
            lib.glinattn_selective_scan_workspace_size.restype = ctypes.c_size_t
            _lib = lib
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"activations must be bf16 or fp32, got {t.dtype}")


def _need(t, name, dtype=None, shape=None, device=None):
    if t is None:
        return
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _call(name, args, stream_handle):
    rc = getattr(library(), name)(ctypes.byref(args), stream_handle)
    if rc != 0:
        raise GlinattnError(rc, name)


def glinattn_prefill(q, k, v, alpha, beta=None, S0=None, *, variant=GLA, conv_w=None,
                     conv_in=None, qk_l2norm=False, out_dtype=None, o=None, S_T=None,
                     conv_out=None, dev_status=None, stream=None, workspace=None,
                     state_every=0, S_blocks=None, conv_blocks=None, z0=None, z_T=None):
    """Prefill one segment.  q, k [B,T,Hq,dk], v [B,T,H,dv] (bf16 or fp32;
    Hq < H shares q, k across groups of H // Hq heads);
    alpha/beta [B,T,H] fp32; S0 [B,H,dk,dv] fp32 or None.  Outputs, and the
    scratch space the chunked Gated DeltaNet kernels need, are allocated when
    not given.  Returns (o, S_T, conv_out); with state_every > 0 also
    S_blocks [B, T // state_every, H, dk, dv], the state after every
    state_every tokens of the segment, and conv_blocks [B, T // state_every,
    3, Cch], the conv cache at the same points (None without a conv).
    variant=NLA (normalised linear attention: no gates, alpha may be None)
    returns (o, S_T, None, z_T), the normaliser z [B,H,dk] beside the state."""
    B, T, Hq, dk = q.shape
    H, dv = v.shape[2], v.shape[3]
    dev = q.device
    act = q.dtype
    _need(q, "q", act, (B, T, Hq, dk), dev)
    _need(k, "k", act, (B, T, Hq, dk), dev)
    _need(v, "v", act, (B, T, H, dv), dev)
    _need(alpha, "alpha", torch.float32, (B, T, H), dev)
    _need(beta, "beta", torch.float32, (B, T, H), dev)
    _need(S0, "S0", torch.float32, (B, H, dk, dv), dev)
    out_dtype = act if out_dtype is None else out_dtype
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=out_dtype, device=dev)
    if S_T is None:
        S_T = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    Cch = H * (2 * dk + dv)
    if conv_w is not None:
        _need(conv_w, "conv_w", torch.float32, (Cch, 4), dev)
        _need(conv_in, "conv_in", act, (B, 3, Cch), dev)
        if conv_out is None:
            conv_out = torch.empty((B, 3, Cch), dtype=act, device=dev)
        _need(conv_out, "conv_out", act, (B, 3, Cch), dev)
    _need(o, "o", out_dtype, (B, T, H, dv), dev)
    _need(S_T, "S_T", torch.float32, (B, H, dk, dv), dev)
    nla = variant == NLA
    if nla:
        _need(z0, "z0", torch.float32, (B, H, dk), dev)
        if z_T is None:
            z_T = torch.empty((B, H, dk), dtype=torch.float32, device=dev)
        _need(z_T, "z_T", torch.float32, (B, H, dk), dev)
    if state_every < 0:
        raise ValueError("state_every must be >= 0")
    nblk = T // state_every if state_every else 0
    if state_every and S_blocks is None:
        S_blocks = torch.empty((B, nblk, H, dk, dv), dtype=torch.float32, device=dev)
    if state_every:
        _need(S_blocks, "S_blocks", torch.float32, (B, nblk, H, dk, dv), dev)
        if conv_w is not None:
            if conv_blocks is None:
                conv_blocks = torch.empty((B, nblk, 3, Cch), dtype=act, device=dev)
            _need(conv_blocks, "conv_blocks", act, (B, nblk, 3, Cch), dev)
        else:
            conv_blocks = None
    a = PrefillArgs(variant=variant, in_dtype=_dtype_code(q), out_dtype=_dtype_code(o),
                    qk_l2norm=int(bool(qk_l2norm)), batch=B, seqlen=T, heads=H, dk=dk, dv=dv,
                    q=_ptr(q), k=_ptr(k), v=_ptr(v), alpha=_ptr(alpha), beta=_ptr(beta),
                    S0=_ptr(S0), S_T=_ptr(S_T), o=_ptr(o), conv_w=_ptr(conv_w),
                    conv_in=_ptr(conv_in), conv_out=_ptr(conv_out), dev_status=_ptr(dev_status),
                    state_every=state_every, S_blocks=_ptr(S_blocks) if nblk else None,
                    conv_blocks=_ptr(conv_blocks) if nblk else None, qk_heads=Hq,
                    z0=_ptr(z0) if nla else None, z_T=_ptr(z_T) if nla else None)
    ws_bytes = library().glinattn_prefill_workspace_size(ctypes.byref(a))
    ws = None
    if ws_bytes:
        if workspace is not None and workspace.numel() * workspace.element_size() >= ws_bytes:
            ws = workspace
        else:
            ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        a.workspace = _ptr(ws)
        a.workspace_bytes = ws_bytes
    _call("glinattn_prefill", a, _stream_handle(stream, dev))
    if nla:
        return o, S_T, None, z_T
    if state_every:
        return o, S_T, conv_out, S_blocks, conv_blocks
    return o, S_T, conv_out


def glinattn_decode(q, k, v, alpha, beta, state_pool, slot_ids, *, variant=GDN, conv_w=None,
                    conv_pool=None, qk_l2norm=False, out_dtype=None, o=None, dev_status=None,
                    stream=None, z_pool=None):
    """One decode step.  q, k [N,Hq,dk], v [N,H,dv]; alpha/beta [N,H];
    state_pool [P,H,dk,dv] fp32 and conv_pool [P,3,Cch] updated in place at
    slot_ids [N] int32.  Returns o [N,H,dv]."""
    N, Hq, dk = q.shape
    H, dv = v.shape[1], v.shape[2]
    dev = q.device
    act = q.dtype
    P = state_pool.shape[0]
    _need(q, "q", act, (N, Hq, dk), dev)
    _need(k, "k", act, (N, Hq, dk), dev)
    _need(v, "v", act, (N, H, dv), dev)
    _need(alpha, "alpha", torch.float32, (N, H), dev)
    _need(beta, "beta", torch.float32, (N, H), dev)
    _need(state_pool, "state_pool", torch.float32, (P, H, dk, dv), dev)
    _need(z_pool, "z_pool", torch.float32, (P, H, dk), dev)
    _need(slot_ids, "slot_ids", torch.int32, (N,), dev)
    Cch = H * (2 * dk + dv)
    if conv_w is not None:
        _need(conv_w, "conv_w", torch.float32, (Cch, 4), dev)
        _need(conv_pool, "conv_pool", act, (P, 3, Cch), dev)
    out_dtype = act if out_dtype is None else out_dtype
    if o is None:
        o = torch.empty((N, H, dv), dtype=out_dtype, device=dev)
    _need(o, "o", out_dtype, (N, H, dv), dev)
    a = DecodeArgs(variant=variant, in_dtype=_dtype_code(q), out_dtype=_dtype_code(o),
                   qk_l2norm=int(bool(qk_l2norm)), num_req=N, heads=H, dk=dk, dv=dv,
                   pool_slots=P, qk_heads=Hq, q=_ptr(q), k=_ptr(k), v=_ptr(v), alpha=_ptr(alpha),
                   beta=_ptr(beta), state_pool=_ptr(state_pool), slot_ids=_ptr(slot_ids),
                   o=_ptr(o), conv_w=_ptr(conv_w), conv_pool=_ptr(conv_pool) if conv_w is not None else None,
                   dev_status=_ptr(dev_status), z_pool=_ptr(z_pool))
    _call("glinattn_decode", a, _stream_handle(stream, dev))
    return o


def glinattn_spec_decode(q, k, v, alpha, beta, state_pool, src_slots, dst_slots, *, variant=GDN,
                         conv_w=None, conv_pool=None, qk_l2norm=False, out_dtype=None, o=None,
                         dev_status=None, stream=None, z_pool=None):
    """D draft steps per request.  q, k [N,D,Hq,dk], v [N,D,H,dv];
    alpha/beta [N,D,H]; src_slots [N], dst_slots [N,D] int32.  The state after
    draft i is written to state_pool[dst_slots[n, i]]; dst_slots=None only
    verifies (outputs, no state written: see glinattn_replay; at d = 128 the
    gated forms compute them in the chunked form over the drafts, equal to the
    per-draft outputs up to fp32 rounding).  Returns
    o [N,D,H,dv]."""
    N, D, Hq, dk = q.shape
    H, dv = v.shape[2], v.shape[3]
    dev = q.device
    act = q.dtype
    P = state_pool.shape[0]
    _need(q, "q", act, (N, D, Hq, dk), dev)
    _need(k, "k", act, (N, D, Hq, dk), dev)
    _need(v, "v", act, (N, D, H, dv), dev)
    _need(alpha, "alpha", torch.float32, (N, D, H), dev)
    _need(beta, "beta", torch.float32, (N, D, H), dev)
    _need(state_pool, "state_pool", torch.float32, (P, H, dk, dv), dev)
    _need(z_pool, "z_pool", torch.float32, (P, H, dk), dev)
    _need(src_slots, "src_slots", torch.int32, (N,), dev)
    _need(dst_slots, "dst_slots", torch.int32, (N, D), dev)
    Cch = H * (2 * dk + dv)
    if conv_w is not None:
        _need(conv_w, "conv_w", torch.float32, (Cch, 4), dev)
        _need(conv_pool, "conv_pool", act, (P, 3, Cch), dev)
    out_dtype = act if out_dtype is None else out_dtype
    if o is None:
        o = torch.empty((N, D, H, dv), dtype=out_dtype, device=dev)
    _need(o, "o", out_dtype, (N, D, H, dv), dev)
    a = SpecArgs(variant=variant, in_dtype=_dtype_code(q), out_dtype=_dtype_code(o),
                 qk_l2norm=int(bool(qk_l2norm)), num_req=N, draft_len=D, heads=H, dk=dk, dv=dv,
                 pool_slots=P, qk_heads=Hq, q=_ptr(q), k=_ptr(k), v=_ptr(v), alpha=_ptr(alpha),
                 beta=_ptr(beta), state_pool=_ptr(state_pool), src_slots=_ptr(src_slots),
                 dst_slots=_ptr(dst_slots),
                 o=_ptr(o), conv_w=_ptr(conv_w), conv_pool=_ptr(conv_pool) if conv_w is not None else None,
                 dev_status=_ptr(dev_status), z_pool=_ptr(z_pool))
    _call("glinattn_spec_decode", a, _stream_handle(stream, dev))
    return o


def glinattn_replay(k, v, alpha, beta, state_pool, slot_ids, accept, *, q=None, variant=GDN,
                    conv_w=None, conv_pool=None, qk_l2norm=False, dev_status=None, stream=None,
                    z_pool=None):
    """Apply the first accept[n] recorded draft steps to state_pool[slot_ids[n]]
    (and its conv cache) in place.  k [N,D,Hq,dk], v [N,D,H,dv], alpha/beta
    [N,D,H], q [N,D,Hq,dk] (its raw values enter the conv cache; defaults to k
    when there is no conv); slot_ids, accept [N] int32."""
    N, D, Hq, dk = k.shape
    H, dv = v.shape[2], v.shape[3]
    dev = k.device
    act = k.dtype
    P = state_pool.shape[0]
    if q is None:
        if conv_w is not None:
            raise ValueError("q is needed with a conv: its raw values enter the conv cache")
        q = k
    _need(q, "q", act, (N, D, Hq, dk), dev)
    _need(k, "k", act, (N, D, Hq, dk), dev)
    _need(v, "v", act, (N, D, H, dv), dev)
    _need(alpha, "alpha", torch.float32, (N, D, H), dev)
    _need(beta, "beta", torch.float32, (N, D, H), dev)
    _need(state_pool, "state_pool", torch.float32, (P, H, dk, dv), dev)
    _need(z_pool, "z_pool", torch.float32, (P, H, dk), dev)
    _need(slot_ids, "slot_ids", torch.int32, (N,), dev)
    _need(accept, "accept", torch.int32, (N,), dev)
    Cch = H * (2 * dk + dv)
    if conv_w is not None:
        _need(conv_w, "conv_w", torch.float32, (Cch, 4), dev)
        _need(conv_pool, "conv_pool", act, (P, 3, Cch), dev)
    a = ReplayArgs(variant=variant, in_dtype=_dtype_code(k), qk_l2norm=int(bool(qk_l2norm)), num_req=N,
                   draft_len=D, heads=H, dk=dk, dv=dv, pool_slots=P, qk_heads=Hq, q=_ptr(q), k=_ptr(k),
                   v=_ptr(v),
                   alpha=_ptr(alpha), beta=_ptr(beta), state_pool=_ptr(state_pool), slot_ids=_ptr(slot_ids),
                   accept=_ptr(accept), conv_w=_ptr(conv_w),
                   conv_pool=_ptr(conv_pool) if conv_w is not None else None, dev_status=_ptr(dev_status),
                   z_pool=_ptr(z_pool))
    _call("glinattn_replay", a, _stream_handle(stream, dev))
    return state_pool


def glinattn_state_copy(state_pool, src_slots, dst_slots, *, conv_pool=None, dev_status=None,
                        stream=None):
    """state_pool[dst_slots[i]] = state_pool[src_slots[i]] (and the same for
    conv_pool [P,3,Cch] when given), in place.  state_pool [P,H,dk,dv] fp32;
    src_slots, dst_slots [n] int32.  Destination slots must be distinct and
    must not be a source of another pair of the same call."""
    P, H, dk, dv = state_pool.shape
    dev = state_pool.device
    n = src_slots.shape[0]
    _need(state_pool, "state_pool", torch.float32, (P, H, dk, dv), dev)
    _need(src_slots, "src_slots", torch.int32, (n,), dev)
    _need(dst_slots, "dst_slots", torch.int32, (n,), dev)
    in_dtype = BF16
    if conv_pool is not None:
        _need(conv_pool, "conv_pool", conv_pool.dtype, (P, 3, H * (2 * dk + dv)), dev)
        in_dtype = _dtype_code(conv_pool)
    a = CopyArgs(n=n, pool_slots=P, heads=H, dk=dk, dv=dv, in_dtype=in_dtype,
                 state_pool=_ptr(state_pool), conv_pool=_ptr(conv_pool), src_slots=_ptr(src_slots),
                 dst_slots=_ptr(dst_slots), dev_status=_ptr(dev_status))
    _call("glinattn_state_copy", a, _stream_handle(stream, dev))
    return state_pool


def glinattn_selective_scan(x, delta, Bm, Cm, A, h0=None, *, out_dtype=None, y=None, h_T=None,
                            workspace=None, dev_status=None, stream=None):
    """Mamba's selective scan over a segment.  x, delta [B,T,D], Bm, Cm
    [B,T,N] (bf16 or fp32); A [D,N] fp32; h0 [B,D,N] fp32 or None.  Returns
    (y [B,T,D], h_T [B,D,N])."""
    B, T, D = x.shape
    N = Bm.shape[-1]
    dev = x.device
    act = x.dtype
    _need(x, "x", act, (B, T, D), dev)
    _need(delta, "delta", act, (B, T, D), dev)
    _need(Bm, "Bm", act, (B, T, N), dev)
    _need(Cm, "Cm", act, (B, T, N), dev)
    _need(A, "A", torch.float32, (D, N), dev)
    _need(h0, "h0", torch.float32, (B, D, N), dev)
    out_dtype = act if out_dtype is None else out_dtype
    if y is None:
        y = torch.empty((B, T, D), dtype=out_dtype, device=dev)
    if h_T is None:
        h_T = torch.empty((B, D, N), dtype=torch.float32, device=dev)
    _need(y, "y", out_dtype, (B, T, D), dev)
    _need(h_T, "h_T", torch.float32, (B, D, N), dev)
    a = ScanArgs(in_dtype=_dtype_code(x), out_dtype=_dtype_code(y), batch=B, seqlen=T, channels=D, state=N,
                 x=_ptr(x), delta=_ptr(delta), Bm=_ptr(Bm), Cm=_ptr(Cm), A=_ptr(A), h0=_ptr(h0), h_T=_ptr(h_T),
                 y=_ptr(y), dev_status=_ptr(dev_status))
    need = library().glinattn_selective_scan_workspace_size(ctypes.byref(a))
    if need:
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        a.workspace = _ptr(workspace)
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    _call("glinattn_selective_scan", a, _stream_handle(stream, dev))
    return y, h_T


def glinattn_selective_scan_decode(x, delta, Bm, Cm, A, state_pool, slot_ids, *, out_dtype=None, y=None,
                                   dev_status=None, stream=None):
    """One selective-scan step for R requests: x, delta [R,D], Bm, Cm [R,N];
    state_pool [P,D,N] fp32 updated in place at slot_ids [R] int32.  Returns y [R,D]."""
    R, D = x.shape
    N = Bm.shape[-1]
    P = state_pool.shape[0]
    dev = x.device
    act = x.dtype
    _need(x, "x", act, (R, D), dev)
    _need(delta, "delta", act, (R, D), dev)
    _need(Bm, "Bm", act, (R, N), dev)
    _need(Cm, "Cm", act, (R, N), dev)
    _need(A, "A", torch.float32, (D, N), dev)
    _need(state_pool, "state_pool", torch.float32, (P, D, N), dev)
    _need(slot_ids, "slot_ids", torch.int32, (R,), dev)
    out_dtype = act if out_dtype is None else out_dtype
    if y is None:
        y = torch.empty((R, D), dtype=out_dtype, device=dev)
    _need(y, "y", out_dtype, (R, D), dev)
    a = ScanDecodeArgs(in_dtype=_dtype_code(x), out_dtype=_dtype_code(y), num_req=R, channels=D, state=N,
                       pool_slots=P, x=_ptr(x), delta=_ptr(delta), Bm=_ptr(Bm), Cm=_ptr(Cm), A=_ptr(A),
                       state_pool=_ptr(state_pool), slot_ids=_ptr(slot_ids), y=_ptr(y),
                       dev_status=_ptr(dev_status))
    _call("glinattn_selective_scan_decode", a, _stream_handle(stream, dev))
    return y


def version() -> int:
    return library().glinattn_version()


def status_string(code: int) -> str:
    return library().glinattn_status_string(code).decode()


def state_bytes(heads: int, dk: int, dv: int) -> int:
    return library().glinattn_state_bytes(heads, dk, dv)


def prefill_workspace_size(batch, seqlen, heads, d, variant=GDN, in_dtype=BF16, out_dtype=F32) -> int:
    a = PrefillArgs(variant=variant, in_dtype=in_dtype, out_dtype=out_dtype, batch=batch,
                    seqlen=seqlen, heads=heads, dk=d, dv=d)
    return library().glinattn_prefill_workspace_size(ctypes.byref(a))
