"""The C-ABI library: loads, exports every declared symbol, matches the
header's struct layout, and rejects bad arguments on the host (no launch)."""
import ctypes
import json
import os
import re
import subprocess

import pytest

from gated_deltanet_02_gb300 import glinattn as G

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "glinattn.h")


def _declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(glinattn_\w+)\s*\(", text, re.M)))


def test_library_exports_every_declared_symbol():
    lib = G.library()
    names = _declared_functions()
    assert {"glinattn_prefill", "glinattn_decode", "glinattn_spec_decode", "glinattn_state_copy",
            "glinattn_replay",
            "glinattn_status_string", "glinattn_version"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", G._build.LIB], capture_output=True,
                         text=True, check=True).stdout
    for name in names:
        assert re.search(rf"\bT {name}$", out, re.M), name


STRUCTS = ((G.PrefillArgs, "glinattn_prefill_args"), (G.DecodeArgs, "glinattn_decode_args"),
           (G.SpecArgs, "glinattn_spec_args"), (G.ReplayArgs, "glinattn_replay_args"),
           (G.CopyArgs, "glinattn_copy_args"), (G.ScanArgs, "glinattn_scan_args"),
           (G.ScanDecodeArgs, "glinattn_scan_decode_args"))


def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "glinattn.h"', "int main(void){"]
    for ct, cname in STRUCTS:
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in ct._fields_:
            lines.append(f'printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines.append("return 0;}")
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n"):
        if line:
            s, f, v = line.split()
            got[(s, f)] = int(v)
    for ct, cname in STRUCTS:
        assert got[(cname, "size")] == ctypes.sizeof(ct)
        for fname, _ in ct._fields_:
            assert got[(cname, fname)] == getattr(ct, fname).offset, (cname, fname)


def test_version_status_and_state_size():
    lib = G.library()
    assert lib.glinattn_version() >= 100
    for code in range(6):
        assert G.status_string(code) != "unknown status"
    assert G.status_string(99) == "unknown status"
    ledger = json.load(open(os.path.join(ROOT, "tests", "golden", "memory_ledger.json")))
    d = ledger["head_state_shape"][0]
    assert G.state_bytes(1, d, d) == ledger["head_state_bytes_fp32"]
    per_layer = G.state_bytes(ledger["heads_per_linear_layer"], d, d)
    assert per_layer * ledger["linear_layers"] == ledger["state_bytes_per_request"]
    # the conv cache of one layer: [q | k | v] channels of every head
    assert ledger["heads_per_linear_layer"] * 3 * d == ledger["conv_channels_per_layer"]
    assert G.state_bytes(0, 128, 128) == 0


# Fake, aligned device addresses: validation must reject before any dereference.
A = 0x10000


def _prefill(**kw):
    base = dict(variant=G.GDN, in_dtype=G.BF16, out_dtype=G.F32, qk_l2norm=1, batch=2, seqlen=100,
                heads=4, dk=128, dv=128, q=A, k=A * 2, v=A * 3, alpha=A * 4, beta=A * 5, S0=None,
                S_T=A * 6, o=A * 7)
    base.update(kw)
    return G.PrefillArgs(**base)


def _decode(**kw):
    base = dict(variant=G.GDN, in_dtype=G.BF16, out_dtype=G.F32, num_req=4, heads=2, dk=64, dv=64,
                pool_slots=8, q=A, k=A * 2, v=A * 3, alpha=A * 4, beta=A * 5, state_pool=A * 6,
                slot_ids=A * 7, o=A * 8)
    base.update(kw)
    return G.DecodeArgs(**base)


def _spec(**kw):
    base = dict(variant=G.GDN, in_dtype=G.BF16, out_dtype=G.F32, num_req=4, draft_len=3, heads=2,
                dk=64, dv=64, pool_slots=32, q=A, k=A * 2, v=A * 3, alpha=A * 4, beta=A * 5,
                state_pool=A * 6, src_slots=A * 7, dst_slots=A * 8, o=A * 9)
    base.update(kw)
    return G.SpecArgs(**base)


INVALID, UNSUPPORTED = 1, 2


@pytest.mark.parametrize("kw,code", [
    (dict(variant=7), INVALID),
    (dict(in_dtype=5), INVALID),
    (dict(out_dtype=-1), INVALID),
    (dict(dk=96, dv=96), UNSUPPORTED),
    (dict(dk=128, dv=32), UNSUPPORTED),
    (dict(dk=64, dv=128), UNSUPPORTED),
    (dict(qk_heads=3), INVALID),         # does not divide heads = 4
    (dict(qk_heads=-1), INVALID),
    (dict(qk_heads=2, conv_w=A * 9), UNSUPPORTED),  # grouped heads take no convolution
    (dict(variant=3), INVALID),
    (dict(variant=G.NLA, qk_l2norm=0, z_T=None), INVALID),   # the normaliser must go somewhere
    (dict(variant=G.NLA, qk_l2norm=0, z_T=A * 10, conv_w=A * 9), UNSUPPORTED),
    (dict(variant=G.NLA, qk_l2norm=0, z_T=A * 10, state_every=64, S_blocks=A * 11), UNSUPPORTED),
    (dict(variant=G.NLA, qk_l2norm=0, z_T=A * 10 + 4), INVALID),
    (dict(heads=0), INVALID),
    (dict(batch=-1), INVALID),
    (dict(seqlen=-5), INVALID),
    (dict(q=None), INVALID),
    (dict(beta=None), INVALID),          # Gated DeltaNet needs beta
    (dict(S_T=None), INVALID),
    (dict(o=None), INVALID),
    (dict(q=A + 8), INVALID),            # 16-byte alignment
    (dict(S0=A * 6 + 64), INVALID),      # S0 partially overlaps S_T
    (dict(state_every=-1), INVALID),
    (dict(state_every=50), INVALID),     # two blocks to emit but no S_blocks
    (dict(state_every=50, S_blocks=A * 9 + 4), INVALID),
    (dict(state_every=50, S_blocks=A * 9), UNSUPPORTED),  # chunked kernels: multiples of 64 only
])
def test_prefill_rejects(kw, code):
    rc = G.library().glinattn_prefill(ctypes.byref(_prefill(**kw)), None)
    assert rc == code


def test_prefill_null_args_and_empty_batch():
    lib = G.library()
    assert lib.glinattn_prefill(None, None) == INVALID
    # B = 0 is a no-op that launches nothing, even with null tensors
    assert lib.glinattn_prefill(ctypes.byref(_prefill(batch=0, q=None, o=None)), None) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(pool_slots=0), INVALID),
    (dict(slot_ids=None), INVALID),
    (dict(state_pool=None), INVALID),
    (dict(state_pool=A * 6 + 4), INVALID),
    (dict(dk=48, dv=48), UNSUPPORTED),
    (dict(conv_w=A * 9, conv_pool=None), INVALID),
    (dict(num_req=-1), INVALID),
    (dict(qk_heads=3), INVALID),
    (dict(qk_heads=1, conv_w=A * 9, conv_pool=A * 10), UNSUPPORTED),
    (dict(variant=G.NLA, qk_l2norm=0), INVALID),              # no normaliser pool
    (dict(variant=G.NLA, z_pool=A * 11, conv_w=A * 9, conv_pool=A * 10), UNSUPPORTED),
])
def test_decode_rejects(kw, code):
    assert G.library().glinattn_decode(ctypes.byref(_decode(**kw)), None) == code


@pytest.mark.parametrize("kw,code", [
    (dict(draft_len=0), INVALID),
    (dict(o=None), INVALID),             # dst_slots may be NULL (verify only), o may not
    (dict(src_slots=None), INVALID),
    (dict(variant=G.GDN, beta=None), INVALID),
])
def test_spec_rejects(kw, code):
    assert G.library().glinattn_spec_decode(ctypes.byref(_spec(**kw)), None) == code


def test_zero_requests_is_a_noop():
    lib = G.library()
    assert lib.glinattn_decode(ctypes.byref(_decode(num_req=0, q=None)), None) == 0
    assert lib.glinattn_spec_decode(ctypes.byref(_spec(num_req=0, q=None)), None) == 0


def _copy(**kw):
    base = dict(n=3, pool_slots=8, heads=2, dk=64, dv=64, in_dtype=G.BF16, state_pool=A,
                conv_pool=A * 2, src_slots=A * 3, dst_slots=A * 4)
    base.update(kw)
    return G.CopyArgs(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(n=-1), INVALID),
    (dict(pool_slots=0), INVALID),
    (dict(heads=0), INVALID),
    (dict(in_dtype=5), INVALID),
    (dict(state_pool=None), INVALID),
    (dict(src_slots=None), INVALID),
    (dict(dst_slots=None), INVALID),
    (dict(state_pool=A + 4), INVALID),
    (dict(conv_pool=A * 2 + 8), INVALID),
    (dict(n=70000), UNSUPPORTED),
    (dict(dk=3, dv=3, conv_pool=None), UNSUPPORTED),  # a slot of 18 floats: not whole 16-byte words
])
def test_state_copy_rejects(kw, code):
    assert G.library().glinattn_state_copy(ctypes.byref(_copy(**kw)), None) == code


def test_state_copy_zero_pairs_is_a_noop():
    lib = G.library()
    assert lib.glinattn_state_copy(None, None) == INVALID
    assert lib.glinattn_state_copy(ctypes.byref(_copy(n=0, state_pool=None)), None) == 0


def _replay(**kw):
    base = dict(variant=G.GDN, in_dtype=G.BF16, qk_l2norm=1, num_req=4, draft_len=3, heads=2, dk=64, dv=64,
                pool_slots=8, q=A, k=A * 2, v=A * 3, alpha=A * 4, beta=A * 5, state_pool=A * 6,
                slot_ids=A * 7, accept=A * 8)
    base.update(kw)
    return G.ReplayArgs(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(accept=None), INVALID),
    (dict(slot_ids=None), INVALID),
    (dict(state_pool=None), INVALID),
    (dict(draft_len=0), INVALID),
    (dict(pool_slots=0), INVALID),
    (dict(variant=G.GDN, beta=None), INVALID),
    (dict(conv_w=A * 9, conv_pool=None), INVALID),
    (dict(dk=48, dv=48), UNSUPPORTED),
    (dict(k=A * 2 + 2), INVALID),
])
def test_replay_rejects(kw, code):
    assert G.library().glinattn_replay(ctypes.byref(_replay(**kw)), None) == code


def test_replay_zero_requests_is_a_noop():
    lib = G.library()
    assert lib.glinattn_replay(None, None) == INVALID
    assert lib.glinattn_replay(ctypes.byref(_replay(num_req=0, k=None)), None) == 0


def _scan(**kw):
    base = dict(in_dtype=G.F32, out_dtype=G.F32, batch=2, seqlen=100, channels=64, state=16, x=A, delta=A * 2,
                Bm=A * 3, Cm=A * 4, A=A * 5, h0=None, h_T=A * 6, y=A * 7)
    base.update(kw)
    return G.ScanArgs(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(in_dtype=5), INVALID),
    (dict(state=12), UNSUPPORTED),
    (dict(state=64), UNSUPPORTED),
    (dict(channels=0), INVALID),
    (dict(A=None), INVALID),
    (dict(h_T=None), INVALID),
    (dict(x=None), INVALID),
    (dict(h_T=A * 6 + 4), INVALID),
    (dict(h0=A * 6 + 64), INVALID),      # partial overlap with h_T
    (dict(), INVALID),                   # no workspace for a non-empty segment
])
def test_selective_scan_rejects(kw, code):
    assert G.library().glinattn_selective_scan(ctypes.byref(_scan(**kw)), None) == code


def test_selective_scan_workspace_and_empty_batch():
    lib = G.library()
    a = _scan(batch=2, seqlen=130, channels=64, state=16)
    nc = 3  # chunks of 64
    assert lib.glinattn_selective_scan_workspace_size(ctypes.byref(a)) >= 2 * 2 * nc * 64 * 16 * 4
    assert lib.glinattn_selective_scan(ctypes.byref(_scan(batch=0, x=None)), None) == 0
    assert lib.glinattn_selective_scan(None, None) == INVALID


def _scan_dec(**kw):
    base = dict(in_dtype=G.BF16, out_dtype=G.F32, num_req=4, channels=64, state=16, pool_slots=8, x=A,
                delta=A * 2, Bm=A * 3, Cm=A * 4, A=A * 5, state_pool=A * 6, slot_ids=A * 7, y=A * 8)
    base.update(kw)
    return G.ScanDecodeArgs(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(slot_ids=None), INVALID),
    (dict(state_pool=A * 6 + 8), INVALID),
    (dict(pool_slots=0), INVALID),
    (dict(state=4), UNSUPPORTED),
    (dict(num_req=70000), UNSUPPORTED),
])
def test_selective_scan_decode_rejects(kw, code):
    assert G.library().glinattn_selective_scan_decode(ctypes.byref(_scan_dec(**kw)), None) == code
