"""GB300-native (sm_103a) state-passing linear-attention layer.

Gated linear attention (including the SSD form of Mamba2: a 128 x 64 state,
q / k shared by groups of heads), Gated DeltaNet and normalised kernelised
linear attention: chunked tensor-core prefill with optional prefix-cache
checkpoints, recurrent decode from a slot-indexed state pool, speculative
decode with one state per draft position or a verify-only round plus replay,
slot copies; and Mamba's selective scan.  All of it sits behind the C ABI
declared in ``include/glinattn.h``; ``glinattn`` is the Python binding and
``inputs`` holds the seeded synthetic input generators.
"""
from .glinattn import (BF16, F32, GDN, GLA, NLA, GlinattnError, glinattn_decode, glinattn_prefill,
                       glinattn_replay, glinattn_selective_scan, glinattn_selective_scan_decode,
                       glinattn_spec_decode, glinattn_state_copy, library, state_bytes, status_string, version)

__all__ = ["GLA", "GDN", "NLA", "F32", "BF16", "GlinattnError", "glinattn_prefill", "glinattn_decode",
           "glinattn_spec_decode", "glinattn_replay", "glinattn_state_copy", "glinattn_selective_scan",
           "glinattn_selective_scan_decode", "library", "version", "status_string", "state_bytes"]
