"""GB300-native (sm_103a) state-passing linear-attention layer.

Gated linear attention and Gated DeltaNet: chunked tensor-core prefill,
recurrent decode and speculative decode with one state per draft position,
behind the C ABI declared in ``include/glinattn.h``.  ``glinattn`` is the
Python binding; ``inputs`` holds the seeded synthetic input generators.
"""
from .glinattn import (BF16, F32, GDN, GLA, NLA, GlinattnError, glinattn_decode, glinattn_prefill,
                       glinattn_replay, glinattn_selective_scan, glinattn_selective_scan_decode,
                       glinattn_spec_decode, glinattn_state_copy, library, state_bytes, status_string, version)

__all__ = ["GLA", "GDN", "NLA", "F32", "BF16", "GlinattnError", "glinattn_prefill", "glinattn_decode",
           "glinattn_spec_decode", "glinattn_replay", "glinattn_state_copy", "glinattn_selective_scan",
           "glinattn_selective_scan_decode", "library", "version", "status_string", "state_bytes"]
