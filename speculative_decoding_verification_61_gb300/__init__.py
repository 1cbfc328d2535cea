"""GB300 (sm_103a) verify-and-resample step of speculative decoding.

Python binding of the C ABI in include/spec_verify.h.  Every step of the
computation runs in the CUDA library (_build/libspecverify.so); this module
only marshals torch tensors (device memory, streams) into pointers.  If the
library is missing or cannot be loaded, every call raises: there is no CPU
fallback.

    from speculative_decoding_verification_61_gb300 import spec_verify, spec_draft_sample
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    ABI_VERSION,
    AdaptiveK,
    BF16,
    F32,
    MAX_B,
    MAX_K,
    MAX_SHARDS,
    MAX_TREE_NODES,
    MAX_V,
    NOALLOC_SCRATCH_BYTES,
    SPEC_ERRORS,
    SpecError,
    exported_symbols,
    lib,
    lib_path,
    noalloc_bytes,
    selfcheck_wait_timeout,
    shard_workspace,
    shard_workspace_bytes,
    shutdown,
    spec_draft_sample,
    spec_draft_sample_lse,
    spec_round,
    spec_round_host,
    spec_shard_decide,
    spec_shard_draw,
    spec_shard_stats,
    spec_tree_draft_sample,
    spec_tree_verify,
    spec_verify,
    spec_verify_lse,
    spec_verify_noalloc,
    workspace_bytes,
    workspace_status,
)
