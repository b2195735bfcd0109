"""GB300-native batched draft-token verification for speculative decoding.

The verification step of speculative decoding (the Leviathan/Chen rule as the
pages "Speculative decoding and EAGLE", "Speculative decoding: draft, verify,
repeat" and "Speculative Decoding: from idea to SOTA" define it) as hand-written
sm_103a CUDA behind a C ABI (include/spec_verify.h, libspecverify.so); this
package is the thin binding plus the seeded workload generators.
"""
from .binding import (  # noqa: F401
    SPEC_BF16, SPEC_DRAFT_LOGITS, SPEC_DRAFT_PROBS, SPEC_F32, SPEC_MAX_K, SPEC_MAX_TREE_NODES,
    SpecError, declared_functions, last_error, lib, spec_debug_residual, spec_debug_stall, spec_profile_begin,
    spec_profile_end, spec_tree_workspace_bytes, spec_verify_greedy, spec_verify_sample,
    spec_verify_sample_noalloc, spec_tree_mask, spec_kv_commit, spec_row_stats, spec_tree_draft,
    spec_verify_tree_greedy, spec_workspace_bytes, status_string, workspace,
)
