"""GB300-native batched draft-verification sampler for speculative decoding.

The computation lives in libspecverify.so (hand-written sm_103a CUDA behind
the C ABI of include/specverify.h); this package is its Python binding.
"""
from ._binding import (ROW_STATUS, SPEC_BF16, SPEC_F32, SPEC_GREEDY, SPEC_STOCHASTIC,  # noqa: F401
                       SpecError, debug_force_wait_timeout, get_wait_timeout_ns, lib,
                       set_wait_timeout_ns, spec_adaptive_tree_policy, spec_drift_residuals,
                       spec_kv_compact_tree,
                       spec_rollback_lengths, spec_verify_chain, spec_verify_tree)
