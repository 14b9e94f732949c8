"""GB300-native verification step of speculative decoding.

The compute path is the C-ABI library ``libspec_verify.so`` (hand-written CUDA
for sm_103a); this package is its thin Python binding (argument marshalling
only).  The library is loaded on first use; importing the package (or its
``workloads`` input generator) does not touch CUDA.
"""
from __future__ import annotations

__all__ = ["spec_verify", "spec_verify_ex", "spec_verify_host", "spec_verify_noalloc", "spec_verify_points",
           "spec_verify_tree_greedy", "spec_verify_tree", "spec_verify_trees_greedy", "spec_verify_trees",
           "spec_tree_mask", "spec_tree_max_depth", "spec_ngram_propose", "spec_topk", "spec_eagle2_expand",
           "spec_eagle2_rerank", "spec_selftest_wait", "spec_get_status", "spec_arm_rows_event", "spec_arm_timer",
           "spec_debug_fail_launch", "spec_noalloc_get_status", "spec_debug_noalloc_status",
           "spec_error_string", "spec_last_error_message", "spec_shutdown",
           "SpecError", "library"]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
