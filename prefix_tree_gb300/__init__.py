"""prefix_tree_gb300 — GB300 (sm_103a) hot path of prefix-tree (rollout-tree) training.

The CUDA library libtt (C ABI in include/tt.h) computes every token's
log-probability of a DFS-serialised rollout tree exactly once: tree tables,
tree attention forward/backward (whole tree or path-at-a-time chunks), the
branch-fraction weighted log-prob loss, and that loss fused with the LM head. This package is its thin binding.
"""
from ._native import (KERNEL_CLASSES, TTError, Tree, DTA_DEFAULT_SLOTS, DTA_ORDER_GREEDY, DTA_ORDER_INDEX,  # noqa
                      DtaPlan, check_err,
                      dta_leaf_order, dta_tree_attn, dta_workspace_bytes, exported_symbols,
                      kernel_timing, kernel_timing_read, lib, lmhead_logprob, lmhead_logprob_bwd, new_err, tree_attn_bwd,
                      tree_attn_chunk_bwd,
                      tree_attn_chunk_fwd, tree_attn_fwd, tree_build, tree_partition, tree_schedules, trie_build,
                      weighted_logprob)

__all__ = ["DTA_DEFAULT_SLOTS", "DTA_ORDER_GREEDY", "DTA_ORDER_INDEX", "DtaPlan", "KERNEL_CLASSES", "TTError", "Tree", "check_err", "dta_leaf_order",
           "dta_tree_attn", "dta_workspace_bytes", "exported_symbols",
           "kernel_timing", "kernel_timing_read", "lib", "lmhead_logprob", "lmhead_logprob_bwd", "new_err", "tree_attn_bwd", "tree_attn_chunk_bwd", "tree_attn_chunk_fwd",
           "tree_attn_fwd", "tree_build", "tree_partition", "tree_schedules", "trie_build", "weighted_logprob"]
