"""GB300-native token-tree verification for EAGLE-style speculative decoding.

Two calls make up the hot path, both hand-written CUDA for sm_103a behind a C ABI
(``include/spectree.h``, built into ``libspectree.so``):

* ``spec_tree_attention`` -- tree-masked split-KV attention of the draft tree's queries over each
  sequence's KV-cache prefix and the node's own ancestors;
* ``spec_tree_verify`` -- speculative-sampling accept/reject over the tree, the walk to the accepted
  path and the bonus-token resample (greedy argmax matching at temperature 0).

Beside them: ``spec_tree_attention_paged`` (the same attention over a paged KV cache) and
``spec_kv_compact`` / ``spec_kv_compact_paged`` (after verification, the accepted path's keys and
values move next to the root), ``spec_tree_verify_filtered`` (verification against the top-k /
top-p filtered target distribution), and ``spec_tree_expand`` / ``spec_tree_finalize`` (dynamic
draft-tree construction, one level per drafter step), ``spec_lm_head_stats`` (the LM head fused
with the per-row statistics verification reads), ``spec_tree_verify_greedy`` (temperature-0
verification from those statistics' argmax, no logit rows) and ``spec_tree_verify_head``
(verification from the nodes' hidden states and the LM head: full logit rows only where the walk
needs residual rounds or the bonus draw).

The Python functions of the same names only marshal torch tensors into pointers and the current
CUDA stream.  There is no CPU fallback: a missing library raises.
"""
from ._binding import (  # noqa: F401
    SpecError,
    spec_kv_compact,
    spec_lm_head_pack,
    spec_lm_head_packed_bytes,
    spec_lm_head_stats,
    spec_lm_head_stats_workspace,
    spec_kv_compact_paged,
    spec_tree_attention,
    spec_tree_attention_paged,
    spec_tree_attention_workspace,
    spec_tree_build_workspace,
    spec_tree_expand,
    spec_tree_finalize,
    spec_tree_verify,
    spec_tree_verify_filtered,
    spec_tree_verify_filtered_workspace,
    spec_tree_verify_greedy,
    spec_tree_verify_head,
    spec_tree_verify_head_workspace,
    spec_tree_verify_noalloc,
    spec_tree_verify_workspace,
    spec_status_string,
    spec_debug_set_verify_wait_polls,
    lib,
)
