"""CPU oracle for the token-tree verification step (test infrastructure, not product code).

A plain, slow, float64 NumPy restatement of what the method computes, written from the method's
published definitions:

* ``oracle.attention`` -- tree-masked attention: every draft-tree node attends to its sequence's
  KV-cache prefix and to its own ancestors (itself included), found by walking parent pointers.
  EAGLE paper explainer, "Static tree" section; speculative-decoding survey explainer, "Token Tree
  verification" paragraph.
* ``oracle.paged`` -- the paged KV cache (slot s of sequence b in page block_table[b, s // P], row
  s % P) and post-accept compaction (the accepted path's keys and values move next to the root).
  Survey explainer, "vLLMでの実装状況" section (speculative decoding on PagedAttention); EAGLE
  explainer, vLLM usage section (the tree's extra KV-cache memory).
* ``oracle.dyntree`` -- dynamic (EAGLE-2-style) draft-tree construction: level-by-level expansion
  of the best frontier nodes by their top draft tokens, then the best candidates by cumulative
  draft log-probability.  EAGLE-3 explainer, 背景と動機 / EAGLE-2との統合 (EAGLE-2's dynamic
  tree).
* ``oracle.lmhead`` -- the LM head reduced to what verification reads: per row the max, the sum of
  exp((l - max) / T), the argmax and the logits of tested tokens.  EAGLE explainer (the target
  forward over the tree); survey explainer, Formal Definition (q_j and q_j(x~)).
* ``oracle.filtering`` -- top-k / top-p filtered target distributions (the filtered logits feed
  ``oracle.verify`` unchanged).  Survey explainer, verification taxonomy (speculative sampling
  with top-k / top-p).
* ``oracle.verify`` -- speculative-sampling accept/reject over the tree, the walk to the accepted
  path and the resample of the bonus token from norm(max(0, q - p)); temperature 0 is greedy
  argmax matching.  Survey explainer, "Formal Definition" (draft / verify / accept-reject
  equations) and the verification taxonomy table.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg import this package.
It shares no code with the CUDA path and imports nothing from it.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py`` against library routines,
closed forms, exact rational enumeration and brute force (none re-types the oracle's formulas).
"""
from . import attention, dyntree, filtering, lmhead, paged, verify  # noqa: F401
