"""Oracle: the target model's LM head reduced to the statistics verification reads, float64
(test infrastructure).

Pages followed: EAGLE explainer, the target model's forward pass over the tree (the LM head turns
each node's hidden state into next-token logits, the rows the verification reads); survey explainer,
Formal Definition, 検証フェーズ (q_j = softmax of the target logits at node j, and each draft token
x~ is tested against q_j(x~)).  Reading: the verification needs, per row, the max m, the sum
S = sum_y exp((l_y - m) / T), the argmax (for T = 0) and the logits of the tokens it tests, so
q_j(x~) = exp((l_x~ - m) / T) / S; the full logit row need not exist.

logits = hidden @ weight^T with hidden [M, H] and weight [V, H], both bf16 in the caller's tensors
(their exact values are used here, in float64).
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

from . import verify as _verify


def logits(hidden, weight) -> np.ndarray:
    """[M, V] = hidden [M, H] @ weight [V, H]^T in float64."""
    return np.asarray(hidden, np.float64) @ np.asarray(weight, np.float64).T


def row_stats(lg, T: float, gather_idx: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """Per row of lg [M, V]: max, sumexp = sum exp((l - max) / T), argmax (lowest index among
    equal maxima), and the logits at gather_idx [M, G] (-1: none, gives NaN)."""
    lg = np.asarray(lg, np.float64)
    m = lg.max(axis=1)
    s = np.exp((lg - m[:, None]) / float(T)).sum(axis=1)
    am = np.argmax(lg, axis=1).astype(np.int32)  # first occurrence: lowest index
    out = {"max": m, "sumexp": s, "argmax": am}
    if gather_idx is not None:
        gi = np.asarray(gather_idx)
        g = np.full(gi.shape, np.nan)
        ok = gi >= 0
        rows = np.nonzero(ok)[0]
        g[ok] = lg[rows, gi[ok]]
        out["gather"] = g
    # the gap between the two largest distinct logits of each row (argmax near-tie accounting)
    part = np.sort(lg, axis=1)
    out["top_gap"] = part[:, -1] - part[:, -2] if lg.shape[1] > 1 else np.full(lg.shape[0], np.inf)
    return out


def lm_head_stats(hidden, weight, T: float, gather_idx=None) -> Dict[str, np.ndarray]:
    return row_stats(logits(hidden, weight), T, gather_idx)


def tree_verify_from_head(hidden, weight, draft_probs, tree_tokens, tree_parent, uniforms,
                          T: float, with_table: bool = False):
    """Tree verification (oracle/verify.py, survey explainer, Formal Definition, 検証フェーズ) of the
    logits the LM head gives at every node (EAGLE explainer: the target's forward over the tree):
    hidden [B, N, H] and weight [V, H], the exact values of the bf16 operands, in float64.  The
    method never needs the logit matrix as a whole; its results are defined by it."""
    h = np.asarray(hidden, np.float64)
    B, N, H = h.shape
    lg = logits(h.reshape(B * N, H), weight).reshape(B, N, -1)
    return _verify.tree_verify(lg, draft_probs, tree_tokens, tree_parent, uniforms, T,
                               with_table=with_table)
