"""Oracle: tree-masked attention in float64 (test infrastructure).

Definition followed (EAGLE paper explainer, "Static tree" section: the target model verifies all
tree paths in one forward pass with a tree attention mask; survey explainer, verification taxonomy,
"Token Tree verification"): node i of the draft tree sees

    K_i = {prefix positions 0 .. L_b - 1}  U  {L_b + j : j is an ancestor of i, or i itself}

and its output for query head h is the softmax-weighted sum of the values over K_i, with scores
scale * <q, k_t>.  Query head h reads KV head floor(h / g), g = Hq / Hkv (contiguous grouping, a
reading: the pages are silent on GQA).  The caller stores node j's key/value at cache slot L_b + j.
The ancestor set is found by walking parent pointers; no bitmask is involved.
"""
from __future__ import annotations

from typing import Iterable, Optional, Tuple

import numpy as np


def ancestor_set(parent_row, i: int) -> list:
    """Node i and all its ancestors, by following parent pointers up to the root (-1)."""
    out = []
    seen = 0
    while i >= 0:
        out.append(int(i))
        i = int(parent_row[i])
        seen += 1
        if seen > len(parent_row):
            raise ValueError("parent pointers contain a cycle")
    return sorted(out)


def node_attention(q_rows: np.ndarray, k_seq: np.ndarray, v_seq: np.ndarray, prefix_len: int,
                   tree_keys: Iterable[int], scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """Attention of ``q_rows`` [g, D] over prefix keys 0..L-1 plus the listed tree slots.

    Returns (out [g, D], lse [g]).  Scores are computed for the prefix slice and for the tree slots
    separately and concatenated: the key set is exactly K_i.
    """
    slots = [prefix_len + int(j) for j in tree_keys]
    k_set = np.concatenate([k_seq[:prefix_len], k_seq[slots]], axis=0)
    v_set = np.concatenate([v_seq[:prefix_len], v_seq[slots]], axis=0)
    s = scale * (q_rows @ k_set.T)                      # [g, |K_i|]
    m = s.max(axis=1, keepdims=True)
    w = np.exp(s - m)
    l = w.sum(axis=1, keepdims=True)
    out = (w @ v_set) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


def tree_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                   prefix_lens: np.ndarray, tree_parent: np.ndarray, scale: float,
                   nodes: Optional[Iterable[Tuple[int, int]]] = None):
    """Float64 tree attention.

    q [B, N, Hq, D], k_cache / v_cache [B, Hkv, Lmax, D] (float64), prefix_lens [B],
    tree_parent [B, N].  Returns (out [B, N, Hq, D], lse [B, Hq, N]).  If ``nodes`` lists
    (b, i) pairs, only those nodes are computed (the rest stay NaN).
    """
    B, N, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    g = Hq // Hkv
    out = np.full((B, N, Hq, D), np.nan)
    lse = np.full((B, Hq, N), np.nan)
    todo = nodes if nodes is not None else [(b, i) for b in range(B) for i in range(N)]
    for b, i in todo:
        L = int(prefix_lens[b])
        anc = ancestor_set(tree_parent[b], i)
        for kvh in range(Hkv):
            hs = slice(kvh * g, (kvh + 1) * g)
            o, ls = node_attention(q[b, i, hs], k_cache[b, kvh], v_cache[b, kvh], L, anc, scale)
            out[b, i, hs] = o
            lse[b, hs, i] = ls
    return out, lse
