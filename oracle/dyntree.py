"""Oracle: dynamic (EAGLE-2-style) draft-tree construction, in float64 (test infrastructure).

Pages followed: EAGLE-3 explainer, 背景と動機 and EAGLE-2との統合 (EAGLE-2 turns the static draft
tree into a dynamic one, built at inference time from the draft head's outputs, and EAGLE-3's head
plugs into that construction); survey explainer, 検証方式による分類 (token-tree verification
consumes such trees).  The pages give no procedure; this follows EAGLE-2's published
expand-then-rerank construction, restated:

* The value of a drafted node is the sum, along its path from the root, of the draft model's
  log-probabilities log softmax(l)[token] of each token under its parent's draft logits l (the
  root has value 0).
* Level 1 expands the root; level d > 1 expands the frontier chosen at level d - 1.  Expanding a
  frontier node (frontier slot i) makes candidates of its K highest draft logits (ties: lower token
  id first), in that order; candidate order within the level is i * K + r for the r-th token of
  slot i.  Every candidate joins the pool.
* The next frontier is the K candidates of the level with the highest values (ties: lower
  candidate order), listed in that order; its draft rows are the next level's input, slot by slot.
* The tree is the root plus the N - 1 pool candidates with the highest values (ties: shallower
  first, then lower candidate order).  A candidate's value is at most its parent's, so the chosen
  set contains every chosen node's parent.  Nodes are numbered by (depth, candidate order), which
  puts every parent before its children.

Draft rows are addressed in the order the levels consume them: row 0 is the root's (level 1), row
1 + (d - 2) K + i is frontier slot i's at level d >= 2.  A tree node's `node_row` is the row of
its own draft logits when it was expanded, else -1 (a node with children always has one).
"""
from __future__ import annotations

from typing import Dict, List

import numpy as np


def log_softmax(row) -> np.ndarray:
    """log softmax of one row in float64 (max subtracted before exponentiation)."""
    x = np.asarray(row, dtype=np.float64)
    m = x.max()
    return x - (m + np.log(np.exp(x - m).sum()))


def top_tokens(row, K: int) -> List[int]:
    """The K highest entries of a row, highest first, lower index first among equal values."""
    x = np.asarray(row, dtype=np.float64)
    order = np.lexsort((np.arange(x.shape[0]), -x))  # by -x, then by index
    return [int(t) for t in order[:K]]


class TreeBuilder:
    """One sequence's construction state: the pool of drafted candidates and the frontier."""

    def __init__(self, K: int):
        self.K = int(K)
        # pool entries: token (-1 for the root), parent pool index, value, depth, order in level
        self.token = [-1]
        self.parent = [-1]
        self.value = [0.0]
        self.depth = [0]
        self.order = [0]
        self.row_of = {}                # pool index -> draft row index (expanded nodes)
        self.frontier = [0]             # pool indices whose draft rows the next level reads
        self.level = 0
        self.frontier_margin = np.inf   # smallest gap at a frontier boundary (near-tie accounting)

    def expand(self, rows) -> List[int]:
        """Consume this level's draft rows (one per frontier slot, in slot order); return the new
        frontier (pool indices)."""
        rows = np.asarray(rows)
        assert rows.shape[0] == len(self.frontier)
        self.level += 1
        base = 0 if self.level == 1 else 1 + (self.level - 2) * self.K  # this level's first row
        for i, f in enumerate(self.frontier):
            self.row_of[f] = base + i
        cand = []
        for i, f in enumerate(self.frontier):
            lp = log_softmax(rows[i])
            for r, t in enumerate(top_tokens(rows[i], self.K)):
                self.token.append(t)
                self.parent.append(f)
                self.value.append(self.value[f] + float(lp[t]))
                self.depth.append(self.level)
                self.order.append(i * self.K + r)
                cand.append(len(self.token) - 1)
        # next frontier: the K best candidates of this level
        ranked = sorted(cand, key=lambda c: (-self.value[c], self.order[c]))
        nxt = ranked[: self.K]
        if len(ranked) > self.K:
            gap = self.value[ranked[self.K - 1]] - self.value[ranked[self.K]]
            self.frontier_margin = min(self.frontier_margin, gap)
        self.frontier = nxt
        return nxt

    def finalize(self, root_token: int, N: int) -> Dict[str, np.ndarray]:
        """The tree of the root and the N - 1 best candidates, numbered by (depth, order)."""
        cands = list(range(1, len(self.token)))
        ranked = sorted(cands, key=lambda c: (-self.value[c], self.depth[c], self.order[c]))
        n_sel = min(N - 1, len(ranked))
        chosen = ranked[:n_sel]
        rerank_margin = np.inf
        if len(ranked) > n_sel > 0:
            rerank_margin = self.value[ranked[n_sel - 1]] - self.value[ranked[n_sel]]
        nodes = [0] + sorted(chosen, key=lambda c: (self.depth[c], self.order[c]))
        pos = {c: j for j, c in enumerate(nodes)}
        n = len(nodes)
        out = {
            "tree_tokens": np.full(N, -1, np.int32),
            "tree_parent": np.full(N, -1, np.int32),
            "node_row": np.full(N, -1, np.int32),
            "node_value": np.full(N, np.nan),
            "n_nodes": n,
            "frontier_margin": self.frontier_margin,
            "rerank_margin": rerank_margin,
        }
        for j, c in enumerate(nodes):
            out["tree_tokens"][j] = root_token if c == 0 else self.token[c]
            out["tree_parent"][j] = -1 if c == 0 else pos[self.parent[c]]
            out["node_row"][j] = self.row_of.get(c, -1)
            out["node_value"][j] = self.value[c]
        return out


def build_tree(level_rows, root_token: int, K: int, N: int) -> Dict[str, np.ndarray]:
    """One sequence: level_rows[d - 1] holds level d's draft rows ([1, V] for d = 1, [K, V] after;
    only the first len(frontier) rows of a level are read)."""
    tb = TreeBuilder(K)
    for rows in level_rows:
        tb.expand(np.asarray(rows)[: len(tb.frontier)])
    return tb.finalize(root_token, N)


def build_trees(draft_rows, root_tokens, K: int, D: int, N: int) -> Dict[str, np.ndarray]:
    """A batch: draft_rows [B, 1 + (D - 1) K, V] in the row order above."""
    draft_rows = np.asarray(draft_rows)
    B = draft_rows.shape[0]
    outs = []
    for b in range(B):
        levels = [draft_rows[b, :1]] + [draft_rows[b, 1 + (d - 2) * K: 1 + (d - 1) * K]
                                         for d in range(2, D + 1)]
        outs.append(build_tree(levels, int(root_tokens[b]), K, N))
    res = {k: np.stack([o[k] for o in outs]) for k in ("tree_tokens", "tree_parent", "node_row",
                                                       "node_value")}
    for k in ("n_nodes", "frontier_margin", "rerank_margin"):
        res[k] = np.array([o[k] for o in outs])
    return res
