"""Oracle: speculative-sampling verification of a draft token tree (test infrastructure).

Definitions followed (speculative-decoding survey explainer, "Formal Definition"):

* drafts x~_i are sampled from the draft distribution p_i; the target gives q_i at every position,
  one more than the number of drafts, so that a token can be sampled where the walk stops;
* draft x~_i is accepted if r < min(1, q_i(x~_i) / p_i(x~_i)), r ~ U[0, 1);
* at the first rejected position c the next token is drawn from norm(max(0, q_c - p_c));
* greedy verification (the taxonomy table) accepts a draft when it equals the target's greedy
  choice.

Tree form (token-tree verification row of the taxonomy; EAGLE explainer "Static tree").  The pages
give the rule for a chain only; the reading used here, and listed with the other readings in the
design notes, is the sibling-ordered residual rule: the children of the current node c are tried in
ascending node index against the current target distribution q (initially q_c); child k is accepted
iff r_k * p_c(x~_k) < q(x~_k) (the division-free form of the pages' test); on rejection q becomes
norm(max(0, q - p_c)) (kept unchanged if that residual sums to 0); on acceptance the walk moves to
child k.  When every child of c is rejected, or c has no children, the bonus token is drawn from the
current q by inverse CDF with u = uniforms[0]:  y = min{y : sum_{z<=y} w(z) > u * sum_z w(z)}, and if
rounding leaves no such y, the last y with w(y) > 0.  Temperature T > 0 means q_j = softmax(l_j / T);
T = 0 is greedy: accept the first child whose token equals argmax l_c (lowest index on ties), bonus
= argmax l_c.  Row j of the logits / draft probabilities belongs to node j's children.

The walk (``verify_walk``) is generic over the number type: it runs on float64 arrays and on object
arrays of ``fractions.Fraction`` (used by the exact enumeration tests).
"""
from __future__ import annotations

from typing import Callable, Dict, List, Optional, Sequence

import numpy as np

# per-sequence status bits (same meaning as the library's)
ST_BAD_TREE = 1
ST_BAD_LEN = 2
ST_BAD_TOKEN = 4
ST_NONFINITE = 8

NEAR_TIE = 1e-6


# ----------------------------------------------------------------------------------------------
# building blocks
# ----------------------------------------------------------------------------------------------
def target_distribution(logits_row, T: float) -> np.ndarray:
    """q = softmax(l / T) in float64 (max subtracted before exponentiation)."""
    x = np.asarray(logits_row, dtype=np.float64) / float(T)
    w = np.exp(x - x.max())
    return w / w.sum()


def children(parent_row) -> Dict[int, List[int]]:
    """Children of every node, in ascending node index."""
    kids: Dict[int, List[int]] = {i: [] for i in range(len(parent_row))}
    for i in range(1, len(parent_row)):
        kids[int(parent_row[i])].append(i)
    return kids


def residual(q, p):
    """norm(max(0, q - p)) and its normaliser beta; q is kept when beta == 0."""
    r = np.maximum(q - p, 0 * q)
    beta = r.sum()
    if beta > 0:
        return r / beta, beta
    return q, beta


def sibling_tests(q, p, child_tokens: Sequence[int], child_r: Sequence):
    """Sibling-ordered accept/reject at one node.

    Returns (position of the accepted child or None, per-child records (q_used, p_x, r, accepted)
    for the children tested, distribution to sample from if no child is accepted).
    """
    records = []
    for pos, (x, r) in enumerate(zip(child_tokens, child_r)):
        qx, px = q[x], p[x]
        accepted = bool(r * px < qx)
        records.append((qx, px, r, accepted))
        if accepted:
            return pos, records, q
        q, _ = residual(q, p)
    return None, records, q


def greedy_choice(logits_row) -> int:
    """argmax with the lowest index on ties."""
    return int(np.argmax(np.asarray(logits_row)))


def inverse_cdf(w, u):
    """Inverse-CDF draw from unnormalised weights w with uniform u.

    Returns (y, gap) where gap is the distance from u * S to the nearest cumulative boundary of y,
    divided by S (the CDF margin of the decision).
    """
    S = w.sum()
    t = u * S
    C = np.cumsum(w)
    above = np.nonzero(np.array([bool(c > t) for c in C]) if C.dtype == object else (C > t))[0]
    if len(above):
        y = int(above[0])
    else:
        nz = np.nonzero(np.array([bool(x > 0) for x in w]) if w.dtype == object else (w > 0))[0]
        y = int(nz[-1])
    lower = C[y - 1] if y > 0 else 0 * S
    gap = min(C[y] - t, t - lower) / S
    return y, gap


def decision_margin(r, qx, px):
    """Distance of r from the decision boundary q/p of the test r * p < q."""
    if px > 0:
        return abs(r - qx / px)
    return qx


# ----------------------------------------------------------------------------------------------
# the walk
# ----------------------------------------------------------------------------------------------
def verify_walk(tokens, parent, uniforms, q_of: Callable[[int], np.ndarray],
                p_of: Callable[[int], np.ndarray]):
    """Speculative-sampling walk over one sequence's tree (T > 0 form).

    ``q_of(j)`` / ``p_of(j)`` give the target / draft distributions at node j.  Returns a dict with
    the accepted node path (root excluded), the bonus token, the per-node test records and the
    margins of every decision taken along the way.
    """
    kids = children(parent)
    c = 0
    path: List[int] = []
    tests = {}
    margins = []
    while True:
        ks = kids[c]
        if not ks:
            terminal = q_of(c)
            break
        pos, recs, q_final = sibling_tests(q_of(c), p_of(c), [int(tokens[k]) for k in ks],
                                           [uniforms[k] for k in ks])
        for k, rec in zip(ks, recs):
            tests[k] = rec
            margins.append(decision_margin(rec[2], rec[0], rec[1]))
        if pos is None:
            terminal = q_final
            break
        c = ks[pos]
        path.append(c)
    bonus, gap = inverse_cdf(terminal, uniforms[0])
    margins.append(gap)
    return {"path": path, "bonus": bonus, "tests": tests, "margins": margins,
            "terminal": terminal, "last": c}


def greedy_walk(tokens, parent, logits):
    """Temperature-0 walk: follow the first child whose token is the parent's argmax."""
    kids = children(parent)
    c = 0
    path: List[int] = []
    while True:
        a = greedy_choice(logits[c])
        nxt = next((k for k in kids[c] if int(tokens[k]) == a), None)
        if nxt is None:
            return {"path": path, "bonus": a, "last": c}
        c = nxt
        path.append(c)


def node_test_table(tokens, parent, uniforms, q_of, p_of):
    """Sibling tests at every internal node (on or off the accepted path).

    Returns {child node: (q_used, p_x, r, accepted)} for every child that gets tested, i.e. every
    child whose earlier siblings were all rejected.
    """
    kids = children(parent)
    table = {}
    for j, ks in kids.items():
        if not ks:
            continue
        _, recs, _ = sibling_tests(q_of(j), p_of(j), [int(tokens[k]) for k in ks],
                                   [uniforms[k] for k in ks])
        for k, rec in zip(ks, recs):
            table[k] = rec
    return table


# ----------------------------------------------------------------------------------------------
# validation (status bits)
# ----------------------------------------------------------------------------------------------
def tree_status(parent_row, tokens_row=None, V: Optional[int] = None) -> int:
    """Status bits for one sequence's tree: bad parent pointers, draft tokens outside [0, V)."""
    st = 0
    n = len(parent_row)
    if int(parent_row[0]) != -1 or any(not (0 <= int(parent_row[i]) < i) for i in range(1, n)):
        st |= ST_BAD_TREE
    if tokens_row is not None and V is not None:
        if any(not (0 <= int(tokens_row[i]) < V) for i in range(1, n)):
            st |= ST_BAD_TOKEN
    return st


# ----------------------------------------------------------------------------------------------
# batched entry point (float64)
# ----------------------------------------------------------------------------------------------
def tree_verify(target_logits, draft_probs, tree_tokens, tree_parent, uniforms, temperature,
                with_table: bool = False):
    """Float64 verification of a batch.  Returns a dict of numpy arrays:

    accept_len [B], accepted_tokens [B, N] (-1 padded), accepted_nodes [B, N] (-1 padded),
    bonus [B], status [B], min_margin [B] (smallest fp64 decision margin along the walk; +inf for
    T = 0), near_tie [B] (min_margin < 1e-6), and with ``with_table`` child_q [B, N] (q used in
    each tested child's test, NaN where a node is not tested).
    """
    B, N, V = target_logits.shape
    T = float(temperature)
    out = {
        "accept_len": np.full(B, -1, np.int32),
        "accepted_tokens": np.full((B, N), -1, np.int32),
        "accepted_nodes": np.full((B, N), -1, np.int32),
        "bonus": np.full(B, -1, np.int32),
        "status": np.zeros(B, np.int32),
        "min_margin": np.full(B, np.inf),
        "near_tie": np.zeros(B, bool),
        "child_q": np.full((B, N), np.nan),
    }
    for b in range(B):
        st = tree_status(tree_parent[b], tree_tokens[b], V)
        if st:
            out["status"][b] = st
            continue
        par, tok = tree_parent[b], tree_tokens[b]
        if T == 0.0:
            res = greedy_walk(tok, par, target_logits[b])
        else:
            cache: Dict[int, np.ndarray] = {}

            def q_of(j, _b=b):
                if j not in cache:
                    cache[j] = target_distribution(target_logits[_b, j], T)
                return cache[j]

            def p_of(j, _b=b):
                return np.asarray(draft_probs[_b, j], dtype=np.float64)

            unif = [float(x) for x in uniforms[b]]
            res = verify_walk(tok, par, unif, q_of, p_of)
            out["min_margin"][b] = min(res["margins"])
            out["near_tie"][b] = out["min_margin"][b] < NEAR_TIE
            if with_table:
                for k, rec in node_test_table(tok, par, unif, q_of, p_of).items():
                    out["child_q"][b, k] = rec[0]
        path = res["path"]
        out["accept_len"][b] = len(path)
        out["accepted_nodes"][b, :len(path)] = path
        out["accepted_tokens"][b, :len(path)] = [int(tok[k]) for k in path]
        out["bonus"][b] = res["bonus"]
    return out
