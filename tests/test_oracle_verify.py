"""Pins for the verification oracle (CPU only).

What pins what:
* softmax at temperature T           -> scipy.special.softmax (library routine)
* greedy walk                        -> brute force over every root path of the tree
* sampling walk + residual + bonus   -> exact rational enumeration of every draft draw, every
                                        accept/reject branch and every bonus token: the emitted
                                        tokens followed by target sampling are distributed exactly
                                        as the target model (the pages' lossless claim); the
                                        rejected "independent flags" reading fails the same check
* chain acceptance                   -> closed form E[accept_len] = sum_k prod_{j<=k} alpha_j,
                                        alpha_j = sum_y min(p_j, q_j) (expectation of the EAGLE-3
                                        explainer's chained-acceptance product)
* residual                           -> sums to 1, non-negative, beta = 1 - sum min(p, q)
* inverse CDF                        -> exact boundaries on rational weights, fallback rule
* T -> 0                             -> sampling at tiny T equals greedy on untied rows
* near-tie margins (decision_margin, -> hand-derived rationals, and the defining property: moving
  the CDF gap of inverse_cdf, a walk's   a decision's uniform by less than its margin keeps the
  min_margin)                             outcome, by slightly more towards the boundary changes it
                                        (per test, per draw, and for a whole walk's minimum)
"""
import itertools
from fractions import Fraction as F

import numpy as np
import pytest
import scipy.special

from oracle import verify as OV
from speculative_decoding_token_spec_gb300 import workloads as W


# ----------------------------------------------------------------------------------------------
def test_target_distribution_matches_scipy_softmax():
    rng = np.random.default_rng(0)
    for T in (0.3, 1.0, 1.7):
        row = (rng.standard_normal(5000) * 3).astype(np.float32)
        ref = scipy.special.softmax(row.astype(np.float64) / T)
        np.testing.assert_allclose(OV.target_distribution(row, T), ref, rtol=1e-12, atol=1e-300)


def test_greedy_choice_lowest_index_on_ties():
    assert OV.greedy_choice(np.array([1.0, 3.0, 3.0, 2.0])) == 1
    assert OV.greedy_choice(np.array([-np.inf, -5.0, -5.0])) == 1


# ----------------------------------------------------------------------------------------------
def _all_paths(parent):
    """Every root->node path, listed as node sequences (root excluded)."""
    paths = []
    for i in range(1, len(parent)):
        p, n = [], i
        while n > 0:
            p.append(n)
            n = int(parent[n])
        paths.append(p[::-1])
    return paths


@pytest.mark.parametrize("seed", range(12))
def test_greedy_walk_is_longest_matching_path(seed):
    """Brute force: the accepted path is the longest root path whose every token is its parent's
    argmax (sibling tokens are distinct, as top-k drafting gives), bonus = argmax at its end."""
    rng = np.random.default_rng(seed)
    N, V = 15, 6
    par = W.make_tree(rng, N, 4, 5)
    logits = rng.standard_normal((N, V))
    kids = OV.children(par)
    tok = np.zeros(N, dtype=np.int64)
    for j, ks in kids.items():
        if not ks:
            continue
        # distinct sibling tokens; bias towards the argmax so long matches happen
        choice = list(rng.permutation(V)[:len(ks)])
        a = int(np.argmax(logits[j]))
        if a not in choice and rng.random() < 0.7:
            choice[int(rng.integers(len(choice)))] = a
        for k, t in zip(ks, choice):
            tok[k] = t
    best = []
    for path in _all_paths(par):
        ok = all(tok[n] == np.argmax(logits[int(par[n])]) for n in path)
        if ok and len(path) > len(best):
            best = path
    res = OV.greedy_walk(tok, par, logits)
    assert res["path"] == best
    end = best[-1] if best else 0
    assert res["bonus"] == int(np.argmax(logits[end]))


# ----------------------------------------------------------------------------------------------
# exact losslessness
# ----------------------------------------------------------------------------------------------
def _rand_dist(rng, V, zeros=True):
    w = [int(x) for x in rng.integers(0 if zeros else 1, 7, size=V)]
    if sum(w) == 0:
        w[int(rng.integers(V))] = 1
    s = sum(w)
    return np.array([F(x, s) for x in w], dtype=object)


def _tables(rng, V, depth):
    """Target and draft distributions for every token prefix of length <= depth."""
    q, p = {}, {}
    for L in range(depth + 1):
        for s in itertools.product(range(V), repeat=L):
            q[s] = _rand_dist(rng, V)
            p[s] = _rand_dist(rng, V)
    return q, p


def _threshold(qx, px):
    if px > 0:
        return min(F(1), qx / px)
    return F(1) if qx > 0 else F(0)


def _path_tokens(parent, tokens, j):
    out = []
    while j > 0:
        out.append(int(tokens[j]))
        j = int(parent[j])
    return tuple(out[::-1])


def _emitted_distribution(parent, V, qtab, ptab, walk):
    """Exact distribution of the emitted token sequence (accepted drafts + bonus).

    Enumerates every draft assignment (drafts drawn from the parent's draft row, siblings i.i.d.),
    every accept/reject branch (r = 0 realises 'r < threshold', r = 1 realises 'r >= threshold';
    branch weight = threshold or 1 - threshold; nodes never tested must carry r = 0) and every
    bonus token (u set to the lower CDF boundary of y, weight w(y) / S).  ``walk`` is the walk under
    test; it returns (path nodes, tests {node: (q, p, r, accepted)}, terminal weights, bonus).
    """
    N = len(parent)
    dist = {}
    for draft in itertools.product(range(V), repeat=N - 1):
        tokens = np.array((0,) + draft)
        pa = F(1)
        for i in range(1, N):
            pa *= ptab[_path_tokens(parent, tokens, int(parent[i]))][tokens[i]]
            if pa == 0:
                break
        if pa == 0:
            continue

        def q_of(j, _t=tokens):
            return qtab[_path_tokens(parent, _t, j)]

        def p_of(j, _t=tokens):
            return ptab[_path_tokens(parent, _t, j)]

        for rbits in itertools.product((0, 1), repeat=N - 1):
            unif = [F(0)] + [F(b) for b in rbits]
            path, tests, terminal, _ = walk(tokens, parent, unif, q_of, p_of)
            wgt = pa
            for k in range(1, N):
                if k in tests:
                    t = _threshold(tests[k][0], tests[k][1])
                    wgt *= t if rbits[k - 1] == 0 else (1 - t)
                elif rbits[k - 1] == 1:
                    wgt = 0
                if wgt == 0:
                    break
            if wgt == 0:
                continue
            S = terminal.sum()
            C = np.cumsum(terminal)
            for y in range(V):
                if terminal[y] == 0:
                    continue
                lower = C[y - 1] if y > 0 else F(0)
                unif[0] = lower / S
                path2, _, _, bonus = walk(tokens, parent, unif, q_of, p_of)
                assert path2 == path and bonus == y      # inverse CDF hits y at its boundary
                seq = tuple(int(tokens[n]) for n in path) + (y,)
                dist[seq] = dist.get(seq, F(0)) + wgt * terminal[y] / S
    return dist


def _check_lossless(dist, qtab, V, depth):
    """P(E_1..k = e, |E| >= k) + sum_{j<k} P(E = e_1..j) prod_{t>j} q(e_t|e_<t) == prod q(e_t|e_<t)."""
    assert sum(dist.values()) == 1
    bad = []
    for k in range(1, depth + 2):
        for e in itertools.product(range(V), repeat=k):
            target = F(1)
            for t in range(k):
                target *= qtab[e[:t]][e[t]]
            lhs = sum((pr for s, pr in dist.items() if len(s) >= k and s[:k] == e), F(0))
            for j in range(1, k):
                pr = dist.get(e[:j], F(0))
                if pr:
                    tail = F(1)
                    for t in range(j, k):
                        tail *= qtab[e[:t]][e[t]]
                    lhs += pr * tail
            if lhs != target:
                bad.append((e, lhs, target))
    return bad


def _oracle_walk(tokens, parent, unif, q_of, p_of):
    res = OV.verify_walk(tokens, parent, unif, q_of, p_of)
    return res["path"], res["tests"], res["terminal"], res["bonus"]


def _depth(parent):
    d = [0] * len(parent)
    for i in range(1, len(parent)):
        d[i] = d[int(parent[i])] + 1
    return max(d)


TREES = {
    "chain3": [-1, 0, 1, 2],
    "two_siblings": [-1, 0, 0],
    "three_siblings": [-1, 0, 0, 0],
    "mixed": [-1, 0, 0, 1, 2],
    "sibling_subtrees": [-1, 0, 0, 1, 1],
}


@pytest.mark.parametrize("name", sorted(TREES))
@pytest.mark.parametrize("seed", [0, 1])
def test_lossless_exact_enumeration(name, seed):
    parent = np.array(TREES[name])
    V = 3
    rng = np.random.default_rng(1000 * seed + len(name))
    depth = _depth(parent)
    qtab, ptab = _tables(rng, V, depth + 1)
    dist = _emitted_distribution(parent, V, qtab, ptab, _oracle_walk)
    assert _check_lossless(dist, qtab, V, depth) == []


def _independent_flags_walk(tokens, parent, unif, q_of, p_of):
    """The rejected reading: every child tested against the unmodified q of its parent."""
    kids = OV.children(parent)
    c, path, tests = 0, [], {}
    while True:
        ks = kids[c]
        if not ks:
            terminal = q_of(c)
            break
        q, p = q_of(c), p_of(c)
        nxt = None
        for k in ks:
            x = int(tokens[k])
            acc = bool(unif[k] * p[x] < q[x])
            tests[k] = (q[x], p[x], unif[k], acc)
            if acc:
                nxt = k
                break
        if nxt is None:
            terminal, _ = OV.residual(q, p)
            break
        c = nxt
        path.append(c)
    y, _ = OV.inverse_cdf(terminal, unif[0])
    return path, tests, terminal, y


def test_independent_flags_reading_is_not_lossless():
    parent = np.array(TREES["two_siblings"])
    rng = np.random.default_rng(3)
    qtab, ptab = _tables(rng, 3, 2)
    dist = _emitted_distribution(parent, 3, qtab, ptab, _independent_flags_walk)
    assert _check_lossless(dist, qtab, 3, 1) != []


def test_first_emitted_token_is_target_distributed_mixed_tree_v4():
    """Larger alphabet on a branching tree: the first emitted token is distributed as q_root."""
    parent = np.array([-1, 0, 0, 1])
    V = 4
    rng = np.random.default_rng(44)
    qtab, ptab = _tables(rng, V, 3)
    dist = _emitted_distribution(parent, V, qtab, ptab, _oracle_walk)
    first = [sum((pr for s, pr in dist.items() if s[0] == y), F(0)) for y in range(V)]
    assert first == list(qtab[()])


# ----------------------------------------------------------------------------------------------
def test_chain_expected_accept_length_closed_form():
    """Chain whose rows do not depend on the prefix: E[accept_len] = sum_k prod_{j<=k} alpha_j."""
    V, K = 3, 3
    rng = np.random.default_rng(9)
    rows_q = [_rand_dist(rng, V) for _ in range(K + 1)]
    rows_p = [_rand_dist(rng, V, zeros=False) for _ in range(K + 1)]
    parent = np.array(W.chain_tree(K + 1))
    qtab, ptab = {}, {}
    for L in range(K + 2):
        for s in itertools.product(range(V), repeat=L):
            qtab[s], ptab[s] = rows_q[min(L, K)], rows_p[min(L, K)]
    dist = _emitted_distribution(parent, V, qtab, ptab, _oracle_walk)
    e_len = sum(pr * (len(s) - 1) for s, pr in dist.items())
    alpha = [sum(min(a, b) for a, b in zip(rows_p[j], rows_q[j])) for j in range(K)]
    closed = sum(np.prod(alpha[:k + 1]) for k in range(K))
    assert e_len == closed


# ----------------------------------------------------------------------------------------------
def test_residual_invariants():
    rng = np.random.default_rng(2)
    for _ in range(20):
        q = _rand_dist(rng, 6)
        p = _rand_dist(rng, 6)
        r, beta = OV.residual(q, p)
        assert beta == 1 - sum(min(a, b) for a, b in zip(p, q))
        if beta > 0:
            assert sum(r) == 1 and all(x >= 0 for x in r)
            assert all(r[y] == 0 for y in range(6) if q[y] <= p[y])
    q = np.array([F(1, 2), F(1, 2)], dtype=object)
    r, beta = OV.residual(q, q.copy())
    assert beta == 0 and list(r) == list(q)          # all-zero residual keeps q


def test_inverse_cdf_boundaries_and_fallback():
    w = np.array([F(0), F(1, 4), F(0), F(1, 2), F(1, 4)], dtype=object)
    assert OV.inverse_cdf(w, F(0))[0] == 1
    assert OV.inverse_cdf(w, F(1, 4))[0] == 3                  # C(1) = 1/4 is not > 1/4
    assert OV.inverse_cdf(w, F(3, 4) - F(1, 10**9))[0] == 3
    assert OV.inverse_cdf(w, F(3, 4))[0] == 4
    assert OV.inverse_cdf(w, F(1))[0] == 4                     # no C > S: last y with w > 0
    wf = np.array([0.0, 0.5, 0.5, 0.0])
    assert OV.inverse_cdf(wf, 1.0)[0] == 2


def test_small_temperature_matches_greedy():
    rng = np.random.default_rng(4)
    N, V = 12, 50
    for trial in range(5):
        par = W.make_tree(rng, N, 4, 4)
        logits = rng.standard_normal((N, V)) * 3
        kids = OV.children(par)
        tok = np.zeros(N, dtype=np.int64)
        for j, ks in kids.items():
            order = np.argsort(-logits[j])
            for r, k in enumerate(ks):
                tok[k] = order[r if rng.random() < 0.5 else min(r + 1, V - 1)]
        probs = np.full((N, V), 1.0 / V)
        unif = rng.random(N) * 0.98 + 0.01
        g = OV.greedy_walk(tok, par, logits)
        s = OV.verify_walk(tok, par, list(unif),
                           lambda j: OV.target_distribution(logits[j], 1e-3),
                           lambda j: probs[j])
        assert s["path"] == g["path"] and s["bonus"] == g["bonus"]


def test_batched_entry_point_and_status():
    cfg = W.config("tiny")
    case = W.make_verify_case(cfg, 1.0, seed=0)
    res = OV.tree_verify(case.target_logits, case.draft_probs, case.tree_tokens, case.tree_parent,
                         case.uniforms, 1.0, with_table=True)
    assert res["status"][0] == 0 and res["accept_len"][0] >= 0 and res["bonus"][0] >= 0
    L = res["accept_len"][0]
    assert (res["accepted_nodes"][0, :L] == np.arange(1, L + 1)).all()     # chain
    assert (res["accepted_tokens"][0, L:] == -1).all()
    bad = case.tree_parent.copy()
    bad[0, 3] = 3
    r2 = OV.tree_verify(case.target_logits, case.draft_probs, case.tree_tokens, bad,
                        case.uniforms, 1.0)
    assert r2["status"][0] == OV.ST_BAD_TREE and r2["bonus"][0] == -1
    tok = case.tree_tokens.copy()
    tok[0, 2] = cfg.V
    r3 = OV.tree_verify(case.target_logits, case.draft_probs, tok, case.tree_parent,
                        case.uniforms, 1.0)
    assert r3["status"][0] == OV.ST_BAD_TOKEN


def test_monte_carlo_chain_acceptance_fp64():
    """Float64 path at V = 1000: mean accept length over many uniforms vs the closed form."""
    rng = np.random.default_rng(12)
    K, V = 4, 1000
    logits = rng.standard_normal((K + 1, V)) * 2
    draft = logits + rng.standard_normal((K + 1, V)) * 0.5
    p = scipy.special.softmax(draft, axis=1)
    q = scipy.special.softmax(logits, axis=1)
    alpha = np.minimum(p, q).sum(axis=1)
    closed = sum(np.prod(alpha[:k + 1]) for k in range(K))
    par = W.chain_tree(K + 1)
    n = 4000
    tot = 0
    cdf = np.cumsum(p, axis=1)
    for _ in range(n):
        tok = np.zeros(K + 1, dtype=np.int64)
        for i in range(1, K + 1):
            tok[i] = min(np.searchsorted(cdf[i - 1], rng.random() * cdf[i - 1, -1], "right"), V - 1)
        res = OV.verify_walk(tok, par, list(rng.random(K + 1)), lambda j: q[j], lambda j: p[j])
        tot += len(res["path"])
    mean = tot / n
    # variance of the accept length is at most K^2 / 4
    assert abs(mean - closed) < 4 * (K / 2) / np.sqrt(n)


# ----------------------------------------------------------------------------------------------
# near-tie accounting: the margins that decide which sequences the GPU comparison skips
# ----------------------------------------------------------------------------------------------
# The accept test of a child is r * p < q (survey explainer, Formal Definition, 検証フェーズ:
# r < min(1, q / p)); the bonus is y = min{y : C(y) > u S}.  A decision's margin is how far its
# uniform may move before the decision changes: |r - q / p| for a test (q itself when p = 0, where
# no r changes it), and the distance of u from the nearer CDF boundary of y, in units of S, for
# the draw.  The pins below use hand-derived rationals and the defining property (a move smaller
# than the margin keeps the outcome, a slightly larger one towards the boundary changes it).
EPS = F(1, 2**40)


def _accept(r, qx, px):
    return r * px < qx


def test_decision_margin_hand_values():
    assert OV.decision_margin(F(1, 2), F(3, 10), F(1, 2)) == F(1, 10)     # q/p = 3/5
    assert OV.decision_margin(F(9, 10), F(1, 5), F(1, 10)) == F(11, 10)   # q/p = 2 (> 1)
    assert OV.decision_margin(F(1, 4), F(1, 8), F(1, 2)) == F(0)          # on the boundary
    assert OV.decision_margin(F(1, 3), F(3, 7), F(0)) == F(3, 7)          # p = 0: q
    assert OV.decision_margin(F(1, 3), F(0), F(0)) == F(0)


@pytest.mark.parametrize("seed", range(4))
def test_decision_margin_is_the_flip_distance(seed):
    rng = np.random.default_rng(seed)
    for _ in range(200):
        r = F(int(rng.integers(0, 2**24)), 2**24)
        px = F(int(rng.integers(1, 1000)), 1000)
        qx = F(int(rng.integers(0, 1000)), 1000)
        m = OV.decision_margin(r, qx, px)
        d = _accept(r, qx, px)
        assert m >= 0
        for s in (1, -1):                      # a smaller move keeps the decision
            assert _accept(r + s * m * (1 - EPS), qx, px) == d
        if m > 0:                              # a slightly larger move towards q/p flips it
            toward = 1 if qx / px > r else -1
            assert _accept(r + toward * m * (1 + EPS), qx, px) != d
        # p = 0: no r changes the decision; q moved by its margin (to 0) does
        assert _accept(r, qx, F(0)) == (qx > 0)
        assert _accept(r, qx - OV.decision_margin(r, qx, F(0)), F(0)) is False


def test_inverse_cdf_gap_hand_values():
    w = np.array([F(1), F(2), F(3), F(4)], dtype=object)       # S = 10, C = 1, 3, 6, 10
    assert OV.inverse_cdf(w, F(7, 20)) == (2, F(1, 20))         # uS = 7/2: lower 3, upper 6
    assert OV.inverse_cdf(w, F(1, 20)) == (0, F(1, 20))         # uS = 1/2: lower 0, upper 1
    assert OV.inverse_cdf(w, F(1, 2)) == (2, F(1, 10))          # uS = 5: 1 below C(2) = 6
    assert OV.inverse_cdf(w, F(3, 10)) == (2, F(0))             # uS = C(1): y = 2, on the boundary
    z = np.array([F(1), F(0), F(3)], dtype=object)              # zero weight: C = 1, 1, 4
    assert OV.inverse_cdf(z, F(1, 2)) == (2, F(1, 4))           # uS = 2: lower C(1) = 1, S = 4


@pytest.mark.parametrize("seed", range(4))
def test_inverse_cdf_gap_is_the_flip_distance(seed):
    rng = np.random.default_rng(100 + seed)
    for _ in range(200):
        V = int(rng.integers(2, 9))
        w = np.array([F(int(x)) for x in rng.integers(1, 50, size=V)], dtype=object)
        S = w.sum()
        u = F(int(rng.integers(0, 2**24)), 2**24)
        y, gap = OV.inverse_cdf(w, u)
        assert gap >= 0
        for s in (1, -1):
            v = u + s * gap * (1 - EPS)
            if 0 <= v < 1:
                assert OV.inverse_cdf(w, v)[0] == y
        C = np.cumsum(w)
        lower = C[y - 1] if y > 0 else F(0)
        # the nearer boundary; its crossing changes y unless it is the total (u -> 1)
        if u * S - lower <= C[y] - u * S:
            if gap > 0 and y > 0:
                assert OV.inverse_cdf(w, u - gap * (1 + EPS))[0] == y - 1
        elif C[y] < S:
            assert OV.inverse_cdf(w, u + gap * (1 + EPS))[0] == y + 1


def _outcome(tokens, parent, unif, q_of, p_of):
    res = OV.verify_walk(tokens, parent, unif, q_of, p_of)
    return tuple(res["path"]), res["bonus"], res


@pytest.mark.parametrize("name", sorted(TREES))
@pytest.mark.parametrize("seed", range(3))
def test_walk_min_margin_is_smallest_flip_of_any_uniform(name, seed):
    """min(margins) of a walk: no single uniform moved by less changes the path or the bonus, and
    some uniform moved by slightly more towards its boundary does.  A test uniform moves over the
    reals (the test r * p < q is defined there: with q / p > 1 the margin is the distance to a
    ratio that fp32 rounding could bring below r); the draw's u stays in [0, 1).  The draws avoid
    p = 0; a draw whose nearer boundary is 0 or the total S is skipped, because no u in [0, 1)
    crosses it there (the margin is conservative by construction)."""
    parent = np.array(TREES[name])
    V = 5
    rng = np.random.default_rng(7 * seed + len(name))
    depth = _depth(parent)
    qtab, ptab = {}, {}
    for L in range(depth + 1):
        for s in itertools.product(range(V), repeat=L):
            qtab[s] = _rand_dist(rng, V)
            ptab[s] = _rand_dist(rng, V, zeros=False)
    checked = 0
    for trial in range(30):
        tokens = np.array([0] + [int(x) for x in rng.integers(0, V, size=len(parent) - 1)])

        def q_of(j, _t=tokens):
            return qtab[_path_tokens(parent, _t, j)]

        def p_of(j, _t=tokens):
            return ptab[_path_tokens(parent, _t, j)]

        unif = [F(int(x), 2**20) for x in rng.integers(0, 2**20, size=len(parent))]
        path, bonus, res = _outcome(tokens, parent, unif, q_of, p_of)
        m = min(res["margins"])
        used = sorted(res["tests"]) + [0]        # the uniforms the walk read
        for k in used:
            for s in (1, -1):
                v = list(unif)
                v[k] = unif[k] + s * m * (1 - EPS)
                if k > 0 or 0 <= v[k] < 1:
                    assert _outcome(tokens, parent, v, q_of, p_of)[:2] == (path, bonus), (k, s)
        w = res["terminal"]
        S = w.sum()
        C = np.cumsum(w)
        lower, upper = (C[bonus - 1] if bonus else F(0)), C[bonus]
        near = lower if unif[0] * S - lower <= upper - unif[0] * S else upper
        if m == 0 or (m == res["margins"][-1] and near in (0, S)):
            continue          # the draw's nearer boundary is an end of [0, S]: nothing flips
        flipped = False
        for k in used:
            for s in (1, -1):
                v = list(unif)
                v[k] = unif[k] + s * m * (1 + EPS)
                if (k > 0 or 0 <= v[k] < 1) and _outcome(tokens, parent, v, q_of, p_of)[:2] != (path, bonus):
                    flipped = True
        assert flipped, (trial, m)
        checked += 1
    assert checked >= 10


def test_batched_min_margin_and_near_tie_flag():
    """tree_verify reports the walk's smallest margin per sequence and flags it below 1e-6: a
    uniform placed 1e-9 from its child's q/p is a near tie, the same draw 0.25 away is not."""
    V, N = 4, 3
    parent = np.array([[-1, 0, 0]])
    logits = np.log(np.array([[[0.4, 0.3, 0.2, 0.1]] * N]))
    probs = np.array([[[0.1, 0.2, 0.3, 0.4]] * N])
    tokens = np.array([[0, 3, 1]])
    q = OV.target_distribution(logits[0, 0], 1.0)
    ratio = q[3] / probs[0, 0, 3]                               # 0.25
    for off, near in ((1e-9, True), (0.25, False)):
        unif = np.array([[0.5, ratio + off, 0.9]])
        out = OV.tree_verify(logits, probs, tokens, parent, unif, 1.0)
        assert bool(out["near_tie"][0]) == near
        assert out["min_margin"][0] <= off + 1e-12
