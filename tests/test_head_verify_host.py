"""Verification from the LM head's statistics: CPU checks (no GPU).

* The composed oracle (oracle/lmhead.py: tree_verify_from_head) reduces to oracle/verify.py's
  tree_verify when the head is the identity and the hidden states are the logits themselves.
* The lattice inputs of make_head_verify_case give logits that are exact in float32 whatever the
  order of the sums (integer products, |sum| far below 2^24 units): an int64 matrix product equals
  the oracle's float64 one, and a float32 round trip changes nothing.
* The decomposition the kernels use -- accept first children from (m, S, l_x~) alone, and process
  the node where that stops from its full row (every child re-tested, residual rounds, bonus) --
  gives tree_verify's results, written here as a plain loop over the oracle's building blocks.
* tree_depth against a brute-force ancestor count.
"""
import numpy as np
import pytest

from oracle import lmhead as OL
from oracle import verify as OV
from speculative_decoding_token_spec_gb300 import workloads as W


def _bf16_exact(x):
    b = W.bf16_bits(np.asarray(x, np.float32))
    assert np.array_equal(W.bf16_to_f64(b), np.asarray(x, np.float64))
    return b


@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
def test_identity_head_reduces_to_tree_verify(T):
    rng = np.random.default_rng(4)
    B, N, V = 3, 9, 40
    par = np.stack([W.make_tree(np.random.default_rng(10 + b), N, 4, 3) for b in range(B)])
    lg = rng.integers(-24, 25, size=(B, N, V)) / 8.0  # exact in bf16
    hidden = W.bf16_to_f64(_bf16_exact(lg))
    head = np.eye(V)
    dp = rng.random((B, N, V))
    dp /= dp.sum(axis=-1, keepdims=True)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    uni = rng.integers(0, 1 << 24, size=(B, N)) / float(1 << 24)
    got = OL.tree_verify_from_head(hidden, head, dp, tok, par, uni, T)
    ref = OV.tree_verify(lg, dp, tok, par, uni, T)
    for k in ("accept_len", "accepted_nodes", "accepted_tokens", "bonus", "status"):
        assert np.array_equal(got[k], ref[k]), k
    assert np.array_equal(got["min_margin"], ref["min_margin"])


@pytest.mark.parametrize("H", [64, 512])
def test_lattice_logits_exact_in_float32(H):
    case = W.make_head_verify_case(W.config("eagle_vicuna7b", B=2, N=8, V=300), H, 1.0, seed=3)
    h = W.bf16_to_f64(case.hidden).reshape(-1, H)
    w = W.bf16_to_f64(case.head)
    lg = OL.logits(h, w)
    ha = np.round(h * 4).astype(np.int64)
    s = int(np.round(-np.log2(np.min(np.abs(w[w != 0])))))
    wa = np.round(w * 2.0 ** s).astype(np.int64)
    assert np.array_equal(ha / 4.0, h) and np.array_equal(wa / 2.0 ** s, w)
    assert np.abs(ha).max() <= 3 and np.abs(wa).max() <= 7
    exact = (ha @ wa.T).astype(np.float64) * 2.0 ** -(2 + s)
    assert np.array_equal(lg, exact)
    assert np.abs(ha @ wa.T).max() < 2 ** 24
    assert np.array_equal(lg.astype(np.float32).astype(np.float64), lg)


def _decomposed_walk(lg, dp, tok, par, uni, T):
    """First children accepted from (m, S, l_x~); the stop node from its full row."""
    kids = OV.children(par)
    c, path = 0, []
    while True:
        ks = kids[c]
        if ks:
            row = np.asarray(lg[c], np.float64)
            m = row.max()
            S = np.exp((row - m) / T).sum()
            x = int(tok[ks[0]])
            if uni[ks[0]] * dp[c][x] * S < np.exp((row[x] - m) / T):
                path.append(ks[0])
                c = ks[0]
                continue
        # the stop node: every child tested again from the full row, as tree_verify does
        q = OV.target_distribution(lg[c], T)
        pos, _, qf = OV.sibling_tests(q, np.asarray(dp[c], np.float64),
                                      [int(tok[k]) for k in ks], [uni[k] for k in ks])
        if pos is None:
            return path, OV.inverse_cdf(qf, uni[0])[0]
        c = ks[pos]
        path.append(c)


@pytest.mark.parametrize("T", [0.7, 1.0])
def test_decomposition_equals_the_definition(T):
    mism = near = 0
    for seed in range(6):
        case = W.make_head_verify_case(W.config("eagle_vicuna7b", B=4, V=400), 64, T, seed=seed,
                                       sigma_d=0.7)
        B, N, H = case.hidden.shape
        lg = OL.logits(W.bf16_to_f64(case.hidden).reshape(B * N, H),
                       W.bf16_to_f64(case.head)).reshape(B, N, -1)
        ref = OV.tree_verify(lg, case.draft_probs, case.tree_tokens, case.tree_parent,
                             case.uniforms, T)
        for b in range(B):
            if ref["near_tie"][b]:
                near += 1
                continue
            path, bonus = _decomposed_walk(lg[b], case.draft_probs[b].astype(np.float64),
                                           case.tree_tokens[b], case.tree_parent[b],
                                           [float(u) for u in case.uniforms[b]], T)
            n = int(ref["accept_len"][b])
            ok = path == list(ref["accepted_nodes"][b, :n]) and bonus == ref["bonus"][b]
            mism += 0 if ok else 1
    assert mism == 0 and near <= 2


def test_tree_depth_brute_force():
    for seed in range(5):
        par = W.make_tree(np.random.default_rng(seed), 40, 6, 10)
        depths = []
        for i in range(len(par)):
            d, k = 0, i
            while par[k] >= 0:
                k = int(par[k])
                d += 1
            depths.append(d)
        assert W.tree_depth(par) == max(depths)
    assert W.tree_depth(W.chain_tree(7)) == 6
    assert W.tree_depth(np.array([-1], np.int32)) == 0
