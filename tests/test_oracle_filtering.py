"""Pins for the top-k / top-p filtering oracle (CPU only).

* Brute force: the kept set equals the smallest prefix of the tokens sorted by logit (whole tie
  groups at a time) whose count reaches k, resp. whose probability reaches top_p -- written as a
  loop over tie groups, not as the oracle's mass-of-greater-tokens rule.
* Nucleus properties on random rows: kept mass >= top_p, and dropping the least probable kept tie
  group leaves < top_p (minimality).
* Top-k = 1 at T > 0 makes the target one-hot at the argmax, so filtered verification must walk
  exactly like greedy (T = 0) verification: same accepted path, same bonus (through the verify
  oracle, on generated trees).
* Off switches: top_k <= 0 or >= V, top_p >= 1 and T = 0 leave the logits unchanged.
"""
import numpy as np
import pytest

from oracle import filtering as OF
from oracle import verify as OV
from speculative_decoding_token_spec_gb300 import workloads as W


def _groups_desc(l):
    """Tie groups of the logits, largest first: list of index arrays."""
    vals = np.unique(l)[::-1]
    return [np.flatnonzero(l == v) for v in vals]


def _brute_keep(l, T, k, p):
    V = len(l)
    keep = np.ones(V, dtype=bool)
    if T <= 0:
        return keep
    if 0 < k < V:
        kk = np.zeros(V, dtype=bool)
        n = 0
        for g in _groups_desc(l):
            kk[g] = True
            n += len(g)
            if n >= k:
                break
        keep = kk
    if p < 1.0:
        q = np.zeros(V)
        q[keep] = np.exp((l[keep] - l[keep].max()) / T)
        q /= q.sum()
        kp = np.zeros(V, dtype=bool)
        mass = 0.0
        for g in _groups_desc(np.where(keep, l, -np.inf)):
            if mass >= p:
                break
            kp[g] = True
            mass += q[g].sum()
        keep = keep & kp
    return keep


@pytest.mark.parametrize("seed", range(12))
def test_keep_mask_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(2, 40))
    l = np.round(rng.standard_normal(V) * 2, 1)        # rounding makes ties frequent
    for T in (0.5, 1.0, 2.0):
        for k in (0, 1, 2, 5, V - 1, V, V + 3):
            for p in (0.05, 0.3, 0.5, 0.9, 0.999, 1.0):
                got = OF.keep_mask(l, T, k, p)
                want = _brute_keep(l, T, k, p)
                assert np.array_equal(got, want), (V, T, k, p)


@pytest.mark.parametrize("seed", range(6))
def test_nucleus_mass_and_minimality(seed):
    rng = np.random.default_rng(50 + seed)
    l = rng.standard_normal(300) * 3
    T, p = 0.8, float(rng.uniform(0.1, 0.95))
    keep = OF.keep_mask(l, T, 0, p)
    q = np.exp((l - l.max()) / T)
    q /= q.sum()
    assert q[keep].sum() >= p
    smallest = l[keep].min()
    assert q[keep & (l > smallest)].sum() < p


def test_off_switches():
    rng = np.random.default_rng(3)
    l = rng.standard_normal(50)
    for T, k, p in [(1.0, 0, 1.0), (1.0, 50, 1.0), (1.0, 80, 1.0), (0.0, 3, 0.2)]:
        assert np.array_equal(OF.filter_logits(l, T, k, p), l)


@pytest.mark.parametrize("seed", range(5))
def test_top_k_one_walks_like_greedy(seed):
    cfg = W.config("eagle_vicuna7b", B=4, N=24, depth=4, width=8, V=300)
    vc = W.make_verify_case(cfg, 1.0, seed=seed, sigma_d=0.5)
    filt = OF.filter_logits(vc.target_logits, 1.0, 1, 1.0)
    got = OV.tree_verify(filt, vc.draft_probs, vc.tree_tokens, vc.tree_parent, vc.uniforms, 1.0)
    ref = OV.tree_verify(vc.target_logits, None, vc.tree_tokens, vc.tree_parent, vc.uniforms, 0.0)
    assert np.array_equal(got["accept_len"], ref["accept_len"])
    assert np.array_equal(got["accepted_tokens"], ref["accepted_tokens"])
    assert np.array_equal(got["bonus"], ref["bonus"])


def test_top_p_margin_locates_the_boundaries():
    l = np.log(np.array([0.5, 0.3, 0.2]))
    # strictly-greater masses: 0, 0.5, 0.8
    assert OF.top_p_margin(l, 1.0, 0, 0.52) == pytest.approx(0.02)
    assert OF.top_p_margin(l, 1.0, 0, 0.79) == pytest.approx(0.01)
    assert OF.top_p_margin(l, 1.0, 0, 1.0) == np.inf
