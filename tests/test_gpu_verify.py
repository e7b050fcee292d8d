"""GPU parity of spec_tree_verify against the fp64 oracle (through the C ABI).

Integer outputs (accept lengths, accepted tokens / nodes, bonus tokens, status) are bit-exact
except in sequences whose fp64 decision margin |r - q/p| or CDF gap is below 1e-6; those are
counted and printed.  The q used in every child's test matches to 1e-5 absolute.
"""
import numpy as np
import pytest

from speculative_decoding_token_spec_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_lib):
    import torch
    return torch.device("cuda:0")


def _check(case, dev, want_child_q=True, max_near=None):
    got = P.run_verify_gpu(case, dev, want_child_q=want_child_q)
    ref = P.oracle_verify(case, with_table=want_child_q)
    stats = P.compare_verify(got, ref, case, check_child_q=want_child_q)
    B = case.target_logits.shape[0]
    if max_near is None:
        max_near = max(1, B // 8)
    assert stats["near_ties"] <= max_near, stats
    print(f"B={B} T={case.temperature}: {stats}, mean accept "
          f"{np.mean(got['accept_len'][got['accept_len'] >= 0]):.2f}")
    return got, ref


@pytest.mark.parametrize("T", [1.0, 0.0, 0.3])
def test_tiny_chain(dev, T):
    cfg = W.config("tiny")
    for seed in range(6):
        _check(W.make_verify_case(cfg, T, seed=seed), dev)


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_eagle_static_tree_vicuna7b(dev, T):
    cfg = W.config("eagle_vicuna7b")
    for seed in range(4):
        _check(W.make_verify_case(cfg, T, seed=seed), dev)


def test_eagle_tree_batched_many_seeds(dev):
    """Config-2 tree and vocabulary, 48 independently seeded sequences in one call."""
    cfg = W.config("eagle_vicuna7b", B=48)
    for T in (1.0, 0.0):
        _check(W.make_verify_case(cfg, T, seed=11), dev)


@pytest.mark.parametrize("child_q", [True, False])  # every internal node / the path only
def test_llama3_8b_gqa_vocab_128k(dev, child_q):
    cfg = W.config("llama3_8b_gqa")
    _check(W.make_verify_case(cfg, 0.7, seed=0), dev, want_child_q=child_q)


@pytest.mark.parametrize("child_q", [True, False])
def test_llama70b_longctx_vocab_128k(dev, child_q):
    cfg = W.config("llama70b_longctx")
    _check(W.make_verify_case(cfg, 1.0, seed=0), dev, want_child_q=child_q)


@pytest.mark.parametrize("N", [10, 40, 60])
def test_stress_sweep(dev, N):
    """Tree size x temperature x draft noise (sets the acceptance rate); reduced batch."""
    tree = "chain" if N == 10 else "static"
    for T in (0.0, 0.5, 1.0, 1.5):
        for sd in (0.25, 1.0, 3.0):
            cfg = W.config("stress", B=6, N=N, tree=tree)
            _check(W.make_verify_case(cfg, T, seed=int(T * 10 + sd * 100), sigma_d=sd), dev,
                   want_child_q=(T == 1.0))


def test_stress_full_batch(dev):
    """Full batch of the stress shape (64 sequences, 60-node trees) at one setting."""
    cfg = W.config("stress")
    _check(W.make_verify_case(cfg, 1.0, seed=3, sigma_d=1.0), dev, want_child_q=False, max_near=4)


@pytest.mark.parametrize("T,sd", [(0.0, 1.0), (0.5, 0.25), (1.5, 3.0), (1.0, 0.25)])
def test_path_form_full_batch(dev, T, sd):
    """Large problems without per-child q take the path-only form (one cluster per sequence,
    only the nodes the walk reaches): full stress batch over temperatures and draft noise (long
    and short accepted paths), chains included."""
    for N, tree in ((60, "static"), (10, "chain")):
        cfg = W.config("stress", N=N, tree=tree)
        _check(W.make_verify_case(cfg, T, seed=int(T * 10 + sd * 100) + N, sigma_d=sd), dev,
               want_child_q=False, max_near=4)


def test_path_form_reads_only_the_walk(dev):
    """Path-only form: NaN in a row the walk never reaches leaves the sequence alone (its result is
    the oracle's); NaN in the root row (always read) flags it.  The all-nodes form, taken when
    per-child q is requested, reads every internal row and flags both."""
    cfg = W.config("eagle_vicuna7b", B=8, N=60, V=40000)  # 77 MB of logits: a large problem
    case = W.make_verify_case(cfg, 1.0, seed=31)
    ref = P.oracle_verify(case, with_table=False)
    b_off = next(b for b in range(1, 8) if not ref["near_tie"][b])
    walk = set(int(x) for x in ref["accepted_nodes"][b_off] if x >= 0) | {0}
    internal = set(int(p) for p in case.tree_parent[b_off, 1:])
    off = min(internal - walk)
    case.target_logits[b_off, off, 5] = np.nan
    case.target_logits[0, 0, 9] = np.nan
    got = P.run_verify_gpu(case, dev, want_child_q=False)
    assert got["status"][0] == 8 and got["accept_len"][0] == -1
    assert got["status"][b_off] == 0
    assert got["accept_len"][b_off] == ref["accept_len"][b_off]
    assert got["bonus"][b_off] == ref["bonus"][b_off]
    np.testing.assert_array_equal(got["accepted_nodes"][b_off], ref["accepted_nodes"][b_off])
    every = P.run_verify_gpu(case, dev, want_child_q=True)
    assert every["status"][0] == 8 and every["status"][b_off] == 8


# ------------------------------------------------------------------------------------------------
# edge cases
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("V", [1, 3, 1001, 32003])
def test_ragged_vocab_and_unaligned_rows(dev, V):
    cfg = W.config("eagle_vicuna7b", B=3, V=V, N=12, depth=3, width=5)
    for T in (0.0, 1.0):
        _check(W.make_verify_case(cfg, T, seed=V), dev)


def test_root_only_tree(dev):
    """N = 1: nothing to verify, the bonus is drawn from the root's target distribution."""
    cfg = W.config("eagle_vicuna7b", B=4, N=1, V=5000)
    for T in (0.0, 1.0):
        got, ref = _check(W.make_verify_case(cfg, T, seed=2), dev)
        assert (got["accept_len"] == 0).all()


def test_max_nodes_64(dev):
    cfg = W.config("eagle_vicuna7b", B=2, N=64, depth=7, width=10, V=4000)
    for T in (0.0, 1.0):
        _check(W.make_verify_case(cfg, T, seed=5), dev)


def test_star_tree_many_siblings(dev):
    """One node with 40 children: up to 39 residual rounds at a single node."""
    N = 41
    par = np.array([[-1] + [0] * (N - 1)] * 3, dtype=np.int32)
    cfg = W.config("eagle_vicuna7b", B=3, N=N, V=2000)
    for sd in (0.5, 3.0):
        _check(W.make_verify_case(cfg, 1.0, seed=9, sigma_d=sd, tree_parent=par), dev)


def test_bad_trees_tokens_and_nonfinite(dev):
    cfg = W.config("eagle_vicuna7b", B=5, N=10, depth=3, width=4, V=3000)
    case = W.make_verify_case(cfg, 1.0, seed=1)
    case.tree_parent[1, 4] = 4            # self-parent
    case.tree_parent[2, 0] = 0            # root with a parent
    case.tree_tokens[3, 5] = cfg.V        # token out of range
    case.target_logits[4, 0, 17] = np.nan  # NaN in the root row (always read)
    got = P.run_verify_gpu(case, dev)
    assert got["status"][0] == 0
    assert got["status"][1] == 1 and got["status"][2] == 1
    assert got["status"][3] == 4
    assert got["status"][4] == 8
    for b in (1, 2, 3, 4):
        assert got["accept_len"][b] == -1 and got["bonus"][b] == -1
        assert (got["accepted_tokens"][b] == -1).all()
    ref = P.oracle_verify(W.VerifyCase(case.target_logits[:1], case.draft_probs[:1],
                                       case.tree_tokens[:1], case.tree_parent[:1],
                                       case.uniforms[:1], 1.0))
    if not ref["near_tie"][0]:
        assert got["bonus"][0] == ref["bonus"][0] and got["accept_len"][0] == ref["accept_len"][0]


def test_greedy_ignores_draft_probs(dev):
    cfg = W.config("eagle_vicuna7b", B=4, N=20, depth=4, width=6, V=3000)
    case = W.make_verify_case(cfg, 0.0, seed=4)
    got = P.run_verify_gpu(case, dev, pass_probs=False)
    ref = P.oracle_verify(case)
    P.compare_verify(got, ref, case)


def test_argument_errors(dev):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    cfg = W.config("tiny")
    case = W.make_verify_case(cfg, 1.0)
    t = lambda a: P.dev_tensor(a, dev)  # noqa: E731
    with pytest.raises(st.SpecError):
        st.spec_tree_verify(t(case.target_logits), t(case.draft_probs), t(case.tree_tokens),
                            t(case.tree_parent), t(case.uniforms), -1.0)
    with pytest.raises(st.SpecError):
        st.spec_tree_verify(t(case.target_logits), None, t(case.tree_tokens),
                            t(case.tree_parent), t(case.uniforms), 1.0)
    torch.cuda.synchronize()


def test_deterministic_repeat(dev):
    cfg = W.config("eagle_vicuna7b", B=8)
    case = W.make_verify_case(cfg, 1.0, seed=21)
    a = P.run_verify_gpu(case, dev)
    b = P.run_verify_gpu(case, dev)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


def test_acceptance_statistics_chain(dev):
    """Mean accepted length over many uniforms matches the closed form sum_k prod alpha_j."""
    import torch
    import speculative_decoding_token_spec_gb300 as st
    K, V, B = 4, 500, 4096
    rng = np.random.default_rng(77)
    logits = (rng.standard_normal((K + 1, V)) * 2).astype(np.float32)
    draft = logits + (rng.standard_normal((K + 1, V)) * 0.7).astype(np.float32)
    p64 = np.exp(draft.astype(np.float64) - draft.max(1, keepdims=True))
    p64 /= p64.sum(1, keepdims=True)
    q64 = np.exp(logits.astype(np.float64) - logits.max(1, keepdims=True))
    q64 /= q64.sum(1, keepdims=True)
    alpha = np.minimum(p64, q64).sum(1)
    closed = sum(np.prod(alpha[:k + 1]) for k in range(K))
    cdf = np.cumsum(p64, axis=1)
    toks = np.zeros((B, K + 1), np.int32)
    for i in range(1, K + 1):
        u = rng.random(B) * cdf[i - 1, -1]
        toks[:, i] = np.minimum(np.searchsorted(cdf[i - 1], u, side="right"), V - 1)
    case = W.VerifyCase(np.broadcast_to(logits, (B, K + 1, V)).copy(),
                        np.broadcast_to(p64.astype(np.float32), (B, K + 1, V)).copy(),
                        toks, np.broadcast_to(W.chain_tree(K + 1), (B, K + 1)).copy(),
                        (rng.integers(0, 1 << 24, (B, K + 1)) / float(1 << 24)).astype(np.float32),
                        1.0)
    got = P.run_verify_gpu(case, dev, want_child_q=False)
    mean = got["accept_len"].mean()
    assert abs(mean - closed) < 4 * (K / 2) / np.sqrt(B), (mean, closed)
    # first emitted token ~ q_root: chi-square over the 20 most likely tokens + the rest
    first = np.where(got["accept_len"] > 0, toks[:, 1], got["bonus"])
    top = np.argsort(-q64[0])[:20]
    obs = np.array([(first == y).sum() for y in top] + [(~np.isin(first, top)).sum()])
    exp = np.array(list(q64[0, top] * B) + [(1 - q64[0, top].sum()) * B])
    chi2 = ((obs - exp) ** 2 / exp).sum()
    assert chi2 < 60, chi2   # 20 dof: p ~ 1e-5
    torch.cuda.synchronize()
    del st
