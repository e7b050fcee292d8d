"""Verification of small problems without per-child q: the walk follows the nodes' hand-over
words as they finish, and nodes still in their residual rounds stop once the walk has ended.

Its results must equal the every-node form's (per-child q requested: every node completes and
the last one walks) bit for bit, and the oracle's outside near ties; a CUDA graph replayed with
new inputs (same call generation) must give each replay's own results; a non-finite row flags
the sequence only when the walk depends on it.
"""
import numpy as np
import pytest

from speculative_decoding_token_spec_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

KEYS = ("accept_len", "accepted_tokens", "bonus", "accepted_nodes", "status")


@pytest.fixture(scope="module")
def dev(cuda_lib):
    import torch
    return torch.device("cuda:0")


def _small(case):
    B, N, V = case.target_logits.shape
    return B * N * V * 4 <= (64 << 20)


def _check(case, dev, max_near=None):
    assert _small(case)
    got = P.run_verify_gpu(case, dev, want_child_q=False)
    every = P.run_verify_gpu(case, dev, want_child_q=True)
    for k in KEYS:
        np.testing.assert_array_equal(got[k], every[k], err_msg=k)
    ref = P.oracle_verify(case, with_table=False)
    stats = P.compare_verify(got, ref, case, check_child_q=False)
    B = case.target_logits.shape[0]
    assert stats["near_ties"] <= (max_near if max_near is not None else max(1, B // 8)), stats
    return got


@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
def test_eagle_tree_single_and_batched(dev, T):
    for B, seeds in ((1, range(6)), (8, range(2))):
        cfg = W.config("eagle_vicuna7b", B=B)
        for seed in seeds:
            _check(W.make_verify_case(cfg, T, seed=100 + seed), dev)


@pytest.mark.parametrize("N", [10, 40, 60])
def test_stress_shapes(dev, N):
    """Tree sizes, temperatures and draft noise of the stress sweep at batch 8."""
    tree = "chain" if N == 10 else "static"
    for T in (0.0, 0.5, 1.0, 1.5):
        for sd in (0.25, 1.0, 3.0):
            cfg = W.config("stress", B=8, N=N, tree=tree)
            _check(W.make_verify_case(cfg, T, seed=int(T * 10 + sd * 100) + 7, sigma_d=sd), dev,
                   max_near=2)


def test_star_tree_long_rounds(dev):
    """One node with 40 children (up to 39 residual rounds): the node that stops early and the
    node the walk ends at are the same node, so nothing may stop before the walk is done."""
    N = 41
    par = np.array([[-1] + [0] * (N - 1)] * 3, dtype=np.int32)
    cfg = W.config("eagle_vicuna7b", B=3, N=N, V=2000)
    for sd in (0.5, 3.0):
        _check(W.make_verify_case(cfg, 1.0, seed=9, sigma_d=sd, tree_parent=par), dev)


def test_two_level_stars(dev):
    """The root's children each have many children: siblings off the walk run many rounds and
    stop when the walk has ended."""
    K = 7
    par = [-1] + [0] * K
    for c in range(1, K + 1):
        par += [c] * K
    N = len(par)
    parr = np.array([par] * 4, dtype=np.int32)
    cfg = W.config("eagle_vicuna7b", B=4, N=N, V=3000)
    for T, sd in ((1.0, 3.0), (0.7, 1.0), (1.5, 3.0)):
        _check(W.make_verify_case(cfg, T, seed=5, sigma_d=sd, tree_parent=parr), dev)


def test_root_only_and_max_nodes(dev):
    for T in (0.0, 1.0):
        got = _check(W.make_verify_case(W.config("eagle_vicuna7b", B=4, N=1, V=5000), T, seed=2),
                     dev)
        assert (got["accept_len"] == 0).all()
        _check(W.make_verify_case(W.config("eagle_vicuna7b", B=2, N=64, depth=7, width=10,
                                           V=4000), T, seed=5), dev)


def test_nonfinite_rows_on_and_off_the_walk(dev):
    cfg = W.config("eagle_vicuna7b", B=1, V=4000)
    base = W.make_verify_case(cfg, 1.0, seed=12)
    clean = P.run_verify_gpu(base, dev, want_child_q=False)
    assert clean["status"][0] == 0
    acc = [int(x) for x in clean["accepted_nodes"][0] if x >= 0]
    on = {0} | set(acc)
    par = base.tree_parent[0]
    internal = [i for i in range(1, 60) if (par == i).any()]
    off = [i for i in internal if i not in on]
    assert off
    # an internal node off the walk: nothing the walk depends on, so the same results, no flag
    case = W.make_verify_case(cfg, 1.0, seed=12)
    case.target_logits[0, off[0], 5] = np.nan
    got = P.run_verify_gpu(case, dev, want_child_q=False)
    for k in KEYS:
        np.testing.assert_array_equal(got[k], clean[k], err_msg=k)
    # every node processed in full (per-child q asked for): the row is read and flagged
    every = P.run_verify_gpu(case, dev, want_child_q=True)
    assert every["status"][0] == 8 and every["accept_len"][0] == -1
    # the node where the walk stops: flagged, no outputs
    terminal = acc[-1] if acc else 0
    for node in (0, terminal):
        case = W.make_verify_case(cfg, 1.0, seed=12)
        case.target_logits[0, node, 7] = np.inf
        got = P.run_verify_gpu(case, dev, want_child_q=False)
        assert got["status"][0] == 8, node
        assert got["accept_len"][0] == -1 and got["bonus"][0] == -1
        assert (got["accepted_tokens"][0] == -1).all()


def test_cuda_graph_replays_with_new_inputs(dev):
    """Replays of one captured call keep the call's generation: each must start from cleared
    hand-over words and give the same results as a direct call on the same inputs."""
    import torch
    import speculative_decoding_token_spec_gb300 as st
    cfg = W.config("eagle_vicuna7b", B=4, V=8000)
    cases = [W.make_verify_case(cfg, 1.0, seed=40 + i) for i in range(6)]
    t = lambda a: P.dev_tensor(a, dev)  # noqa: E731
    bufs = [t(cases[0].target_logits), t(cases[0].draft_probs), t(cases[0].tree_tokens),
            t(cases[0].tree_parent), t(cases[0].uniforms)]
    B, N, V = cases[0].target_logits.shape
    ws = torch.empty((st.spec_tree_verify_workspace(B, N, V),), dtype=torch.uint8, device=dev)
    st.spec_tree_verify(*bufs, 1.0, workspace=ws)  # warm-up outside the capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            out = st.spec_tree_verify(*bufs, 1.0, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    for case in cases + cases[:2]:
        for dst, src in zip(bufs, (case.target_logits, case.draft_probs, case.tree_tokens,
                                   case.tree_parent, case.uniforms)):
            dst.copy_(t(src))
        g.replay()
        torch.cuda.synchronize()
        got = {k: v.cpu().numpy() for k, v in out.items()}
        ref = P.run_verify_gpu(case, dev, want_child_q=False)
        for k in ("accept_len", "accepted_tokens", "bonus", "accepted_nodes"):
            np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
        assert (got["status"] == 0).all()
