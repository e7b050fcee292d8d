"""GPU parity of the dynamic tree construction (spec_tree_expand / spec_tree_finalize) against the
fp64 oracle, through the C ABI.

Exact: every level's frontier (tokens, parent slots), the tree (tokens, parents), each node's draft
row.  Node values within 1e-4 (fp32 arithmetic on the device).  Sequences where the oracle's values
come within 1e-4 of each other at a selection boundary (a frontier's K-th / (K+1)-th candidate, the
tree's (N-1)-th / N-th) are counted, not compared: the device's fp32 values may order them the
other way.  Exact ties (equal logits of one parent) are reproduced bit for bit and stay compared.
Special cases: K = 1 (the greedy chain), -inf entries, NaN rows (SPEC_ST_NONFINITE, the root
alone), an out-of-order level (SPEC_ST_BAD_TREE, state unchanged), and the built tree driving
greedy verification.
"""
import numpy as np
import pytest

from oracle import dyntree as OD
from oracle import verify as OV
from speculative_decoding_token_spec_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

VALUE_TOL = 1e-4


@pytest.fixture(scope="module")
def dev(cuda_lib):
    import torch
    return torch.device("cuda:0")


def _run(case, dev, N, levels=None):
    """All levels on the GPU; returns (per-level frontiers, finalize outputs) as numpy."""
    import torch
    import speculative_decoding_token_spec_gb300 as st
    B, K, D = case.draft_rows.shape[0], case.K, case.D
    ws = torch.empty(st.spec_tree_build_workspace(B, K, D), dtype=torch.uint8, device=dev)
    status = torch.zeros(B, dtype=torch.int32, device=dev)
    fronts = []
    for d in (levels or range(1, D + 1)):
        ft, fs, _ = st.spec_tree_expand(P.dev_tensor(case.level_rows(d), dev), K, D, d, ws,
                                        status=status)
        fronts.append((ft.cpu().numpy(), fs.cpu().numpy()))
    out = st.spec_tree_finalize(ws, P.dev_tensor(case.root_tokens, dev), K, D, N, status=status)
    torch.cuda.synchronize()
    return fronts, {k: v.cpu().numpy() for k, v in out.items()}, ws


def _oracle(case, N):
    """Per sequence: frontiers per level, the tree, and whether a boundary is a near tie."""
    B, K, D = case.draft_rows.shape[0], case.K, case.D
    res = []
    for b in range(B):
        tb = OD.TreeBuilder(K)
        fronts, near = [], False
        for d in range(1, D + 1):
            rows = case.level_rows(d)[b][: len(tb.frontier)]
            before = len(tb.token)
            fr = tb.expand(rows)
            fronts.append(([tb.token[c] for c in fr], [tb.order[c] // K for c in fr]))
            vals = sorted((tb.value[c] for c in range(before, len(tb.token))), reverse=True)
            if len(vals) > K:
                gap = vals[K - 1] - vals[K]
                near |= 0 < gap < VALUE_TOL
        out = tb.finalize(int(case.root_tokens[b]), N)
        allv = sorted(tb.value[1:], reverse=True)
        if len(allv) > N - 1 >= 1:
            gap = allv[N - 2] - allv[N - 1]
            near |= 0 < gap < VALUE_TOL
        res.append((fronts, out, near))
    return res


def _compare(case, dev, N, max_near=None):
    fronts, got, _ = _run(case, dev, N)
    ref = _oracle(case, N)
    B = case.draft_rows.shape[0]
    assert (got["status"] == 0).all(), got["status"]
    near = 0
    for b in range(B):
        rf, ro, is_near = ref[b]
        if is_near:
            near += 1
            continue
        for d, (tok, slot) in enumerate(rf):
            assert list(fronts[d][0][b, :len(tok)]) == tok, (b, d)
            assert list(fronts[d][1][b, :len(slot)]) == slot, (b, d)
        for k in ("tree_tokens", "tree_parent", "node_row"):
            assert np.array_equal(got[k][b], ro[k]), (b, k, got[k][b], ro[k])
        n = ro["n_nodes"]
        assert np.abs(got["node_value"][b, :n] - ro["node_value"][:n]).max() <= VALUE_TOL
        assert np.isnan(got["node_value"][b, n:]).all()
    if max_near is None:
        max_near = max(1, B // 8)
    assert near <= max_near, near
    print(f"B={B} K={case.K} D={case.D} V={case.draft_rows.shape[2]} N={N}: "
          f"{B - near} compared, {near} near ties")
    return got


@pytest.mark.parametrize("B,K,D,V,N,seed", [
    (4, 10, 6, 32000, 60, 0),     # EAGLE-2-like: top-10 expansion, depth 6, 60-node tree
    (3, 4, 3, 1000, 20, 1),
    (2, 16, 4, 128256, 64, 2),    # 128K vocabulary, widest frontier
    (5, 8, 8, 4096, 64, 3),       # pool of 1 + 8 + 7 * 64 = 457
    (4, 3, 5, 517, 30, 4),        # ragged vocabulary
    (16, 10, 6, 32000, 60, 5),    # batched
])
def test_matches_oracle(dev, B, K, D, V, N, seed):
    _compare(W.make_tree_build_case(B, K, D, V, seed=seed), dev, N)


def test_greedy_chain_k1(dev):
    case = W.make_tree_build_case(3, 1, 7, 3000, seed=6)
    got = _compare(case, dev, 8)
    for b in range(3):
        assert list(got["tree_parent"][b]) == [-1] + list(range(7))
        want = [int(np.argmax(case.level_rows(d)[b, 0])) for d in range(1, 8)]
        assert list(got["tree_tokens"][b, 1:]) == want


def test_ties_and_masked_entries(dev):
    """Logits on a coarse grid (equal logits within rows: exact ties, broken by token id and
    candidate order identically on both sides) and -inf entries (masked tokens)."""
    case = W.make_tree_build_case(4, 6, 4, 700, seed=7)
    case.draft_rows[:] = np.round(case.draft_rows)
    rng = np.random.default_rng(7)
    case.draft_rows[rng.random(case.draft_rows.shape) < 0.3] = -np.inf
    _compare(case, dev, 40)


def test_small_n_and_full_pool(dev):
    case = W.make_tree_build_case(3, 4, 3, 900, seed=8)
    _compare(case, dev, 1)                      # the root alone
    _compare(case, dev, 1 + 4 + 2 * 16)         # every candidate


def test_nonfinite_row_stops_the_construction(dev):
    case = W.make_tree_build_case(3, 4, 3, 600, seed=9)
    case.draft_rows[1, 1 + 4 + 2, 17] = np.nan     # level 3, frontier slot 2 of sequence 1
    case.draft_rows[2, 0, 5] = np.inf              # sequence 2's root row
    _, got, _ = _run(case, dev, 10)
    assert got["status"][0] == 0 and got["status"][1] == 8 and got["status"][2] == 8
    for b in (1, 2):
        assert got["tree_tokens"][b, 0] == case.root_tokens[b]
        assert (got["tree_parent"][b, 1:] == -1).all() and (got["tree_tokens"][b, 1:] == -1).all()
    ref = _oracle(W.TreeBuildCase(case.draft_rows[:1], case.root_tokens[:1], 4, 3), 10)
    if not ref[0][2]:
        assert np.array_equal(got["tree_parent"][0], ref[0][1]["tree_parent"])


def test_out_of_order_level_is_flagged_and_harmless(dev):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    case = W.make_tree_build_case(2, 3, 3, 400, seed=10)
    B, K, D = 2, 3, 3
    ws = torch.empty(st.spec_tree_build_workspace(B, K, D), dtype=torch.uint8, device=dev)
    st.spec_tree_expand(P.dev_tensor(case.level_rows(1), dev), K, D, 1, ws)
    _, _, bad = st.spec_tree_expand(P.dev_tensor(case.level_rows(3), dev), K, D, 3, ws)
    torch.cuda.synchronize()
    assert (bad.cpu().numpy() == 1).all()
    st.spec_tree_expand(P.dev_tensor(case.level_rows(2), dev), K, D, 2, ws)
    st.spec_tree_expand(P.dev_tensor(case.level_rows(3), dev), K, D, 3, ws)
    out = st.spec_tree_finalize(ws, P.dev_tensor(case.root_tokens, dev), K, D, 12)
    torch.cuda.synchronize()
    ref = _oracle(case, 12)
    for b in range(B):
        if not ref[b][2]:
            assert np.array_equal(out["tree_parent"][b].cpu().numpy(), ref[b][1]["tree_parent"])
            assert np.array_equal(out["tree_tokens"][b].cpu().numpy(), ref[b][1]["tree_tokens"])


def test_built_tree_drives_greedy_verification(dev):
    """End to end on the device: the constructed tree (tokens, parents) goes to spec_tree_verify at
    T = 0 with target logits for its nodes; the accepted path matches the oracle's on the same
    tree."""
    import torch
    import speculative_decoding_token_spec_gb300 as st
    B, K, D, V, N = 4, 6, 5, 2000, 40
    case = W.make_tree_build_case(B, K, D, V, seed=11)
    _, got, _ = _run(case, dev, N)
    tok, par = got["tree_tokens"], got["tree_parent"]
    rng = np.random.default_rng(11)
    target = (rng.standard_normal((B, N, V)) * 3).astype(np.float32)
    # make the target agree with the draft along some paths: favour each node's first child token
    for b in range(B):
        for j in range(1, N):
            if rng.random() < 0.7:
                target[b, par[b, j], tok[b, j]] += 12.0
    uni = np.zeros((B, N), np.float32)
    res = st.spec_tree_verify(P.dev_tensor(target, dev), None, torch.from_numpy(tok).to(dev),
                              torch.from_numpy(par).to(dev), P.dev_tensor(uni, dev), 0.0)
    torch.cuda.synchronize()
    ref = OV.tree_verify(target, None, tok, par, uni, 0.0)
    assert (res["status"].cpu().numpy() == 0).all()
    assert np.array_equal(res["accept_len"].cpu().numpy(), ref["accept_len"])
    assert np.array_equal(res["accepted_tokens"].cpu().numpy(), ref["accepted_tokens"])
    assert np.array_equal(res["bonus"].cpu().numpy(), ref["bonus"])
    assert ref["accept_len"].max() >= 1


def test_slow_exact_path_and_large_vocab(dev):
    """A tie group of 2560 entries held by five warps puts more than 2048 keys at or above the
    warp-best threshold (the exact per-thread path takes over); V = 150000 takes the one-CTA-per-
    row kernel."""
    case = W.make_tree_build_case(2, 10, 3, 32000, seed=12)
    y = np.arange(32000)
    case.draft_rows[:, :, (y < 8192) & (y % 512 < 160)] = np.float32(100.0)  # warps 0-4, rank 0
    got = _compare(case, dev, 30)
    assert list(np.sort(got["tree_tokens"][0, 1:11])) == list(range(10))  # lowest ids of the ties
    _compare(W.make_tree_build_case(2, 4, 3, 150000, seed=13), dev, 20)


def test_many_rows_take_one_cta_per_row(dev):
    """80 sequences x 8 rows x 4-CTA clusters would exceed 2048 CTAs: one CTA per row instead."""
    _compare(W.make_tree_build_case(80, 8, 3, 20000, seed=14), dev, 40, max_near=12)
