"""GPU parity of verification from the LM head's statistics (spec_tree_verify_head) through the
C ABI, against the fp64 oracle (oracle/lmhead.py: tree verification of hidden @ head^T) and
against spec_tree_verify on the same logits.

Inputs: make_head_verify_case's lattice operands, whose logits are exact in fp32 in any summation
order, so both GPU paths see exactly the oracle's logits.  Bands:
* decisions the oracle takes within 1e-6 (its near-tie band) are not compared, as everywhere;
* a first-child test decided from the statistics uses S, an fp32 sum (each term exp2f of an
  exactly rounded argument, sums of at most 256 + 4 + 5 terms per row): |dS / S| <= 2e-5, so such
  a test can flip only when |r - q / p| <= r |dS / S| < 2e-5; sequences with a first-child test on
  the oracle's walk within 1e-4 are not compared either (counted, and bounded).
Elsewhere the accepted nodes, tokens, lengths and the bonus are bit-exact, and equal to
spec_tree_verify's.
"""
import numpy as np
import pytest

from oracle import lmhead as OL
from oracle import verify as OV
from speculative_decoding_token_spec_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

HEAD_BAND = 1e-4
KEYS = ("accept_len", "accepted_tokens", "bonus", "accepted_nodes", "status")


@pytest.fixture(scope="module")
def dev(cuda_lib):
    import torch
    return torch.device("cuda:0")


def _logits(case):
    B, N, H = case.hidden.shape
    return OL.logits(W.bf16_to_f64(case.hidden).reshape(B * N, H),
                     W.bf16_to_f64(case.head)).reshape(B, N, -1)


def run_head(case, dev, max_depth=None, packed=False, hidden=None):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    B, N, H = case.hidden.shape
    V = case.head.shape[0]
    h = P.dev_tensor(case.hidden if hidden is None else hidden, dev).view(torch.bfloat16)
    w = P.dev_tensor(case.head, dev).view(torch.bfloat16)
    kw = {}
    if packed:
        w = st.spec_lm_head_pack(w)
        kw["packed_vocab"] = V
    T = case.temperature
    res = st.spec_tree_verify_head(
        h, w, P.dev_tensor(case.draft_probs, dev) if T > 0 else None,
        P.dev_tensor(case.tree_tokens, dev), P.dev_tensor(case.tree_parent, dev),
        P.dev_tensor(case.uniforms, dev), T,
        case.max_depth if max_depth is None else max_depth, **kw)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in res.items()}


def run_plain(case, lg, dev):
    vc = W.VerifyCase(lg.astype(np.float32), case.draft_probs, case.tree_tokens, case.tree_parent,
                      case.uniforms, case.temperature)
    return P.run_verify_gpu(vc, dev, want_child_q=False)


def head_near(ref, case):
    """Sequences not compared: the oracle's near ties, and first-child tests on its walk within
    HEAD_BAND (they may be decided from the statistics)."""
    B = case.tree_parent.shape[0]
    near = ref["near_tie"].copy()
    if case.temperature == 0:
        return near
    for b in range(B):
        if ref["status"][b]:
            continue
        kids = OV.children(case.tree_parent[b])
        n = int(ref["accept_len"][b])
        for c in [0] + [int(x) for x in ref["accepted_nodes"][b, :n]]:
            if not kids[c]:
                continue
            k = kids[c][0]
            qx = ref["child_q"][b, k]
            px = float(case.draft_probs[b, c, case.tree_tokens[b, k]])
            if OV.decision_margin(float(case.uniforms[b, k]), qx, px) < HEAD_BAND:
                near[b] = True
    return near


def check(case, dev, max_near=None, packed=False, plain=True):
    lg = _logits(case)
    ref = OV.tree_verify(lg, case.draft_probs, case.tree_tokens, case.tree_parent, case.uniforms,
                         case.temperature, with_table=case.temperature > 0)
    got = run_head(case, dev, packed=packed)
    near = head_near(ref, case)
    np.testing.assert_array_equal(got["status"], ref["status"])
    B = case.tree_parent.shape[0]
    for b in range(B):
        if near[b]:
            continue
        ctx = f"sequence {b}"
        assert got["accept_len"][b] == ref["accept_len"][b], ctx
        assert got["bonus"][b] == ref["bonus"][b], ctx
        np.testing.assert_array_equal(got["accepted_tokens"][b], ref["accepted_tokens"][b], ctx)
        np.testing.assert_array_equal(got["accepted_nodes"][b], ref["accepted_nodes"][b], ctx)
    if plain:
        other = run_plain(case, lg, dev)
        for b in range(B):
            if not near[b]:
                for k in KEYS:
                    np.testing.assert_array_equal(got[k][b], other[k][b], f"{k} {b}")
    assert near.sum() <= (max_near if max_near is not None else max(1, B // 8)), near.sum()
    return got, ref


@pytest.mark.parametrize("T", [0.7, 1.0])
def test_eagle_tree_against_oracle_and_plain(dev, T):
    for B, seeds in ((1, range(4)), (8, range(2))):
        for seed in seeds:
            for sd in (0.5, 1.0):
                cfg = W.config("eagle_vicuna7b", B=B, V=5000)
                check(W.make_head_verify_case(cfg, 512, T, seed=20 + seed, sigma_d=sd), dev)


def test_greedy(dev):
    for seed in range(3):
        cfg = W.config("eagle_vicuna7b", B=8, V=5000)
        got, ref = check(W.make_head_verify_case(cfg, 512, 0.0, seed=seed), dev, max_near=0)
        assert (got["status"] == 0).all()


def test_full_vocabulary_and_hidden_size(dev):
    """The 60-node EAGLE tree at V = 32000, H = 4096 (a Vicuna-7B head)."""
    cfg = W.config("eagle_vicuna7b", B=2)
    for T in (1.0, 0.0):
        check(W.make_head_verify_case(cfg, 4096, T, seed=7), dev)


def test_packed_head_same_bits(dev):
    cfg = W.config("eagle_vicuna7b", B=4, V=3001)
    case = W.make_head_verify_case(cfg, 520, 1.0, seed=3)
    a = run_head(case, dev)
    b = run_head(case, dev, packed=True)
    for k in KEYS:
        np.testing.assert_array_equal(a[k], b[k], k)
    check(case, dev, packed=True, plain=False)


def test_shapes_and_trees(dev):
    """Root only, chains (depth N - 1), stars (many residual rounds at one node), two-level stars,
    64 nodes, ragged batches and odd vocabularies."""
    cases = []
    cfg = W.config("eagle_vicuna7b", B=3, N=1, V=517)
    cases.append(W.make_head_verify_case(cfg, 64, 1.0, seed=1))
    cfg = W.config("eagle_vicuna7b", B=5, N=12, V=1000)
    chain = np.stack([W.chain_tree(12)] * 5)
    for sd in (0.3, 2.0):
        cases.append(W.make_head_verify_case(cfg, 128, 1.0, seed=2, sigma_d=sd, tree_parent=chain))
    star = np.array([[-1] + [0] * 40] * 3, np.int32)
    cfg = W.config("eagle_vicuna7b", B=3, N=41, V=2000)
    for sd in (0.5, 3.0):
        cases.append(W.make_head_verify_case(cfg, 256, 1.0, seed=9, sigma_d=sd, tree_parent=star))
    K = 7
    par = [-1] + [0] * K
    for c in range(1, K + 1):
        par += [c] * K
    two = np.array([par] * 4, np.int32)
    cfg = W.config("eagle_vicuna7b", B=4, N=len(par), V=3000)
    cases.append(W.make_head_verify_case(cfg, 256, 0.7, seed=5, sigma_d=1.0, tree_parent=two))
    cfg = W.config("eagle_vicuna7b", B=2, N=64, depth=7, width=10, V=4003)
    cases.append(W.make_head_verify_case(cfg, 192, 1.0, seed=5))
    # batches: 16 walk blocks; row passes over two 128-row tiles
    cfg = W.config("eagle_vicuna7b", B=64, N=20, depth=4, width=8, V=3000)
    cases.append(W.make_head_verify_case(cfg, 256, 1.0, seed=6))
    cfg = W.config("eagle_vicuna7b", B=130, N=4, depth=2, width=2, V=600)
    cases.append(W.make_head_verify_case(cfg, 64, 0.7, seed=8, sigma_d=0.5))
    for case in cases:
        check(case, dev)


def test_depth_bound_and_bad_trees(dev):
    cfg = W.config("eagle_vicuna7b", B=4, N=12, V=1000)
    chain = np.stack([W.chain_tree(12)] * 4)
    case = W.make_head_verify_case(cfg, 64, 1.0, seed=4, tree_parent=chain)
    assert case.max_depth == 11
    got = run_head(case, dev, max_depth=10)  # one level short: every sequence is flagged
    assert (got["status"] == OV.ST_BAD_TREE).all()
    assert (got["accept_len"] == -1).all() and (got["bonus"] == -1).all()
    assert (got["accepted_tokens"] == -1).all() and (got["accepted_nodes"] == -1).all()
    case = W.make_head_verify_case(W.config("eagle_vicuna7b", B=4, V=1000), 64, 1.0, seed=4)
    case.tree_parent[1, 5] = 7  # a parent after its child
    case.tree_tokens[2, 3] = 1000  # a token outside [0, V)
    got, ref = check(case, dev)
    assert got["status"][1] == OV.ST_BAD_TREE and got["status"][2] == OV.ST_BAD_TOKEN
    assert got["status"][0] == 0 and got["status"][3] == 0


def test_nonfinite_hidden_on_and_off_the_walk(dev):
    import torch  # noqa: F401
    cfg = W.config("eagle_vicuna7b", B=1, V=2000)
    case = W.make_head_verify_case(cfg, 128, 1.0, seed=12)
    clean = run_head(case, dev)
    assert clean["status"][0] == 0
    acc = [int(x) for x in clean["accepted_nodes"][0] if x >= 0]
    on = {0} | set(acc)
    par = case.tree_parent[0]
    internal = [i for i in range(1, case.tree_parent.shape[1]) if (par == i).any()]
    off = [i for i in internal if i not in on]
    assert off
    nan = np.uint16(0x7FC0)  # bf16 NaN
    h = case.hidden.copy()
    h[0, off[0], 3] = nan  # a row nothing on the walk reads: same results, no flag
    got = run_head(case, dev, hidden=h)
    for k in KEYS:
        np.testing.assert_array_equal(got[k], clean[k], k)
    for node in (0, acc[-1] if acc else 0):  # the root, the node where the walk stops
        h = case.hidden.copy()
        h[0, node, 5] = nan
        got = run_head(case, dev, hidden=h)
        assert got["status"][0] == OV.ST_NONFINITE, node
        assert got["accept_len"][0] == -1 and got["bonus"][0] == -1
        assert (got["accepted_tokens"][0] == -1).all()


def test_cuda_graph_replays(dev):
    """The call is a fixed sequence of launches: captured once, replayed on new inputs."""
    import torch
    import speculative_decoding_token_spec_gb300 as st
    cfg = W.config("eagle_vicuna7b", B=4, V=3000)
    cases = [W.make_head_verify_case(cfg, 256, 1.0, seed=40 + i) for i in range(4)]
    depth = max(c.max_depth for c in cases)
    t = lambda a: P.dev_tensor(a, dev)  # noqa: E731
    bufs = [t(cases[0].hidden).view(torch.bfloat16), t(cases[0].head).view(torch.bfloat16),
            t(cases[0].draft_probs), t(cases[0].tree_tokens), t(cases[0].tree_parent),
            t(cases[0].uniforms)]
    B, N, H = cases[0].hidden.shape
    ws = torch.empty((st.spec_tree_verify_head_workspace(B, N, H, 3000, depth),),
                     dtype=torch.uint8, device=dev)
    st.spec_tree_verify_head(*bufs, 1.0, depth, workspace=ws)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            out = st.spec_tree_verify_head(*bufs, 1.0, depth, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    for case in cases + cases[:1]:
        for dst, src in zip(bufs, (case.hidden, case.head, case.draft_probs, case.tree_tokens,
                                   case.tree_parent, case.uniforms)):
            dst.copy_(t(src).view(dst.dtype))
        g.replay()
        torch.cuda.synchronize()
        got = {k: v.cpu().numpy() for k, v in out.items()}
        ref = run_head(case, dev, max_depth=depth)
        for k in KEYS:
            np.testing.assert_array_equal(got[k], ref[k], k)
