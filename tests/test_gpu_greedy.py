"""GPU parity of the greedy verification from each node's argmax (spec_tree_verify_greedy) against
the fp64 oracle's temperature-0 verification, through the C ABI.

The oracle sees logits whose argmax is the given one (1 at that token, 0 elsewhere), so both sides
walk on the same argmax; everything is compared exactly (accept_len, accepted tokens and nodes, the
bonus, the status).  Shapes: B not a multiple of the 8 sequences of a block, N from 1 (the root
alone) to 64 (both node slots of every lane), chain trees (walks of N - 1 steps), siblings with equal
tokens (the lowest index wins), and the error cases: a bad tree, a bad token, an argmax outside
[0, V) at a node the walk reaches (and one it does not reach), checked against the entry's stated
contract (the oracle's walk does not model rows without a maximum).  Then end to end: the fused LM
head's argmax drives it and the walk equals the oracle's on the full fp64 logits (outside near
ties).
"""
import numpy as np
import pytest

from oracle import lmhead as OL
from oracle import verify as OV
from speculative_decoding_token_spec_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_lib):
    import torch
    return torch.device("cuda:0")


def _case(B, N, V, seed, depth=6, follow=0.7):
    """Trees, draft tokens and per-node argmaxes; a node's argmax equals one of its children's
    tokens with probability `follow`, so that walks go deep."""
    rng = np.random.default_rng(seed)
    d = max(1, min(depth, N - 1))
    width = max(10, -(-(N - 1) // d))
    par = np.stack([W.make_tree(rng, N, d, width) for _ in range(B)]).astype(np.int32)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    am = rng.integers(0, V, size=(B, N)).astype(np.int32)
    for b in range(B):
        for j in range(N):
            kids = [i for i in range(1, N) if par[b, i] == j]
            if kids and rng.random() < follow:
                am[b, j] = tok[b, kids[int(rng.integers(len(kids)))]]
    return par, tok, am


def _oracle(par, tok, am, V):
    """The oracle's temperature-0 verification on logits whose argmax is `am` (all in [0, V))."""
    B, N = par.shape
    assert ((am >= 0) & (am < V)).all()
    lg = np.zeros((B, N, V))
    for b in range(B):
        for i in range(N):
            lg[b, i, am[b, i]] = 1.0
    return OV.tree_verify(lg, None, tok, par, np.zeros((B, N), np.float32), 0.0)


def _gpu(par, tok, am, V, dev):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    out = st.spec_tree_verify_greedy(torch.from_numpy(am).to(dev), torch.from_numpy(tok).to(dev),
                                     torch.from_numpy(par).to(dev), V)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _compare(par, tok, am, V, dev):
    got = _gpu(par, tok, am, V, dev)
    ref = _oracle(par, tok, am, V)
    for k in ("accept_len", "accepted_tokens", "accepted_nodes", "bonus"):
        assert np.array_equal(got[k], ref[k]), (k, got[k], ref[k])
    assert np.array_equal(got["status"] != 0, ref["status"] != 0)
    return got, ref


@pytest.mark.parametrize("B,N,V,seed", [
    (37, 60, 32000, 0),    # EAGLE-sized trees, B ragged over blocks of 8
    (8, 64, 1000, 1),      # both node slots of every lane
    (5, 1, 100, 2),        # the root alone: accept nothing, bonus = argmax of the root
    (16, 33, 128256, 3),   # one node in the second slot
])
def test_matches_oracle(dev, B, N, V, seed):
    par, tok, am = _case(B, N, V, seed)
    got, ref = _compare(par, tok, am, V, dev)
    assert (got["status"] == 0).all()
    if N > 1:
        assert ref["accept_len"].max() >= 2


def test_chain_accepts_everything(dev):
    """A chain whose every node's argmax is its child's token: N - 1 accepted (crosses lane 31)."""
    B, N, V = 3, 64, 500
    par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    rng = np.random.default_rng(4)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    am = np.roll(tok, -1, axis=1)
    am[:, -1] = 7
    am[1, 40] = (tok[1, 41] + 1) % V  # sequence 1 stops at node 40
    got, ref = _compare(par, tok, am, V, dev)
    assert list(got["accept_len"]) == [63, 40, 63]
    assert got["bonus"][0] == 7 and got["bonus"][1] == am[1, 40]


def test_equal_sibling_tokens_take_the_lowest_index(dev):
    V = 50
    par = np.array([[-1, 0, 0, 0, 1, 2, 3]], np.int32)
    tok = np.array([[0, 9, 9, 9, 4, 5, 6]], np.int32)
    am = np.array([[9, 4, 5, 6, 1, 1, 1]], np.int32)
    got, _ = _compare(par, tok, am, V, dev)
    assert list(got["accepted_nodes"][0, :2]) == [1, 4]


def test_errors_flag_only_their_sequence(dev):
    """Bad tree, bad token, an argmax outside [0, V) at a node the walk reaches: that sequence
    alone gets its status bit and -1 outputs.  The same argmax at a node the walk does not reach
    changes nothing."""
    B, N, V = 6, 20, 300
    par, tok, am = _case(B, N, V, 5, follow=1.0)
    ref = _oracle(par, tok, am, V)
    par[1, 5] = 7                                  # parent not before the node: bad tree
    tok[2, 3] = V                                  # bad token
    am[3, 0] = -1                                  # the root's row has no maximum
    walk4 = set(int(x) for x in ref["accepted_nodes"][4] if x >= 0) | {0}
    off = next(i for i in range(1, N) if i not in walk4)
    am[4, off] = V + 5                             # not reached: no effect
    n5 = int(ref["accept_len"][5])
    am[5, ref["accepted_nodes"][5, n5 - 1] if n5 else 0] = 2 ** 31 - 1  # the terminal node
    got = _gpu(par, tok, am, V, dev)
    assert list(got["status"]) == [0, 1, 4, 8, 0, 8]
    for b in (1, 2, 3, 5):
        assert got["accept_len"][b] == -1 and got["bonus"][b] == -1
        assert (got["accepted_tokens"][b] == -1).all() and (got["accepted_nodes"][b] == -1).all()
    for b in (0, 4):
        for k in ("accept_len", "accepted_tokens", "accepted_nodes", "bonus"):
            assert np.array_equal(got[k][b], ref[k][b]), (b, k)


def test_fused_lm_head_drives_greedy_verification(dev):
    """spec_lm_head_stats's argmax, viewed as [B, N], into spec_tree_verify_greedy: the walk equals
    the oracle's temperature-0 verification on the full fp64 logits, outside near-tie rows."""
    import torch
    import speculative_decoding_token_spec_gb300 as st
    B, N, H, V = 4, 30, 512, 3000
    case = W.make_lm_head_case(B * N, H, V, 0, seed=6, sigma=4.0)
    h = P.dev_tensor(case.hidden, dev).view(torch.bfloat16)
    w = P.dev_tensor(case.weight, dev).view(torch.bfloat16)
    stats = st.spec_lm_head_stats(h, w, 1.0)
    lg = OL.logits(W.bf16_to_f64(case.hidden), W.bf16_to_f64(case.weight)).reshape(B, N, V)
    am_ref = lg.argmax(axis=2).astype(np.int32)
    rng = np.random.default_rng(6)
    par = np.stack([W.make_tree(rng, N, 5, 8) for _ in range(B)]).astype(np.int32)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    for b in range(B):
        for i in range(1, N):
            if rng.random() < 0.6:
                tok[b, i] = am_ref[b, par[b, i]]
    out = st.spec_tree_verify_greedy(stats["argmax"].view(B, N), torch.from_numpy(tok).to(dev),
                                     torch.from_numpy(par).to(dev), V)
    torch.cuda.synchronize()
    ref = OV.tree_verify(lg, None, tok, par, np.zeros((B, N), np.float32), 0.0)
    near = OL.row_stats(lg.reshape(B * N, V), 1.0)["top_gap"].reshape(B, N) < 1e-3
    compared = 0
    for b in range(B):
        if near[b].any():
            continue
        compared += 1
        assert out["accept_len"][b].item() == ref["accept_len"][b]
        assert np.array_equal(out["accepted_tokens"][b].cpu().numpy(), ref["accepted_tokens"][b])
        assert out["bonus"][b].item() == ref["bonus"][b]
    assert compared >= B - 1 and ref["accept_len"].max() >= 1
