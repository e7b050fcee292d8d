"""GPU parity of the fused LM head (spec_lm_head_stats) against the fp64 oracle, through the C ABI.

Max and the gathered logits within tol(H) = H * 7.5e-8, the log of the sum of exp within
2 tol(H) / T; the argmax exact except in rows whose two largest logits lie within tol(H) (counted).
The bound: the bf16 x bf16 products are exact in fp32, so the error is the tensor core's fp32
accumulation over H / 16 steps of K = 16, each taken as losing at most 2^-23 of a logit of magnitude
<= 10 (logits ~ N(0, 3^2) here): (H / 16) * 2^-23 * 10.  Observed on a GB300: 7.1e-5 at H = 4096,
0.7e-5 to 1.0e-5 at H = 512 / 520 (float32 BLAS accumulation of the same products: about 4e-6).
Shapes: one ragged row tile (M = 60) and several (M = 300), H a multiple of 64 or not, V a whole
number of 256-entry tiles or not, V = 128256; temperatures 1 and 0.7.  The statistics then drive
greedy verification of a tree: the argmax gives the same walk as the full logits.
"""
import numpy as np
import pytest

from oracle import lmhead as OL
from oracle import verify as OV
from speculative_decoding_token_spec_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

def tol(H):
    return H * 7.5e-8


@pytest.fixture(scope="module")
def dev(cuda_lib):
    import torch
    return torch.device("cuda:0")


def _run(case, dev, T):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    h = P.dev_tensor(case.hidden, dev).view(torch.bfloat16)
    w = P.dev_tensor(case.weight, dev).view(torch.bfloat16)
    gi = P.dev_tensor(case.gather_idx, dev) if case.gather_idx.shape[1] else None
    out = st.spec_lm_head_stats(h, w, T, gather_idx=gi)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _check(case, dev, T):
    got = _run(case, dev, T)
    ref = OL.lm_head_stats(W.bf16_to_f64(case.hidden), W.bf16_to_f64(case.weight), T,
                           case.gather_idx if case.gather_idx.shape[1] else None)
    M, H = case.hidden.shape
    TOL = tol(H)
    assert got["status"][0] == 0
    assert np.abs(got["max"] - ref["max"]).max() <= TOL
    lse_err = np.abs(np.log(got["sumexp"]) - np.log(ref["sumexp"])).max()
    assert lse_err <= 2 * TOL / T, lse_err
    near = ref["top_gap"] < TOL
    assert np.array_equal(got["argmax"][~near], ref["argmax"][~near])
    assert near.sum() <= max(1, len(near) // 50), near.sum()
    if "gather" in ref:
        ok = ~np.isnan(ref["gather"])
        assert np.array_equal(ok, ~np.isnan(got["gather"]))
        assert np.abs(got["gather"][ok] - ref["gather"][ok]).max() <= TOL
    print(f"M={M} H={H} V={case.weight.shape[0]} T={T}: max err "
          f"{np.abs(got['max'] - ref['max']).max():.2e}, log-sum-exp err {lse_err:.2e}, "
          f"near-tie rows {int(near.sum())}")


@pytest.mark.parametrize("M,H,V,G,T", [
    (60, 4096, 32000, 10, 1.0),     # one 60-node tree, Vicuna-7B-sized head
    (60, 512, 1000, 4, 0.7),        # a ragged vocabulary tile
    (300, 520, 3000, 6, 1.0),       # three row tiles, a partial hidden slice
    (20, 4096, 128256, 8, 0.7),     # 128K vocabulary
])
def test_matches_oracle(dev, M, H, V, G, T):
    _check(W.make_lm_head_case(M, H, V, G, seed=M + V), dev, T)


def test_statistics_drive_greedy_verification(dev):
    """Fused argmax -> greedy walk equals the walk on the full fp64 logits (outside near ties)."""
    B, N, H, V = 3, 24, 256, 2000
    case = W.make_lm_head_case(B * N, H, V, 0, seed=5, sigma=4.0)
    got = _run(case, dev, 1.0)
    lg = OL.logits(W.bf16_to_f64(case.hidden), W.bf16_to_f64(case.weight)).reshape(B, N, V)
    rng = np.random.default_rng(5)
    par = np.stack([W.make_tree(rng, N, 4, 8) for _ in range(B)]).astype(np.int32)
    am = got["argmax"].reshape(B, N)
    # draft tokens: the target's argmax at the parent for most nodes, so the walk goes deep
    tok = np.zeros((B, N), np.int32)
    for b in range(B):
        for i in range(1, N):
            tok[b, i] = am[b, par[b, i]] if rng.random() < 0.6 else int(rng.integers(V))
    ref = OV.tree_verify(lg, None, tok, par, np.zeros((B, N), np.float32), 0.0)
    # near ties: logits ~ N(0, 4^2) here, so the bound of tol(H) scales by 16 / 10; 1e-4 covers it
    near = OL.row_stats(lg.reshape(B * N, V), 1.0)["top_gap"].reshape(B, N) < 1e-4
    for b in range(B):
        if near[b].any():
            continue
        # the greedy walk from the fused argmax
        path, j = [], 0
        while True:
            kids = [i for i in range(1, N) if par[b, i] == j]
            nxt = next((i for i in kids if tok[b, i] == am[b, j]), None)
            if nxt is None:
                break
            path.append(nxt)
            j = nxt
        assert len(path) == ref["accept_len"][b]
        assert [int(tok[b, i]) for i in path] == list(ref["accepted_tokens"][b, :len(path)])
        assert am[b, j] == ref["bonus"][b]


@pytest.mark.parametrize("M,H,V", [(60, 4096, 32000), (300, 520, 3000), (20, 4096, 1000)])
def test_packed_head_gives_the_same_bits(dev, M, H, V):
    """The tile-major head: the packed buffer holds the weight in the stated order (zero padding),
    and the statistics on it equal those on the row-major head bit for bit."""
    import torch
    import speculative_decoding_token_spec_gb300 as st
    case = W.make_lm_head_case(M, H, V, 5, seed=M * 3 + V)
    h = P.dev_tensor(case.hidden, dev).view(torch.bfloat16)
    w = P.dev_tensor(case.weight, dev).view(torch.bfloat16)
    gi = P.dev_tensor(case.gather_idx, dev)
    packed = st.spec_lm_head_pack(w)
    a = st.spec_lm_head_stats(h, w, 0.8, gather_idx=gi)
    b = st.spec_lm_head_stats(h, packed, 0.8, gather_idx=gi, packed_vocab=V)
    torch.cuda.synchronize()
    nk, nv = -(-H // 64), -(-V // 256)
    pk = packed.cpu().numpy().view(np.uint16).reshape(nv, nk, 256, 64)
    full = np.zeros((nv * 256, nk * 64), np.uint16)
    full[:V, :H] = case.weight
    want = full.reshape(nv, 256, nk, 64).transpose(0, 2, 1, 3)
    assert np.array_equal(pk, want)
    for k in ("max", "sumexp", "gather"):
        assert torch.equal(a[k].view(torch.int32), b[k].view(torch.int32)), k
    assert torch.equal(a["argmax"], b["argmax"])
