"""Pins for the tree-attention oracle (CPU only).

Each check compares the oracle with something other than itself: PyTorch's float64
scaled_dot_product_attention under an explicitly built boolean mask (a library routine), a mask
built by transitive closure of the adjacency matrix (not by walking parent pointers), exact special
cases and invariances.
"""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from speculative_decoding_token_spec_gb300 import workloads as W


def _rand(shape, rng):
    return rng.standard_normal(shape)


def _sdpa(q, k, v, mask, scale):
    """q [B,N,Hq,D], k/v [B,Hkv,L,D] float64, mask [B,N,L] bool -> out [B,N,Hq,D], lse [B,Hq,N]."""
    B, N, Hq, D = q.shape
    g = Hq // k.shape[1]
    qt = torch.from_numpy(q).permute(0, 2, 1, 3)                      # B,Hq,N,D
    kt = torch.from_numpy(k).repeat_interleave(g, dim=1)              # B,Hq,L,D
    vt = torch.from_numpy(v).repeat_interleave(g, dim=1)
    m = torch.from_numpy(mask)[:, None, :, :]                         # B,1,N,L
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)
    s = (qt @ kt.transpose(-1, -2)) * scale
    s = s.masked_fill(~m, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)                                  # B,Hq,N
    return o.permute(0, 2, 1, 3).numpy(), lse.numpy()


def _closure_mask(parent, prefix, Lmax):
    """Visibility from the reflexive-transitive closure of the child->parent adjacency matrix."""
    N = len(parent)
    A = np.zeros((N, N), dtype=np.int64)
    for i in range(1, N):
        A[i, parent[i]] = 1
    R = np.eye(N, dtype=np.int64)
    P = np.eye(N, dtype=np.int64)
    for _ in range(N):
        P = np.minimum(P @ A, 1)
        R = np.minimum(R + P, 1)
    mask = np.zeros((N, Lmax), dtype=bool)
    mask[:, :prefix] = True
    mask[:, prefix:prefix + N] = R.astype(bool)
    return mask


def _case(B, N, Hq, Hkv, D, lens, parents, seed, pad=3):
    rng = np.random.default_rng(seed)
    Lmax = max(lens) + N + pad
    q = _rand((B, N, Hq, D), rng)
    k = _rand((B, Hkv, Lmax, D), rng)
    v = _rand((B, Hkv, Lmax, D), rng)
    par = np.stack([np.asarray(p, dtype=np.int32) for p in parents])
    return q, k, v, np.asarray(lens, dtype=np.int32), par, Lmax


def test_chain_equals_causal_attention():
    """A chain-shaped tree is ordinary causal attention over prefix + chain."""
    N, D = 7, 16
    q, k, v, lens, par, Lmax = _case(2, N, 4, 4, D, [11, 5], [W.chain_tree(N)] * 2, 1)
    mask = np.zeros((2, N, Lmax), dtype=bool)
    for b in range(2):
        L = lens[b]
        mask[b, :, :L] = True
        mask[b, :, L:L + N] = np.tril(np.ones((N, N), dtype=bool))
    scale = 1 / np.sqrt(D)
    o_ref, lse_ref = _sdpa(q, k, v, mask, scale)
    o, lse = OA.tree_attention(q, k, v, lens, par, scale)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_tree_matches_closure_mask_gqa(seed):
    """Random trees with GQA (g = 2): mask from the adjacency closure, heads grouped contiguously."""
    rng = np.random.default_rng(100 + seed)
    N, D = 12, 32
    parents = [W.make_tree(rng, N, 4, 4) for _ in range(3)]
    lens = [0, 9, 23]
    q, k, v, lens, par, Lmax = _case(3, N, 6, 3, D, lens, parents, seed)
    mask = np.stack([_closure_mask(parents[b], lens[b], Lmax) for b in range(3)])
    scale = 0.37
    o_ref, lse_ref = _sdpa(q, k, v, mask, scale)
    o, lse = OA.tree_attention(q, k, v, lens, par, scale)
    np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-11, atol=1e-11)


def test_star_tree_sees_prefix_root_and_self():
    N, D, L = 6, 8, 4
    par = np.array([-1] + [0] * (N - 1), dtype=np.int32)
    q, k, v, lens, P, Lmax = _case(1, N, 2, 2, D, [L], [par], 7)
    scale = 0.5
    o, _ = OA.tree_attention(q, k, v, lens, P, scale)
    for i in range(N):
        keys = list(range(L)) + [L] + ([L + i] if i else [])
        for h in range(2):
            s = scale * k[0, h, keys] @ q[0, i, h]
            w = np.exp(s - s.max())
            ref = (w / w.sum()) @ v[0, h, keys]
            np.testing.assert_allclose(o[0, i, h], ref, rtol=1e-13, atol=1e-13)


def test_root_only_empty_prefix_returns_root_value():
    """L = 0 and N = 1: the only visible key is the root's own, so the output is v_root."""
    q, k, v, lens, par, _ = _case(1, 1, 3, 1, 8, [0], [[-1]], 3)
    o, lse = OA.tree_attention(q, k, v, lens, par, 0.25)
    for h in range(3):
        np.testing.assert_array_equal(o[0, 0, h], v[0, 0, 0])
        assert lse[0, h, 0] == pytest.approx(0.25 * float(q[0, 0, h] @ k[0, 0, 0]), abs=1e-14)


def test_prefix_permutation_invariance():
    rng = np.random.default_rng(5)
    N, D, L = 5, 16, 20
    par = W.make_tree(rng, N, 3, 2)
    q, k, v, lens, P, _ = _case(1, N, 2, 2, D, [L], [par], 9)
    o1, l1 = OA.tree_attention(q, k, v, lens, P, 0.3)
    perm = rng.permutation(L)
    k2, v2 = k.copy(), v.copy()
    k2[0, :, :L] = k[0][:, perm]
    v2[0, :, :L] = v[0][:, perm]
    o2, l2 = OA.tree_attention(q, k2, v2, lens, P, 0.3)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=1e-12, atol=1e-12)


def test_slots_beyond_tree_are_ignored():
    """Cache slots after L_b + N (and other nodes' slots) do not change a node's output."""
    rng = np.random.default_rng(8)
    N, D, L = 6, 8, 3
    par = W.make_tree(rng, N, 3, 3)
    q, k, v, lens, P, Lmax = _case(1, N, 2, 1, D, [L], [par], 4, pad=5)
    o1, _ = OA.tree_attention(q, k, v, lens, P, 0.4)
    k[0, :, L + N:] = 1e3
    v[0, :, L + N:] = -1e3
    o2, _ = OA.tree_attention(q, k, v, lens, P, 0.4)
    np.testing.assert_array_equal(o1, o2)


def test_subset_of_nodes():
    q, k, v, lens, par, _ = _case(2, 4, 2, 2, 8, [3, 6], [W.chain_tree(4)] * 2, 11)
    full, _ = OA.tree_attention(q, k, v, lens, par, 0.3)
    part, _ = OA.tree_attention(q, k, v, lens, par, 0.3, nodes=[(1, 2)])
    np.testing.assert_array_equal(part[1, 2], full[1, 2])
    assert np.isnan(part[0, 0]).all()
