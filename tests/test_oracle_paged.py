"""Pins for the paged-cache and compaction oracle (CPU only).

Each check compares ``oracle.paged`` with something other than itself:

* page round trip -- pages written from a contiguous cache by slicing the cache into page-sized
  blocks (numpy reshapes, not the oracle's slot lookup), then gathered back;
* compaction then plain causal attention -- after the accepted path moves next to the root, the
  last accepted node's query over the committed prefix, computed by PyTorch's float64
  scaled_dot_product_attention with no mask, must equal the tree attention of that node before
  compaction (its visible keys are exactly the prefix, the root and the path);
* invariants -- slots outside L+1..L+len are untouched, failed or malformed requests leave the
  sequence unchanged, the paged and contiguous compactions agree.
"""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import paged as OP
from speculative_decoding_token_spec_gb300 import workloads as W


def _pages_from_contiguous(cache, page_size, rng, spare=2):
    """Cut [B, Hkv, S, D] into pages with numpy reshapes and place them at random physical slots."""
    B, H, S, D = cache.shape
    assert S % page_size == 0
    per = S // page_size
    blocks = cache.reshape(B, H, per, page_size, D).transpose(0, 2, 1, 3, 4)  # B, per, H, P, D
    num_pages = B * per + spare
    perm = rng.permutation(num_pages)
    pages = np.full((num_pages, H, page_size, D), np.nan)
    table = perm[:B * per].reshape(B, per).astype(np.int32)
    pages[table.reshape(-1)] = blocks.reshape(B * per, H, page_size, D)
    return pages, table


@pytest.mark.parametrize("page_size", [1, 4, 16])
def test_gather_round_trip(page_size):
    rng = np.random.default_rng(11)
    cache = rng.standard_normal((3, 2, 48, 5))
    pages, table = _pages_from_contiguous(cache, page_size, rng)
    back = OP.gather_pages(pages, table, page_size, 48)
    assert np.array_equal(back, cache)


def test_gather_marks_missing_pages():
    pages = np.zeros((2, 1, 4, 3))
    table = np.array([[1, -1, 7]], dtype=np.int32)
    g = OP.gather_pages(pages, table, 4, 12)
    assert np.all(g[0, :, :4] == 0) and np.isnan(g[0, :, 4:]).all()


@pytest.mark.parametrize("page_size", [8, 16])
def test_paged_attention_equals_contiguous(page_size):
    rng = np.random.default_rng(5)
    B, N, Hq, Hkv, D = 2, 7, 4, 2, 8
    S = 64
    q = rng.standard_normal((B, N, Hq, D))
    k = rng.standard_normal((B, Hkv, S, D))
    v = rng.standard_normal((B, Hkv, S, D))
    lens = np.array([20, 33], dtype=np.int32)
    par = np.stack([W.make_tree(np.random.default_rng(b), N, 3, 3) for b in range(B)])
    kp, table = _pages_from_contiguous(k, page_size, rng)
    vp = np.full_like(kp, np.nan)
    vp[table.reshape(-1)] = v.reshape(B, Hkv, S // page_size, page_size, D).transpose(
        0, 2, 1, 3, 4).reshape(-1, Hkv, page_size, D)
    o1, l1 = OA.tree_attention(q, k, v, lens, par, 0.3)
    o2, l2 = OP.paged_tree_attention(q, kp, vp, table, page_size, lens, par, 0.3)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def _chain_tree_through(path, n):
    """A tree whose root-to-node path is `path` (root first); other nodes hang off the root."""
    par = np.zeros(n, dtype=np.int32)
    par[0] = -1
    prev = 0
    for x in path:
        par[x] = prev
        prev = x
    return par


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_compaction_then_causal_equals_tree_attention(seed):
    rng = np.random.default_rng(100 + seed)
    Hkv, g, D, N = 2, 2, 8, 12
    Hq = Hkv * g
    L = int(rng.integers(0, 30))
    Lmax = L + N + 4
    ln = int(rng.integers(1, N))
    path = np.sort(rng.choice(np.arange(1, N), size=ln, replace=False)).astype(np.int32)
    par = _chain_tree_through(path, N)
    k = rng.standard_normal((1, Hkv, Lmax, D))
    v = rng.standard_normal((1, Hkv, Lmax, D))
    q = rng.standard_normal((1, N, Hq, D))
    c = int(path[-1])
    before, _ = OA.tree_attention(q, k, v, np.array([L]), par[None], 0.25, nodes=[(0, c)])
    nodes = np.full((1, N), -1, dtype=np.int32)
    nodes[0, :ln] = path
    k2, v2, new_lens, bad = OP.kv_compact(k, v, np.array([L]), np.array([ln]), nodes)
    assert not bad[0] and new_lens[0] == L + 1 + ln
    Lc = L + 1 + ln
    qt = torch.from_numpy(q[0, c]).reshape(Hkv, g, 1, D)               # one query per head
    kt = torch.from_numpy(k2[0, :, :Lc])[:, None].expand(Hkv, g, Lc, D)
    vt = torch.from_numpy(v2[0, :, :Lc])[:, None].expand(Hkv, g, Lc, D)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=0.25)
    np.testing.assert_allclose(o.reshape(Hq, D).numpy(), before[0, c], rtol=1e-12, atol=1e-12)


def test_compaction_touches_only_the_committed_slots():
    cc = W.make_compaction_case(6, 10, 2, 4, seed=3, lens=[-1, 0, 1, 4, 9, 3])
    k = W.bf16_to_f64(cc.k_cache)
    v = W.bf16_to_f64(cc.v_cache)
    k2, v2, new_lens, bad = OP.kv_compact(k, v, cc.prefix_lens, cc.accept_len, cc.accepted_nodes)
    assert not bad.any()
    for b in range(6):
        L, ln = int(cc.prefix_lens[b]), int(cc.accept_len[b])
        moved = set(range(L + 1, L + 1 + max(ln, 0)))
        for s in range(k.shape[2]):
            if s not in moved:
                assert np.array_equal(k2[b, :, s], k[b, :, s]) and np.array_equal(v2[b, :, s], v[b, :, s])
        for i in range(max(ln, 0)):
            src = L + int(cc.accepted_nodes[b, i])
            assert np.array_equal(k2[b, :, L + 1 + i], k[b, :, src])
        assert new_lens[b] == (L if ln < 0 else L + 1 + ln)


def test_compaction_overlapping_moves_read_the_old_values():
    """Path [2, 3]: slot L+2 is both the source of the first move and the target of the second."""
    k = np.arange(10, dtype=np.float64).reshape(1, 1, 10, 1)
    nodes = np.array([[2, 3, -1, -1]], dtype=np.int32)
    k2, _, new_lens, bad = OP.kv_compact(k, k.copy(), np.array([4]), np.array([2]), nodes)
    assert not bad[0] and new_lens[0] == 7
    assert k2[0, 0, :, 0].tolist() == [0, 1, 2, 3, 4, 6, 7, 7, 8, 9]


@pytest.mark.parametrize("nodes,ln,L", [([3, 2, -1, -1], 2, 1),   # not increasing
                                        ([0, 1, -1, -1], 2, 1),   # the root is not a draft
                                        ([1, 5, -1, -1], 2, 1),   # node id >= N
                                        ([1, 2, 3, -1], 3, 5)])   # L + 1 + len > Lmax
def test_compaction_rejects_malformed_requests(nodes, ln, L):
    k = np.arange(8, dtype=np.float64).reshape(1, 1, 8, 1)
    k2, _, new_lens, bad = OP.kv_compact(k, k.copy(), np.array([L]), np.array([ln]),
                                         np.array([nodes], dtype=np.int32))
    assert bad[0] and new_lens[0] == L and np.array_equal(k2, k)


@pytest.mark.parametrize("page_size", [2, 4, 8])
def test_paged_compaction_matches_contiguous(page_size):
    rng = np.random.default_rng(77)
    cc = W.make_compaction_case(4, 8, 2, 3, seed=9, prefix_range=(0, 20), lmax_pad=0)
    k = W.bf16_to_f64(cc.k_cache)
    v = W.bf16_to_f64(cc.v_cache)
    S = k.shape[2]
    S_pad = -(-S // page_size) * page_size
    k = np.concatenate([k, np.zeros((4, 2, S_pad - S, 3))], axis=2)
    v = np.concatenate([v, np.zeros((4, 2, S_pad - S, 3))], axis=2)
    kp, table = _pages_from_contiguous(k, page_size, rng)
    vp = np.full_like(kp, np.nan)
    vp[table.reshape(-1)] = v.reshape(4, 2, S_pad // page_size, page_size, 3).transpose(
        0, 2, 1, 3, 4).reshape(-1, 2, page_size, 3)
    kc, vc, lens_c, bad_c = OP.kv_compact(k, v, cc.prefix_lens, cc.accept_len, cc.accepted_nodes)
    kq, vq, lens_p, bad_p = OP.kv_compact_paged(kp, vp, table, page_size, cc.prefix_lens,
                                                cc.accept_len, cc.accepted_nodes)
    assert np.array_equal(lens_c, lens_p) and np.array_equal(bad_c, bad_p)
    assert np.array_equal(OP.gather_pages(kq, table, page_size, S_pad), kc)
    assert np.array_equal(OP.gather_pages(vq, table, page_size, S_pad), vc)


def test_paged_compaction_rejects_missing_pages():
    pages = np.zeros((2, 1, 4, 1))
    table = np.array([[0, -1]], dtype=np.int32)      # slots 4..7 have no page
    nodes = np.array([[1, 2, 3, -1, -1]], dtype=np.int32)
    kq, _, lens, bad = OP.kv_compact_paged(pages, pages.copy(), table, 4, np.array([2]),
                                           np.array([3]), nodes)
    assert bad[0] and lens[0] == 2 and np.array_equal(kq, pages)
