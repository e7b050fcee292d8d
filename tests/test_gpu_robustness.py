"""Robustness of the C-ABI entry points on the GPU, in the forms that fault and hang nothing.

* Guard bands (canaries): every output and workspace buffer of every entry point is a view into a
  larger buffer whose bytes around the view hold a fixed pattern; after the call the pattern must
  be intact.  Shapes are the odd ones where an index slip shows first: N = 1, V = 1 / 3 / 517,
  D = 64, prefix 0, ragged batches.  This stands in for an out-of-bounds checker, which this setup
  does not run.
* Stale workspace contents: one caller workspace reused by verification calls whose B * N shrinks
  and grows, pre-filled with words an arrival counter could be mistaken for.
* The timeout path: with spec_debug_set_verify_wait_polls(0) every bounded wait of the
  verification kernels gives up on its first attempt, flags SPEC_ST_TIMEOUT and then waits for its
  copies and stores with the normal limit; the call reports the timeout for every sequence, and a
  normal call right after gives the same bits as before.
"""
import numpy as np
import pytest

from speculative_decoding_token_spec_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

GUARD = 64          # guard elements on each side (a multiple of 16 bytes for every dtype used)
PATTERN = 0xA5


@pytest.fixture(scope="module")
def dev(cuda_lib):
    import torch
    return torch.device("cuda:0")


class Guarded:
    """A tensor of `shape` inside a buffer with GUARD elements of PATTERN bytes on each side."""

    def __init__(self, shape, dtype, dev, fill=None):
        import torch
        self.n = int(np.prod(shape)) if len(shape) else 1
        self.buf = torch.empty((self.n + 2 * GUARD,), dtype=dtype, device=dev)
        self.buf.view(torch.uint8).fill_(PATTERN)
        self.t = self.buf[GUARD:GUARD + self.n].view(shape)
        if fill is not None:
            self.t.fill_(fill)

    def intact(self):
        import torch
        torch.cuda.synchronize()
        raw = self.buf.view(torch.uint8)
        es = self.buf.element_size()
        head, tail = raw[:GUARD * es], raw[(GUARD + self.n) * es:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


def _assert_intact(bufs):
    bad = [name for name, g in bufs.items() if not g.intact()]
    assert not bad, f"guard bands overwritten around: {bad}"


def _t(a, dev):
    return P.dev_tensor(a, dev)


# ------------------------------------------------------------------------------------------------
# guard bands: attention, paged attention, compaction
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("B,N,D,prefix", [(1, 1, 64, 0), (3, 7, 64, 5), (2, 64, 128, 131),
                                          (5, 13, 128, 0)])
def test_guard_bands_attention(dev, B, N, D, prefix):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    cfg = W.config("eagle_vicuna7b", B=B, N=N, depth=min(6, max(1, N - 1)), width=16, Hq=4,
                   Hkv=2, D=D, prefix=("fixed", prefix))
    case = W.make_attention_case(cfg, seed=3, lmax_pad=3)
    Hq, Hkv = cfg.Hq, cfg.Hkv
    g = {"out": Guarded((B, N, Hq, D), torch.bfloat16, dev),
         "lse": Guarded((B, Hq, N), torch.float32, dev),
         "status": Guarded((B,), torch.int32, dev, fill=0)}
    st.spec_tree_attention(_t(case.q, dev).view(torch.bfloat16),
                           _t(case.k_cache, dev).view(torch.bfloat16),
                           _t(case.v_cache, dev).view(torch.bfloat16), _t(case.prefix_lens, dev),
                           _t(case.tree_parent, dev), softmax_scale=case.scale, out=g["out"].t,
                           out_lse=g["lse"].t, status=g["status"].t)
    _assert_intact(g)
    assert int(g["status"].t.abs().sum()) == 0
    ref, ref_lse = P.oracle_attention(case)
    err = P.compare_attention(g["out"].t.float().cpu().numpy(), g["lse"].t.cpu().numpy(), ref,
                              ref_lse)
    assert err[0] <= P.ATTN_MAX_ABS and err[1] <= P.ATTN_REL_L2


@pytest.mark.parametrize("page", [16, 64])
def test_guard_bands_paged_attention_and_compaction(dev, page):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    B, N = 3, 9
    cfg = W.config("eagle_vicuna7b", B=B, N=N, depth=3, width=4, Hq=4, Hkv=2, D=64,
                   prefix=("uniform", 0, 40))
    pc = W.make_paged_attention_case(cfg, page, seed=5)
    g = {"out": Guarded((B, N, 4, 64), torch.bfloat16, dev),
         "lse": Guarded((B, 4, N), torch.float32, dev),
         "status": Guarded((B,), torch.int32, dev, fill=0)}
    st.spec_tree_attention_paged(_t(pc.q, dev).view(torch.bfloat16),
                                 _t(pc.k_pages, dev).view(torch.bfloat16),
                                 _t(pc.v_pages, dev).view(torch.bfloat16), _t(pc.block_table, dev),
                                 _t(pc.prefix_lens, dev), _t(pc.tree_parent, dev),
                                 softmax_scale=pc.scale, out=g["out"].t, out_lse=g["lse"].t,
                                 status=g["status"].t)
    _assert_intact(g)
    assert int(g["status"].t.abs().sum()) == 0
    # compaction of a path per sequence on the same pages (in place), and on a contiguous cache
    nodes = np.full((B, N), -1, np.int32)
    lens = np.array([0, 2, 3], np.int32)
    nodes[1, :2] = [1, 4]
    nodes[2, :3] = [2, 5, 8]
    kp = Guarded(pc.k_pages.shape, torch.bfloat16, dev)
    vp = Guarded(pc.v_pages.shape, torch.bfloat16, dev)
    kp.t.copy_(_t(pc.k_pages, dev).view(torch.bfloat16))
    vp.t.copy_(_t(pc.v_pages, dev).view(torch.bfloat16))
    gc = {"k_pages": kp, "v_pages": vp, "new_lens": Guarded((B,), torch.int32, dev),
          "status": Guarded((B,), torch.int32, dev, fill=0)}
    st.spec_kv_compact_paged(kp.t, vp.t, _t(pc.block_table, dev), _t(pc.prefix_lens, dev),
                             _t(lens, dev), _t(nodes, dev), new_prefix_lens=gc["new_lens"].t,
                             status=gc["status"].t)
    _assert_intact(gc)
    assert int(gc["status"].t.abs().sum()) == 0
    np.testing.assert_array_equal(gc["new_lens"].t.cpu().numpy(), pc.prefix_lens + 1 + lens)
    cc = W.make_compaction_case(B, N, 2, 64, seed=6, lens=lens)
    cc.accepted_nodes[:] = nodes
    kc = Guarded(cc.k_cache.shape, torch.bfloat16, dev)
    vc = Guarded(cc.v_cache.shape, torch.bfloat16, dev)
    kc.t.copy_(_t(cc.k_cache, dev).view(torch.bfloat16))
    vc.t.copy_(_t(cc.v_cache, dev).view(torch.bfloat16))
    gk = {"k_cache": kc, "v_cache": vc, "new_lens": Guarded((B,), torch.int32, dev),
          "status": Guarded((B,), torch.int32, dev, fill=0)}
    st.spec_kv_compact(kc.t, vc.t, _t(cc.prefix_lens, dev), _t(lens, dev), _t(nodes, dev),
                       new_prefix_lens=gk["new_lens"].t, status=gk["status"].t)
    _assert_intact(gk)
    assert int(gk["status"].t.abs().sum()) == 0


# ------------------------------------------------------------------------------------------------
# guard bands: verification (plain, filtered, greedy from argmaxes, without workspace)
# ------------------------------------------------------------------------------------------------
def _verify_cfg(B, N, V):
    if N <= 5:
        return W.config("tiny", B=B, N=N, depth=max(1, N - 1), V=V)
    depth = min(6, N - 1)
    return W.config("eagle_vicuna7b", B=B, N=N, depth=depth, width=-(-(N - 1) // depth) + 1, V=V)


def _verify_guards(B, N, V, ws_bytes, dev):
    import torch
    return {"accept_len": Guarded((B,), torch.int32, dev),
            "accepted_tokens": Guarded((B, N), torch.int32, dev),
            "bonus": Guarded((B,), torch.int32, dev),
            "accepted_nodes": Guarded((B, N), torch.int32, dev),
            "child_q": Guarded((B, N), torch.float32, dev),
            "status": Guarded((B,), torch.int32, dev, fill=0),
            "workspace": Guarded((max(ws_bytes, 16),), torch.uint8, dev)}


def _outs(g):
    return {k: v.t for k, v in g.items() if k not in ("status", "workspace")}


@pytest.mark.parametrize("B,N,V", [(1, 1, 1), (3, 5, 3), (3, 20, 517), (5, 1, 517), (2, 64, 1000)])
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_guard_bands_verify(dev, B, N, V, T):
    import speculative_decoding_token_spec_gb300 as st
    case = W.make_verify_case(_verify_cfg(B, N, V), T, seed=9)
    t = lambda a: _t(a, dev)  # noqa: E731
    g = _verify_guards(B, N, V, st.spec_tree_verify_workspace(B, N, V), dev)
    st.spec_tree_verify(t(case.target_logits), t(case.draft_probs), t(case.tree_tokens),
                        t(case.tree_parent), t(case.uniforms), T, outputs=_outs(g),
                        workspace=g["workspace"].t, status=g["status"].t, want_child_q=True)
    _assert_intact(g)
    got = {k: v.t.cpu().numpy() for k, v in g.items() if k != "workspace"}
    P.compare_verify(got, P.oracle_verify(case), case)
    # filtered verification: its workspace also holds the filtered logits
    if T > 0 and V > 1:
        gf = _verify_guards(B, N, V, st.spec_tree_verify_filtered_workspace(B, N, V), dev)
        st.spec_tree_verify_filtered(t(case.target_logits), t(case.draft_probs),
                                     t(case.tree_tokens), t(case.tree_parent), t(case.uniforms),
                                     T, top_k=max(1, V // 3), top_p=0.8, outputs=_outs(gf),
                                     workspace=gf["workspace"].t, status=gf["status"].t,
                                     want_child_q=True)
        _assert_intact(gf)
    # without a workspace argument
    gn = _verify_guards(B, N, V, 16, dev)
    del gn["workspace"]
    st.spec_tree_verify_noalloc(t(case.target_logits), t(case.draft_probs), t(case.tree_tokens),
                                t(case.tree_parent), t(case.uniforms), T, outputs=_outs(gn),
                                status=gn["status"].t)
    _assert_intact(gn)
    for k in ("accept_len", "accepted_tokens", "bonus", "accepted_nodes"):
        np.testing.assert_array_equal(gn[k].t.cpu().numpy(), got[k], err_msg=k)


@pytest.mark.parametrize("B,N,V", [(1, 1, 1), (3, 5, 3), (7, 20, 517)])
def test_guard_bands_greedy_from_argmax(dev, B, N, V):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    case = W.make_verify_case(_verify_cfg(B, N, V), 0.0, seed=12)
    argmax = np.argmax(case.target_logits, axis=2).astype(np.int32)
    g = _verify_guards(B, N, V, 16, dev)
    del g["workspace"], g["child_q"]
    st.spec_tree_verify_greedy(_t(argmax, dev), _t(case.tree_tokens, dev),
                               _t(case.tree_parent, dev), V, outputs=_outs(g),
                               status=g["status"].t)
    _assert_intact(g)
    ref = P.oracle_verify(case, with_table=False)
    np.testing.assert_array_equal(g["accept_len"].t.cpu().numpy(), ref["accept_len"])
    np.testing.assert_array_equal(g["bonus"].t.cpu().numpy(), ref["bonus"])
    del torch


# ------------------------------------------------------------------------------------------------
# guard bands: tree construction and the fused LM head
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("B,K,D,V,N", [(1, 1, 1, 1, 1), (3, 3, 2, 517, 7), (2, 5, 3, 1000, 31)])
def test_guard_bands_tree_build(dev, B, K, D, V, N):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    tc = W.make_tree_build_case(B, K, D, V, seed=4)
    ws = Guarded((st.spec_tree_build_workspace(B, K, D),), torch.uint8, dev)
    g = {"workspace": ws, "ft": Guarded((B, K), torch.int32, dev),
         "fs": Guarded((B, K), torch.int32, dev),
         "status": Guarded((B,), torch.int32, dev, fill=0)}
    for d in range(1, D + 1):
        st.spec_tree_expand(_t(tc.level_rows(d), dev), K, D, d, ws.t,
                            frontier_tokens=g["ft"].t, frontier_parent_slot=g["fs"].t,
                            status=g["status"].t)
    n = min(N, 1 + K + (D - 1) * K * K)
    out = {k: Guarded((B, n), torch.int32, dev) for k in ("tree_tokens", "tree_parent",
                                                          "node_row")}
    out["node_value"] = Guarded((B, n), torch.float32, dev)
    st.spec_tree_finalize(ws.t, _t(tc.root_tokens, dev), K, D, n,
                          outputs={k: v.t for k, v in out.items()}, status=g["status"].t)
    g.update(out)
    _assert_intact(g)
    assert int(g["status"].t.abs().sum()) == 0


@pytest.mark.parametrize("M,H,V,G", [(1, 64, 1, 1), (3, 136, 517, 3), (130, 512, 1000, 2)])
def test_guard_bands_lm_head(dev, M, H, V, G):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    lc = W.make_lm_head_case(M, H, V, G, seed=8)
    hid = _t(lc.hidden, dev).view(torch.bfloat16)
    w = _t(lc.weight, dev).view(torch.bfloat16)
    g = {"max": Guarded((M,), torch.float32, dev), "sumexp": Guarded((M,), torch.float32, dev),
         "argmax": Guarded((M,), torch.int32, dev), "gather": Guarded((M, G), torch.float32, dev),
         "workspace": Guarded((max(st.spec_lm_head_stats_workspace(M, V), 16),), torch.uint8,
                              dev),
         "status": Guarded((1,), torch.int32, dev, fill=0)}
    outs = {k: g[k].t for k in ("max", "sumexp", "argmax", "gather")}
    st.spec_lm_head_stats(hid, w, 1.0, gather_idx=_t(lc.gather_idx, dev), outputs=outs,
                          workspace=g["workspace"].t, status=g["status"].t)
    _assert_intact(g)
    ref = {k: v.clone() for k, v in outs.items()}
    packed = Guarded((st.spec_lm_head_packed_bytes(V, H),), torch.uint8, dev)
    st.spec_lm_head_pack(w, packed=packed.t)
    g2 = {"packed": packed, "max": Guarded((M,), torch.float32, dev),
          "sumexp": Guarded((M,), torch.float32, dev), "argmax": Guarded((M,), torch.int32, dev),
          "gather": Guarded((M, G), torch.float32, dev),
          "workspace": Guarded((max(st.spec_lm_head_stats_workspace(M, V), 16),), torch.uint8,
                               dev),
          "status": Guarded((1,), torch.int32, dev, fill=0)}
    outs2 = {k: g2[k].t for k in ("max", "sumexp", "argmax", "gather")}
    st.spec_lm_head_stats(hid, packed.t, 1.0, gather_idx=_t(lc.gather_idx, dev), outputs=outs2,
                          workspace=g2["workspace"].t, status=g2["status"].t, packed_vocab=V)
    _assert_intact(g2)
    for k in ("max", "sumexp", "argmax"):
        assert torch.equal(outs2[k], ref[k]), k
    assert int(g["status"].t.item()) == 0 and int(g2["status"].t.item()) == 0


# ------------------------------------------------------------------------------------------------
# stale workspace contents
# ------------------------------------------------------------------------------------------------
def _stale_words(n, rng):
    """Words an arrival counter could be mistaken for: a leaf's node record (first_acc = -1,
    nrej = 0), all ones, a count of 0xFFFF or N.. under many generations in the old and the
    current layout, and random bits."""
    tag = 0x5EC7
    pats = [0x00000000FFFFFFFF, 0xFFFFFFFFFFFFFFFF, 0]
    for gen in range(0, 4096, 3):
        pats.append((gen << 16) | 0xFFFF)                       # generation << 16 | count
        pats.append((gen << 32) | (tag << 16) | 0xFFFF)         # tagged, count >= any N
        pats.append((gen << 32) | (tag << 16) | 64)
    w = np.array(pats, dtype=np.uint64)
    reps = int(np.ceil(n / len(w)))
    out = np.concatenate([np.tile(w, reps)[:n // 2],
                          rng.integers(0, 2**63, size=n - n // 2, dtype=np.int64).astype(np.uint64)])
    rng.shuffle(out)
    return out.view(np.int64)


def test_stale_workspace_contents_are_ignored(dev):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    rng = np.random.default_rng(5)
    plan = [(12, 1.0), (5, 1.0), (6, 0.0), (1, 1.0), (12, 1.0), (3, 0.0)]
    cases = [W.make_verify_case(W.config("eagle_vicuna7b", B=B, V=3001), T, seed=60 + i)
             for i, (B, T) in enumerate(plan)]
    nbytes = max(st.spec_tree_verify_workspace(*c.target_logits.shape) for c in cases)
    ws = torch.empty((nbytes // 8 + 2,), dtype=torch.int64, device=dev)
    t = lambda a: _t(a, dev)  # noqa: E731
    for refill in (True, False):
        ws.copy_(torch.from_numpy(_stale_words(ws.numel(), rng)).to(dev))
        for case in cases:
            if refill:
                ws.copy_(torch.from_numpy(_stale_words(ws.numel(), rng)).to(dev))
            got = st.spec_tree_verify(t(case.target_logits), t(case.draft_probs),
                                      t(case.tree_tokens), t(case.tree_parent), t(case.uniforms),
                                      case.temperature, workspace=ws.view(torch.uint8))
            ref = P.run_verify_gpu(case, dev, want_child_q=False)
            for k in ("accept_len", "accepted_tokens", "bonus", "accepted_nodes", "status"):
                np.testing.assert_array_equal(got[k].cpu().numpy(), ref[k], err_msg=k)


# ------------------------------------------------------------------------------------------------
# the timeout path of the verification kernels
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("B,V,T,child_q", [(2, 32000, 1.0, True), (3, 32000, 0.0, False),
                                           (16, 32000, 1.0, False), (16, 32000, 1.0, True),
                                           (16, 32000, 0.0, False)])
def test_verify_wait_timeout_is_reported_and_leaves_no_trace(dev, B, V, T, child_q):
    """Small problems (every node at once) and large ones (B = 16: 123 MB of logits; the path
    form, and every internal node when per-child q is asked for)."""
    import speculative_decoding_token_spec_gb300 as st
    case = W.make_verify_case(W.config("eagle_vicuna7b", B=B, V=V), T, seed=70)
    before = P.run_verify_gpu(case, dev, want_child_q=child_q)
    assert (before["status"] == 0).all()
    try:
        st.spec_debug_set_verify_wait_polls(0)
        flagged = P.run_verify_gpu(case, dev, want_child_q=child_q)
    finally:
        st.spec_debug_set_verify_wait_polls(-1)
    assert (flagged["status"] & 16).all(), flagged["status"]
    assert (flagged["accept_len"] == -1).all() and (flagged["bonus"] == -1).all()
    assert (flagged["accepted_tokens"] == -1).all()
    after = P.run_verify_gpu(case, dev, want_child_q=child_q)
    for k in before:
        np.testing.assert_array_equal(after[k], before[k], err_msg=k)
