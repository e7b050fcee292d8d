"""GPU parity of the paged-cache attention and of post-accept KV compaction (through the C ABI).

* Paged attention against the fp64 oracle on the gathered cache (tolerance as for contiguous
  attention), and bit for bit against the contiguous kernel on the same values: the same chunks,
  the same arithmetic, only the addressing differs.
* Compaction against the oracle byte for byte (a copy), contiguous and paged, including moves
  whose destination is another move's source, failed verifications (len = -1), len = 0 and
  malformed paths (SPEC_ST_BAD_PATH, sequence unchanged).
"""
import numpy as np
import pytest

from oracle import paged as OP
from speculative_decoding_token_spec_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_lib):
    import torch
    return torch.device("cuda:0")


def _bf(x, dev):
    import torch
    return P.dev_tensor(x, dev).view(torch.bfloat16)


def _run_paged(case, dev):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    B = case.q.shape[0]
    status = torch.zeros(B, dtype=torch.int32, device=dev)
    out, lse, status = st.spec_tree_attention_paged(
        _bf(case.q, dev), _bf(case.k_pages, dev), _bf(case.v_pages, dev),
        P.dev_tensor(case.block_table, dev), P.dev_tensor(case.prefix_lens, dev),
        P.dev_tensor(case.tree_parent, dev), softmax_scale=case.scale, status=status)
    torch.cuda.synchronize()
    return out, lse, status.cpu().numpy()


def _sample_nodes(B, N, k, seed):
    rng = np.random.default_rng(seed)
    picks = {(int(rng.integers(B)), int(rng.integers(N))) for _ in range(k)}
    return sorted(picks | {(0, 0), (B - 1, N - 1)})


def _oracle_nodes(case, nodes):
    B, N, Hq, D = case.q.shape
    out = np.full((B, N, Hq, D), np.nan)
    lse = np.full((B, Hq, N), np.nan)
    q = W.bf16_to_f64(case.q)
    kp, vp = W.bf16_to_f64(case.k_pages), W.bf16_to_f64(case.v_pages)
    for b in sorted({b for b, _ in nodes}):
        idx = [i for bb, i in nodes if bb == b]
        o, l = OP.paged_tree_attention(q[b:b + 1], kp, vp, case.block_table[b:b + 1],
                                       case.page_size, case.prefix_lens[b:b + 1],
                                       case.tree_parent[b:b + 1], case.scale,
                                       nodes=[(0, i) for i in idx])
        out[b, idx] = o[0, idx]
        lse[b, :, idx] = l[0][:, idx].T
    return out, lse


@pytest.mark.parametrize("cfg,page_size", [("tiny", 16), ("tiny", 64),
                                           ("eagle_vicuna7b", 16), ("eagle_vicuna7b", 32),
                                           ("eagle_vicuna7b", 128), ("eagle_vicuna7b", 256),
                                           ("llama3_8b_gqa", 16)])
def test_paged_attention_matches_oracle(dev, cfg, page_size):
    case = W.make_paged_attention_case(W.config(cfg), page_size, seed=1)
    B, N = case.q.shape[:2]
    nodes = None if cfg == "tiny" else _sample_nodes(B, N, 6, seed=page_size)
    out, lse, status = _run_paged(case, dev)
    assert (status == 0).all(), status
    if nodes is None:
        nodes = [(b, i) for b in range(B) for i in range(N)]
    ref, ref_lse = _oracle_nodes(case, nodes)
    max_abs, rel, lse_err = P.compare_attention(out.float().cpu().numpy(), lse.cpu().numpy(),
                                                ref, ref_lse)
    print(f"{cfg} P={page_size}: max-abs {max_abs:.3e} rel-L2 {rel:.3e} lse {lse_err:.3e}")
    assert max_abs <= P.ATTN_MAX_ABS and rel <= P.ATTN_REL_L2 and lse_err <= P.LSE_ABS


@pytest.mark.parametrize("cfg,page_size", [("eagle_vicuna7b", 16), ("eagle_vicuna7b", 64),
                                           ("llama3_8b_gqa", 32), ("tiny", 16)])
def test_paged_equals_contiguous_bit_for_bit(dev, cfg, page_size):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    case = W.make_paged_attention_case(W.config(cfg), page_size, seed=2)
    out_p, lse_p, status = _run_paged(case, dev)
    assert (status == 0).all()
    lmax = case.block_table.shape[1] * page_size
    # the contiguous cache these pages stand for (the oracle's gather, on the bf16 bit patterns)
    kc = OP.gather_pages(case.k_pages.astype(np.float64), case.block_table, page_size, lmax)
    vc = OP.gather_pages(case.v_pages.astype(np.float64), case.block_table, page_size, lmax)
    kc = np.nan_to_num(kc, nan=0.0).astype(np.uint16)
    vc = np.nan_to_num(vc, nan=0.0).astype(np.uint16)
    out_c, lse_c, _ = st.spec_tree_attention(
        _bf(case.q, dev), _bf(kc, dev), _bf(vc, dev), P.dev_tensor(case.prefix_lens, dev),
        P.dev_tensor(case.tree_parent, dev), softmax_scale=case.scale)
    torch.cuda.synchronize()
    assert torch.equal(out_p.view(torch.int16), out_c.view(torch.int16))
    assert torch.equal(lse_p.view(torch.int32), lse_c.view(torch.int32))


def test_paged_missing_page_is_flagged(dev):
    case = W.make_paged_attention_case(W.config("eagle_vicuna7b"), 64, seed=3)
    L = int(case.prefix_lens[0])
    case.block_table[0, (L // 2) // 64] = -1                       # a prefix page
    case.block_table[0, (L + 59) // 64] = case.k_pages.shape[0] + 7  # the last tree page
    _, _, status = _run_paged(case, dev)
    assert status[0] & 32


# ------------------------------------------------------------------------------------------------
def _compact_gpu(cc, dev, paged=None):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    B = cc.prefix_lens.shape[0]
    status = torch.zeros(B, dtype=torch.int32, device=dev)
    if paged is None:
        k, v = _bf(cc.k_cache, dev), _bf(cc.v_cache, dev)
        lens, status = st.spec_kv_compact(k, v, P.dev_tensor(cc.prefix_lens, dev),
                                          P.dev_tensor(cc.accept_len, dev),
                                          P.dev_tensor(cc.accepted_nodes, dev), status=status)
    else:
        kp, vp, table = paged
        k, v = _bf(kp, dev), _bf(vp, dev)
        lens, status = st.spec_kv_compact_paged(k, v, P.dev_tensor(table, dev),
                                                P.dev_tensor(cc.prefix_lens, dev),
                                                P.dev_tensor(cc.accept_len, dev),
                                                P.dev_tensor(cc.accepted_nodes, dev),
                                                status=status)
    torch.cuda.synchronize()
    to_u16 = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    return to_u16(k), to_u16(v), lens.cpu().numpy(), status.cpu().numpy()


@pytest.mark.parametrize("D", [64, 128])
def test_compaction_matches_oracle(dev, D):
    cc = W.make_compaction_case(40, 60, 8, D, seed=D)
    cc.accept_len[:4] = [-1, 0, 59, 2]
    cc.accepted_nodes[2, :59] = np.arange(1, 60)        # every move overlaps the next one
    cc.accepted_nodes[3, :2] = [2, 3]
    k, v, lens, status = _compact_gpu(cc, dev)
    rk, rv, rlens, bad = OP.kv_compact(cc.k_cache, cc.v_cache, cc.prefix_lens, cc.accept_len,
                                       cc.accepted_nodes)
    assert not bad.any() and (status == 0).all()
    assert np.array_equal(k, rk) and np.array_equal(v, rv)
    assert np.array_equal(lens, rlens)


def test_compaction_rejects_malformed_paths(dev):
    cc = W.make_compaction_case(4, 10, 2, 128, seed=5, lens=[2, 2, 3, 9])
    cc.accepted_nodes[0, :2] = [4, 4]                   # not increasing
    cc.accepted_nodes[1, :2] = [0, 3]                   # the root
    cc.accepted_nodes[2, :3] = [1, 2, 10]               # node id >= N
    cc.prefix_lens[3] = cc.k_cache.shape[2] - 5         # L + 1 + len > Lmax
    k, v, lens, status = _compact_gpu(cc, dev)
    assert (status == 64).all(), status
    assert np.array_equal(k, cc.k_cache) and np.array_equal(v, cc.v_cache)
    assert np.array_equal(lens, cc.prefix_lens)


@pytest.mark.parametrize("page_size", [1, 16, 64])
def test_paged_compaction_matches_oracle(dev, page_size):
    cc = W.make_compaction_case(12, 60, 4, 128, seed=page_size, prefix_range=(0, 300))
    # pages for the compaction case: a random table over pages drawn as inputs
    rng = np.random.default_rng([page_size, 4])
    lmax = cc.k_cache.shape[2]
    max_pages = -(-lmax // page_size)
    num_pages = 12 * max_pages + 5
    table = rng.permutation(num_pages)[:12 * max_pages].reshape(12, max_pages).astype(np.int32)
    kp = W.bf16_bits(rng.standard_normal((num_pages, 4, page_size, 128), dtype=np.float32))
    vp = W.bf16_bits(rng.standard_normal((num_pages, 4, page_size, 128), dtype=np.float32))
    k, v, lens, status = _compact_gpu(cc, dev, paged=(kp, vp, table))
    rk, rv, rlens, bad = OP.kv_compact_paged(kp, vp, table, page_size, cc.prefix_lens,
                                             cc.accept_len, cc.accepted_nodes)
    assert not bad.any() and (status == 0).all()
    assert np.array_equal(k, rk) and np.array_equal(v, rv) and np.array_equal(lens, rlens)


def test_verify_then_compact_commits_the_accepted_path(dev):
    """End to end through the C ABI: spec_tree_verify's accepted nodes drive spec_kv_compact."""
    import torch
    import speculative_decoding_token_spec_gb300 as st
    cfg = W.config("eagle_vicuna7b", B=4, Hq=8, Hkv=8, V=4000)
    vc = W.make_verify_case(cfg, 1.0, seed=7, sigma_d=0.25)
    res = P.run_verify_gpu(vc, dev, want_child_q=False)
    ac = W.make_attention_case(cfg, seed=7)
    cc = W.CompactCase(ac.k_cache, ac.v_cache, ac.prefix_lens,
                       res["accept_len"].astype(np.int32), res["accepted_nodes"].astype(np.int32))
    k, v, lens, status = _compact_gpu(cc, dev)
    rk, rv, rlens, bad = OP.kv_compact(cc.k_cache, cc.v_cache, cc.prefix_lens, cc.accept_len,
                                       cc.accepted_nodes)
    assert (res["accept_len"] >= 0).all() and not bad.any() and (status == 0).all()
    assert np.array_equal(k, rk) and np.array_equal(lens, rlens)
