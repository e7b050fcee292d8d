"""GPU parity of spec_tree_verify_filtered (top-k / top-p) against the oracle, through the C ABI.

* The filter kernel's output, read back from the workspace (the filtered logits start at the first
  16-byte boundary after the verification scratch): row for row, the kept logits carry the input's
  bits and the rest are -inf, with the kept set equal to oracle.filtering.keep_mask.  Top-k sets
  must match exactly; a top-p set may differ only in a row whose top_p lies within TOP_P_NEAR of
  the mass above a tie group (the kernel sums single-precision exponentials), and such rows are
  counted.
* The verification outputs against oracle.verify.tree_verify run on oracle.filtering.filter_logits:
  bit-exact outside near-tie sequences (fp64 decision margins below 1e-6, as for plain
  verification, or a top-p boundary row in the sequence); child q values to 1e-5.
* Special cases: top_k = 1 and a tiny top_p both reduce to greedy verification; filters that are
  off, and T = 0, give spec_tree_verify's outputs bit for bit; heavy ties at the boundaries, ragged
  vocabularies, -inf entries, NaN and +Inf rows.
"""
import numpy as np
import pytest

from oracle import filtering as OF
from oracle import verify as OV
from speculative_decoding_token_spec_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

TOP_P_NEAR = 4e-6


@pytest.fixture(scope="module")
def dev(cuda_lib):
    import torch
    return torch.device("cuda:0")


def _run(case, dev, top_k, top_p, want_child_q=True):
    """Filtered verification on the GPU; returns (outputs, filtered logits from the workspace)."""
    import torch
    import speculative_decoding_token_spec_gb300 as st
    B, N, V = case.target_logits.shape
    ws = torch.zeros(st.spec_tree_verify_filtered_workspace(B, N, V), dtype=torch.uint8,
                     device=dev)
    status = torch.zeros(B, dtype=torch.int32, device=dev)
    res = st.spec_tree_verify_filtered(
        P.dev_tensor(case.target_logits, dev), P.dev_tensor(case.draft_probs, dev),
        P.dev_tensor(case.tree_tokens, dev), P.dev_tensor(case.tree_parent, dev),
        P.dev_tensor(case.uniforms, dev), case.temperature, top_k=top_k, top_p=top_p,
        workspace=ws, status=status, want_child_q=want_child_q)
    torch.cuda.synchronize()
    off = -(-st.spec_tree_verify_workspace(B, N, V) // 16) * 16
    filt = ws[off:off + B * N * V * 4].view(torch.float32).view(B, N, V).cpu().numpy()
    return {k: v.cpu().numpy() for k, v in res.items()}, filt


def _check_filter(case, filt, top_k, top_p):
    """Row-by-row comparison of the filtered logits; returns the [B, N] mask of top-p near rows."""
    x = case.target_logits
    T = case.temperature
    B, N, _ = x.shape
    near = np.zeros((B, N), bool)
    for b in range(B):
        for j in range(N):
            row = x[b, j]
            if not np.isfinite(row[~np.isneginf(row)]).all():
                assert np.array_equal(filt[b, j].view(np.uint32), row.view(np.uint32)), (b, j)
                continue
            want = np.where(OF.keep_mask(row, T, top_k, top_p), row, np.float32(-np.inf))
            if np.array_equal(filt[b, j].view(np.uint32), want.astype(np.float32).view(np.uint32)):
                continue
            margin = OF.top_p_margin(row, T, top_k, top_p)
            assert margin < TOP_P_NEAR, (b, j, margin)
            near[b, j] = True
    return near


def _check(case, dev, top_k, top_p, want_child_q=True, max_near=None):
    got, filt = _run(case, dev, top_k, top_p, want_child_q)
    near_rows = _check_filter(case, filt, top_k, top_p)
    fl = OF.filter_logits(case.target_logits, case.temperature, top_k, top_p)
    fcase = W.VerifyCase(fl, case.draft_probs, case.tree_tokens, case.tree_parent, case.uniforms,
                         case.temperature)
    ref = P.oracle_verify(fcase, with_table=want_child_q)
    ref["near_tie"] = ref["near_tie"] | near_rows.any(axis=1)
    stats = P.compare_verify(got, ref, fcase, check_child_q=want_child_q and not near_rows.any())
    B = case.target_logits.shape[0]
    if max_near is None:
        max_near = max(1, B // 8)
    assert stats["near_ties"] <= max_near, stats
    kept = np.isfinite(fl).sum(axis=-1)
    ok = got["accept_len"] >= 0
    print(f"T={case.temperature} top_k={top_k} top_p={top_p}: {stats}, top-p near rows "
          f"{int(near_rows.sum())}, kept/row {kept.min()}..{kept.max()}, mean accept "
          f"{np.mean(got['accept_len'][ok]) if ok.any() else float('nan'):.2f}")
    return got, ref


@pytest.mark.parametrize("T", [1.0, 0.7])
@pytest.mark.parametrize("top_k,top_p", [(20, 1.0), (0, 0.9), (50, 0.8), (1000, 0.95), (5, 0.3)])
def test_eagle_tree_vicuna7b(dev, T, top_k, top_p):
    cfg = W.config("eagle_vicuna7b", B=2)
    _check(W.make_verify_case(cfg, T, seed=top_k + int(100 * top_p), sigma_d=0.3), dev, top_k,
           top_p)


def test_llama3_8b_gqa_vocab_128k(dev):
    cfg = W.config("llama3_8b_gqa", B=3)
    _check(W.make_verify_case(cfg, 0.7, seed=5, sigma_d=0.3), dev, 40, 0.95, want_child_q=False)


@pytest.mark.parametrize("B,N,V", [
    (3, 60, 12000),   # 180 rows of two 8192-element slices: one CTA per row, 32 per thread
    (1, 60, 50000),   # 60 rows of seven slices: four CTAs per row, 32 per thread
    (1, 30, 50000),   # 30 rows: one wave of eight CTAs per row, 16 per thread
])
def test_row_count_picks_the_cluster_shape(dev, B, N, V):
    """Many rows take half the CTAs per row with twice the elements per thread; the kept sets and
    the verification are the oracle's either way."""
    cfg = W.config("eagle_vicuna7b", B=B, N=N, V=V, depth=min(6, N - 1))
    _check(W.make_verify_case(cfg, 1.0, seed=V + N, sigma_d=0.3), dev, 40, 0.9)


def test_batched_sequences(dev):
    cfg = W.config("eagle_vicuna7b", B=24, V=4000)
    _check(W.make_verify_case(cfg, 1.0, seed=8, sigma_d=0.4), dev, 30, 0.85,
           want_child_q=False)


@pytest.mark.parametrize("top_k,top_p", [(1, 1.0), (0, 1e-4), (1, 0.5)])
def test_single_token_filters_walk_like_greedy(dev, top_k, top_p):
    """top_k = 1, or top_p below the largest probability, keep the argmax alone: the filtered
    target is one-hot, so the walk and the bonus token are greedy verification's."""
    cfg = W.config("eagle_vicuna7b", B=4, N=24, depth=4, width=8, V=3000)
    case = W.make_verify_case(cfg, 1.0, seed=3, sigma_d=0.3)
    got, _ = _run(case, dev, top_k, top_p, want_child_q=False)
    greedy = P.run_verify_gpu(W.VerifyCase(case.target_logits, None, case.tree_tokens,
                                           case.tree_parent, case.uniforms, 0.0), dev,
                              want_child_q=False, pass_probs=False)
    ref = OV.tree_verify(case.target_logits, None, case.tree_tokens, case.tree_parent,
                         case.uniforms, 0.0)
    for k in ("accept_len", "accepted_tokens", "bonus", "accepted_nodes", "status"):
        assert np.array_equal(got[k], greedy[k]), k
        assert np.array_equal(got[k], ref[k]), k


@pytest.mark.parametrize("T,top_k,top_p", [(1.0, 0, 1.0), (1.0, 3000, 1.0), (0.8, 5000, 1.0),
                                           (0.0, 5, 0.5)])
def test_inactive_filters_equal_plain_verify(dev, T, top_k, top_p):
    cfg = W.config("eagle_vicuna7b", B=3, N=30, depth=5, width=6, V=3000)
    case = W.make_verify_case(cfg, T, seed=6)
    got, _ = _run(case, dev, top_k, top_p)
    plain = P.run_verify_gpu(case, dev)
    for k in plain:
        assert np.array_equal(got[k].view(np.uint32) if got[k].dtype == np.float32 else got[k],
                              plain[k].view(np.uint32) if plain[k].dtype == np.float32
                              else plain[k]), k


@pytest.mark.parametrize("V", [1000, 4099, 517])
def test_ties_at_the_boundaries_and_ragged_vocab(dev, V):
    """Logits on a 0.5 grid: the k-th largest logit and the top-p boundary sit inside tie groups,
    which both filters keep or drop whole."""
    cfg = W.config("eagle_vicuna7b", B=3, N=20, depth=4, width=6, V=V)
    case = W.make_verify_case(cfg, 1.0, seed=V, sigma_d=0.3)
    case.target_logits[:] = np.round(case.target_logits * 2) / 2
    for top_k, top_p in ((7, 1.0), (0, 0.6), (25, 0.75), (V - 1, 0.99)):
        _check(case, dev, top_k, top_p)


def test_masked_entries_and_nonfinite_rows(dev):
    """-inf entries (a masked vocabulary) filter like any small logit; a row holding NaN or +Inf
    passes through unchanged and the verification flags its sequence."""
    cfg = W.config("eagle_vicuna7b", B=4, N=12, depth=3, width=4, V=2000)
    case = W.make_verify_case(cfg, 1.0, seed=12, sigma_d=0.3)
    rng = np.random.default_rng(12)
    mask = rng.random(case.target_logits.shape) < 0.3
    case.target_logits[mask] = -np.inf
    case.target_logits[1, 0, 5] = np.nan        # root rows are always read
    case.target_logits[2, 0, 9] = np.inf
    case.target_logits[3, 4, :] = -np.inf       # a row with nothing left (flagged if read)
    for top_k, top_p in ((10, 1.0), (0, 0.7), (100, 0.9)):
        got, filt = _run(case, dev, top_k, top_p, want_child_q=False)
        near = _check_filter(case, filt, top_k, top_p)
        assert got["status"][1] & 8 and got["status"][2] & 8
        fl = OF.filter_logits(case.target_logits[:1], 1.0, top_k, top_p)
        ref = OV.tree_verify(fl, case.draft_probs[:1], case.tree_tokens[:1],
                             case.tree_parent[:1], case.uniforms[:1], 1.0)
        if not (ref["near_tie"][0] or near[0].any()):
            assert got["status"][0] == 0
            assert got["accept_len"][0] == ref["accept_len"][0]
            assert got["bonus"][0] == ref["bonus"][0]
            assert np.array_equal(got["accepted_tokens"][0], ref["accepted_tokens"][0])


def test_argument_errors(dev):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    cfg = W.config("tiny")
    case = W.make_verify_case(cfg, 1.0, seed=0)
    args = [P.dev_tensor(a, dev) for a in (case.target_logits, case.draft_probs,
                                           case.tree_tokens, case.tree_parent, case.uniforms)]
    for top_k, top_p in ((-2, 0.9), (5, 0.0), (5, 1.01)):
        with pytest.raises(st.SpecError) as e:
            st.spec_tree_verify_filtered(*args, 1.0, top_k=top_k, top_p=top_p)
        assert e.value.code == -1
    small = torch.zeros(st.spec_tree_verify_workspace(1, 5, 1000), dtype=torch.uint8, device=dev)
    with pytest.raises(st.SpecError) as e:
        st.spec_tree_verify_filtered(*args, 1.0, top_k=5, top_p=1.0, workspace=small)
    assert e.value.code == -3
    # with the filters off the verification scratch alone suffices
    st.spec_tree_verify_filtered(*args, 1.0, top_k=0, top_p=1.0, workspace=small)
    torch.cuda.synchronize()


def test_large_threshold_bins_take_the_cluster_path(dev):
    """Thresholds inside a level-1 bin of more than 2048 elements (too many to gather): a very
    low temperature with a large k puts the k-th largest logit among the tail, a tie group of
    most of the vocabulary holds both thresholds, and a row of equal logits keeps everything."""
    cfg = W.config("eagle_vicuna7b", B=2, N=12, depth=3, width=4, V=32000)
    cold = W.make_verify_case(cfg, 0.05, seed=21, sigma_d=0.3)
    _check(cold, dev, 1000, 1.0)
    _check(cold, dev, 3000, 0.999)
    cfg = W.config("eagle_vicuna7b", B=3, N=12, depth=3, width=4, V=6000)
    case = W.make_verify_case(cfg, 1.0, seed=22, sigma_d=0.3)
    rng = np.random.default_rng(22)
    tie = rng.random(case.target_logits.shape) < 0.7
    case.target_logits[tie] = np.float32(1.0)
    case.target_logits[2] = np.float32(0.25)            # every row of sequence 2: one value
    for top_k, top_p in ((3000, 1.0), (0, 0.95), (3000, 0.9), (5999, 0.5)):
        _check(case, dev, top_k, top_p)
