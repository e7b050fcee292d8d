"""GPU parity of spec_tree_attention against the fp64 oracle (through the C ABI).

Tolerance (bf16 inputs, fp32 accumulation): max-abs error <= 2e-2 and rel-L2 <= 1e-2 on the
output; the log-sum-exp within 1e-3.  Full-size shapes compare sampled nodes (every head of each
sampled node) so the oracle stays within seconds.
"""
import numpy as np
import pytest

from speculative_decoding_token_spec_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_lib):
    import torch
    return torch.device("cuda:0")


def _check(case, dev, nodes=None):
    got, got_lse, status = P.run_attention_gpu(case, dev)
    assert (status == 0).all(), status
    ref, ref_lse = P.oracle_attention(case, nodes)
    max_abs, rel, lse_err = P.compare_attention(got, got_lse, ref, ref_lse)
    print(f"shape {case.shape} Lmax {case.Lmax}: max-abs {max_abs:.3e} rel-L2 {rel:.3e} "
          f"lse {lse_err:.3e}")
    assert max_abs <= P.ATTN_MAX_ABS and rel <= P.ATTN_REL_L2 and lse_err <= P.LSE_ABS
    return got


def _sample_nodes(case, k, seed):
    rng = np.random.default_rng(seed)
    B, N = case.q.shape[:2]
    picks = {(int(rng.integers(B)), int(rng.integers(N))) for _ in range(k)}
    picks |= {(0, 0), (B - 1, N - 1)}
    return sorted(picks)


def test_tiny_chain(dev):
    _check(W.make_attention_case(W.config("tiny"), seed=0), dev)


def test_eagle_static_tree_vicuna7b(dev):
    _check(W.make_attention_case(W.config("eagle_vicuna7b"), seed=0), dev)


def test_llama3_8b_gqa_ragged_prefixes(dev):
    case = W.make_attention_case(W.config("llama3_8b_gqa"), seed=0)
    _check(case, dev, nodes=_sample_nodes(case, 40, 1))


def test_llama70b_longctx(dev):
    case = W.make_attention_case(W.config("llama70b_longctx"), seed=0)
    _check(case, dev, nodes=_sample_nodes(case, 8, 2))


def test_stress_shape(dev):
    case = W.make_attention_case(W.config("stress"), seed=0)
    _check(case, dev, nodes=_sample_nodes(case, 24, 3))


# ------------------------------------------------------------------------------------------------
# edge cases
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("L", [0, 1, 63, 64, 65, 200])
def test_prefix_lengths_around_tile_edges(dev, L):
    cfg = W.config("eagle_vicuna7b", B=2, Hq=4, Hkv=2, N=20, depth=4, width=6)
    _check(W.make_attention_case(cfg, seed=L, prefix_lens=[L, L + 7], lmax_pad=5), dev)


def test_head_dim_64_gqa(dev):
    cfg = W.config("llama3_8b_gqa", B=3, Hq=16, Hkv=4, D=64, prefix=("uniform", 30, 300))
    _check(W.make_attention_case(cfg, seed=4), dev)


def test_root_only_tree_and_empty_prefix(dev):
    cfg = W.config("eagle_vicuna7b", B=2, Hq=4, Hkv=4, N=1)
    case = W.make_attention_case(cfg, seed=5, prefix_lens=[0, 3])
    got = _check(case, dev)
    # L = 0, N = 1: output equals the root's value row (bf16)
    v = W.bf16_to_f64(case.v_cache)[0, :, 0]
    np.testing.assert_allclose(got[0, 0], v, atol=1e-2)


def test_max_nodes_and_groups(dev):
    cfg = W.config("llama70b_longctx", B=2, Hq=32, Hkv=2, N=64, depth=7, width=10,
                   prefix=("fixed", 333))
    case = W.make_attention_case(cfg, seed=6)
    _check(case, dev, nodes=_sample_nodes(case, 30, 7))


def test_bad_tree_and_bad_length_flagged(dev):
    import torch
    cfg = W.config("eagle_vicuna7b", B=3, Hq=4, Hkv=4, N=8, depth=3, width=3)
    case = W.make_attention_case(cfg, seed=8, prefix_lens=[10, 20, 30])
    case.tree_parent[1, 3] = 5
    case.prefix_lens[2] = case.Lmax - 2   # prefix + N > Lmax
    got, _, status = P.run_attention_gpu(case, dev)
    assert status.tolist() == [0, 1, 2]
    assert (got[1] == 0).all() and (got[2] == 0).all()
    ref, _ = P.oracle_attention(W.AttnCase(case.q[:1], case.k_cache[:1], case.v_cache[:1],
                                           case.prefix_lens[:1], case.tree_parent[:1],
                                           case.scale, case.Lmax))
    assert np.abs(got[:1] - ref).max() <= P.ATTN_MAX_ABS
    torch.cuda.synchronize()


def test_slots_beyond_tree_do_not_leak(dev):
    cfg = W.config("eagle_vicuna7b", B=1, Hq=2, Hkv=2, N=9, depth=3, width=4)
    case = W.make_attention_case(cfg, seed=9, prefix_lens=[70], lmax_pad=100)
    a, _, _ = P.run_attention_gpu(case, dev)
    big = W.bf16_bits(np.full((2, 100, cfg.D), 300.0, dtype=np.float32))
    case.k_cache[0, :, 70 + 9:] = big
    case.v_cache[0, :, 70 + 9:] = big
    b, _, _ = P.run_attention_gpu(case, dev)
    np.testing.assert_array_equal(a, b)


def test_nan_in_unused_cache_slots(dev):
    # Slots past L_b + N (the rest of the last 64-key tile and beyond) may hold anything a cache
    # allocator left there, NaN included; none of it may reach the output.
    cfg = W.config("eagle_vicuna7b", B=2, Hq=4, Hkv=2, N=13, depth=4, width=5)
    case = W.make_attention_case(cfg, seed=10, prefix_lens=[150, 37], lmax_pad=300)
    a, la, _ = P.run_attention_gpu(case, dev)
    nan_bits = np.uint16(0x7FC0)
    for b, L in enumerate(case.prefix_lens):
        case.k_cache[b, :, L + cfg.N:] = nan_bits
        case.v_cache[b, :, L + cfg.N:] = nan_bits
    got = _check(case, dev)
    assert np.isfinite(got).all()
    b_, lb, _ = P.run_attention_gpu(case, dev)
    np.testing.assert_array_equal(a, b_)
    np.testing.assert_array_equal(la, lb)


@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (4, 1)])
@pytest.mark.parametrize("L", [0, 100, 300, 520, 1000])
def test_split_counts_single_head(dev, Hq, Hkv, L):
    # One KV head per launch: the planner spreads the key range over 1..8 split CTAs (one
    # cluster), with paired key groups (R = 60 <= 64) or one group (R = 240).
    cfg = W.config("eagle_vicuna7b", B=1, Hq=Hq, Hkv=Hkv, N=60)
    _check(W.make_attention_case(cfg, seed=L + Hq, prefix_lens=[L]), dev)


def test_deterministic_repeat(dev):
    case = W.make_attention_case(W.config("eagle_vicuna7b"), seed=12)
    a, la, _ = P.run_attention_gpu(case, dev)
    b, lb, _ = P.run_attention_gpu(case, dev)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)
