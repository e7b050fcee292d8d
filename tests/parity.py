"""Shared helpers of the GPU parity tests: run the C-ABI path and the CPU oracle on the same
seeded inputs and compare them with the stated tolerances."""
from __future__ import annotations

import numpy as np

from oracle import attention as OA
from oracle import verify as OV
from speculative_decoding_token_spec_gb300 import workloads as W

ATTN_MAX_ABS = 2e-2     # bf16 inputs, fp32 accumulation
ATTN_REL_L2 = 1e-2
LSE_ABS = 1e-3
CHILD_Q_ABS = 1e-5      # probabilities
NEAR_TIE = 1e-6         # fp64 decision margins below this are counted, not compared


def dev_tensor(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


# ------------------------------------------------------------------------------------------------
def run_attention_gpu(case: W.AttnCase, dev, status=None):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    B = case.q.shape[0]
    if status is None:
        status = torch.zeros(B, dtype=torch.int32, device=dev)
    out, lse, status = st.spec_tree_attention(
        dev_tensor(case.q, dev).view(torch.bfloat16),
        dev_tensor(case.k_cache, dev).view(torch.bfloat16),
        dev_tensor(case.v_cache, dev).view(torch.bfloat16),
        dev_tensor(case.prefix_lens, dev), dev_tensor(case.tree_parent, dev),
        softmax_scale=case.scale, status=status)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), status.cpu().numpy()


def oracle_attention(case: W.AttnCase, nodes=None):
    """Oracle on the bf16-rounded inputs; with ``nodes`` only those (b, i) pairs."""
    B = case.q.shape[0]
    if nodes is None:
        return OA.tree_attention(W.bf16_to_f64(case.q), W.bf16_to_f64(case.k_cache),
                                 W.bf16_to_f64(case.v_cache), case.prefix_lens,
                                 case.tree_parent, case.scale)
    _, N, Hq, D = case.q.shape
    out = np.full((B, N, Hq, D), np.nan)
    lse = np.full((B, Hq, N), np.nan)
    by_b = {}
    for b, i in nodes:
        by_b.setdefault(b, []).append(i)
    for b, idx in by_b.items():
        o, l = OA.tree_attention(W.bf16_to_f64(case.q[b:b + 1]),
                                 W.bf16_to_f64(case.k_cache[b:b + 1]),
                                 W.bf16_to_f64(case.v_cache[b:b + 1]), case.prefix_lens[b:b + 1],
                                 case.tree_parent[b:b + 1], case.scale,
                                 nodes=[(0, i) for i in idx])
        out[b, idx] = o[0, idx]
        lse[b, :, idx] = l[0][:, idx].T
    return out, lse


def compare_attention(got, got_lse, ref, ref_lse, mask=None):
    """Max-abs and rel-L2 over the compared rows; returns (max_abs, rel_l2, lse_max_abs)."""
    if mask is None:
        mask = ~np.isnan(ref[..., 0])
    g, r = got[mask], ref[mask]
    max_abs = float(np.abs(g - r).max())
    rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    lm = ~np.isnan(ref_lse)
    lse_err = float(np.abs(got_lse[lm] - ref_lse[lm]).max())
    return max_abs, rel, lse_err


# ------------------------------------------------------------------------------------------------
def run_verify_gpu(case: W.VerifyCase, dev, want_child_q=True, pass_probs=True):
    import torch
    import speculative_decoding_token_spec_gb300 as st
    B = case.target_logits.shape[0]
    status = torch.zeros(B, dtype=torch.int32, device=dev)
    res = st.spec_tree_verify(
        dev_tensor(case.target_logits, dev),
        dev_tensor(case.draft_probs, dev) if pass_probs else None,
        dev_tensor(case.tree_tokens, dev), dev_tensor(case.tree_parent, dev),
        dev_tensor(case.uniforms, dev), case.temperature, status=status,
        want_child_q=want_child_q)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in res.items()}


def oracle_verify(case: W.VerifyCase, with_table=True):
    return OV.tree_verify(case.target_logits, case.draft_probs, case.tree_tokens,
                          case.tree_parent, case.uniforms, case.temperature,
                          with_table=with_table)


def compare_verify(got, ref, case: W.VerifyCase, check_child_q=True):
    """Bit-exact comparison of the integer outputs except in near-tie sequences.

    Returns a dict of counters; raises AssertionError on a mismatch.
    """
    B, N, _ = case.target_logits.shape
    near = ref["near_tie"]
    np.testing.assert_array_equal(got["status"], ref["status"])
    checked = 0
    for b in range(B):
        if near[b]:
            continue
        checked += 1
        ctx = f"sequence {b}"
        assert got["accept_len"][b] == ref["accept_len"][b], ctx
        assert got["bonus"][b] == ref["bonus"][b], ctx
        np.testing.assert_array_equal(got["accepted_tokens"][b], ref["accepted_tokens"][b], ctx)
        if "accepted_nodes" in got:
            np.testing.assert_array_equal(got["accepted_nodes"][b], ref["accepted_nodes"][b], ctx)
    q_err = 0.0
    if check_child_q and "child_q" in got and case.temperature > 0:
        for b in range(B):
            if ref["status"][b]:
                continue
            kids = OV.children(case.tree_parent[b])
            for j, ks in kids.items():
                for pos, k in enumerate(ks):
                    rq = ref["child_q"][b, k]
                    if np.isnan(rq):
                        assert got["child_q"][b, k] == -1.0, (b, k)
                        continue
                    q_err = max(q_err, abs(float(got["child_q"][b, k]) - rq))
                    # a near-tie decision at this child may change the siblings after it
                    qx = rq
                    px = float(case.draft_probs[b, j, case.tree_tokens[b, k]])
                    r = float(case.uniforms[b, k])
                    if OV.decision_margin(r, qx, px) < NEAR_TIE:
                        break
        assert q_err <= CHILD_Q_ABS, f"child_q max-abs error {q_err}"
    return {"checked": checked, "near_ties": int(near.sum()), "child_q_err": q_err}
