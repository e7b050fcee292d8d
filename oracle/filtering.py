"""Oracle: top-k / top-p filtered target distributions, in float64 (test infrastructure).

Pages followed: survey explainer, "Token Tree verification" / sampling paragraph of the
verification taxonomy (speculative sampling carries over to top-k and top-p sampling: the target
distribution that the accept/reject test and the residual use is the filtered one).

Readings (the pages give no procedure):

* Order: temperature first, then top-k on the logits, then top-p on the renormalised top-k
  distribution q_k = softmax(l / T) restricted to the top-k set.
* Top-k keeps every token whose logit is >= the k-th largest logit (ties at the boundary are all
  kept).  k <= 0 or k >= V: no top-k.
* Top-p keeps token y when the q_k-mass of the tokens strictly more probable than y is < top_p
  (ties are kept or dropped together; the most probable token is always kept).  top_p >= 1: no
  top-p.  At T = 0 neither filter changes anything (the argmax is always kept), so both are off.
* The filtered target distribution is softmax(l / T) over the kept tokens, renormalised; the
  draft distribution p is the caller's (already filtered by the drafter).

The filtered logits (-inf outside the kept set) fed to ``oracle.verify.tree_verify`` give exactly
that distribution, so verification itself is unchanged.
"""
from __future__ import annotations

import numpy as np


def keep_mask(logits_row, T: float, top_k: int, top_p: float):
    """Boolean mask of the kept tokens of one row (float64 arithmetic)."""
    l = np.asarray(logits_row, dtype=np.float64)
    V = l.shape[0]
    keep = np.ones(V, dtype=bool)
    if T <= 0:
        return keep
    if 0 < top_k < V:
        kth = np.sort(l)[::-1][top_k - 1]
        keep &= l >= kth
    if top_p < 1.0:
        lk = np.where(keep, l, -np.inf)
        m = lk.max()
        e = np.where(keep, np.exp((lk - m) / T), 0.0)
        q = e / e.sum()
        # mass of the strictly more probable tokens, per token
        order = np.argsort(-q, kind="stable")
        qs = q[order]
        csum = np.cumsum(qs)
        gt = np.full(V, np.inf)
        i = 0
        while i < V:
            above = csum[i - 1] if i > 0 else 0.0
            if above >= top_p:   # masses above only grow along the order: the rest is dropped
                break
            j = i
            while j + 1 < V and qs[j + 1] == qs[i]:
                j += 1
            gt[order[i:j + 1]] = above
            i = j + 1
        keep &= gt < top_p
    return keep


def filter_logits(logits, T: float, top_k: int, top_p: float):
    """[..., V] -> float64 logits with -inf outside each row's kept set."""
    l = np.asarray(logits, dtype=np.float64)
    out = np.empty_like(l)
    flat_in, flat_out = l.reshape(-1, l.shape[-1]), out.reshape(-1, l.shape[-1])
    for r in range(flat_in.shape[0]):
        k = keep_mask(flat_in[r], T, top_k, top_p)
        flat_out[r] = np.where(k, flat_in[r], -np.inf)
    return out


def top_p_margin(logits_row, T: float, top_k: int, top_p: float) -> float:
    """Distance of top_p to the nearest boundary mass (for near-tie accounting): min over the
    distinct probabilities v of |mass(q > v) - top_p|.  inf when top-p is off."""
    l = np.asarray(logits_row, dtype=np.float64)
    if T <= 0 or top_p >= 1.0:
        return np.inf
    keep = keep_mask(l, T, top_k, 1.0)
    lk = np.where(keep, l, -np.inf)
    e = np.where(keep, np.exp((lk - lk.max()) / T), 0.0)
    q = np.sort(e / e.sum())[::-1]
    q = q[q > 0]
    vals, starts = np.unique(-q, return_index=True)
    csum = np.concatenate([[0.0], np.cumsum(q)])
    gts = csum[starts]
    return float(np.min(np.abs(gts - top_p)))
