"""Oracle: paged KV cache and post-accept KV compaction, in float64 / exact copies (test
infrastructure).

Pages followed: survey explainer, "vLLMでの実装状況" section (serving stacks run speculative decoding
on PagedAttention, the KV cache split into fixed-size pages reached through a per-sequence table)
and its list of related methods ("KVキャッシュ圧縮", PagedAttention among them); EAGLE explainer,
vLLM usage section (tree verification needs extra KV-cache memory: the tree nodes' keys and values
sit in the cache beside the prefix during the verification step).

Readings (the pages give no layout):

* Paged layout.  Pages of P slots; ``pages[page, kv_head, row, :]``; sequence b's slot s lives in
  page ``block_table[b, s // P]`` at row ``s % P``.  The cache capacity per sequence is
  ``max_pages * P``.
* Compaction.  After verification accepted the path ``nodes[0..len-1]`` (node ids, root excluded),
  the root stays at slot L_b and the accepted nodes' keys and values move to slots
  L_b + 1 .. L_b + len in path order: slot L_b + 1 + k receives what slot L_b + nodes[k] held before
  the call.  The committed length becomes L_b + 1 + len.  A sequence whose verification failed
  (len = -1) keeps its cache and its length.

Everything here is the plain definition: gather by table lookup, copy from a snapshot.
"""
from __future__ import annotations

import numpy as np

from .attention import tree_attention


def gather_pages(pages: np.ndarray, block_table: np.ndarray, page_size: int,
                 num_slots: int) -> np.ndarray:
    """The contiguous cache [B, Hkv, num_slots, D] a paged cache stands for.

    Slots whose table entry is outside [0, num_pages) come out as NaN (a call never reads them).
    """
    num_pages, hkv, p, d = pages.shape
    if p != page_size:
        raise ValueError("page size mismatch")
    B = block_table.shape[0]
    out = np.full((B, hkv, num_slots, d), np.nan)
    for b in range(B):
        for s in range(num_slots):
            lp = s // page_size
            if lp >= block_table.shape[1]:
                continue
            page = int(block_table[b, lp])
            if 0 <= page < num_pages:
                out[b, :, s, :] = pages[page, :, s % page_size, :]
    return out


def paged_tree_attention(q, k_pages, v_pages, block_table, page_size, prefix_lens, tree_parent,
                         scale, nodes=None):
    """Tree attention over a paged cache: the contiguous definition on the gathered cache."""
    num_slots = block_table.shape[1] * page_size
    k = gather_pages(k_pages, block_table, page_size, num_slots)
    v = gather_pages(v_pages, block_table, page_size, num_slots)
    return tree_attention(q, k, v, prefix_lens, tree_parent, scale, nodes=nodes)


def valid_path(nodes_row, length: int, n: int) -> bool:
    """A committed path: node ids in [1, n), strictly increasing (parents precede children)."""
    prev = 0
    for k in range(length):
        x = int(nodes_row[k])
        if not (prev < x < n):
            return False
        prev = x
    return True


def kv_compact(k_cache, v_cache, prefix_lens, accept_len, accepted_nodes):
    """Contiguous cache [B, Hkv, Lmax, D]: returns (k, v, new_lens, bad) after compaction.

    ``bad[b]`` is True where the request was malformed (path not strictly increasing inside
    [1, N), or the committed length would exceed Lmax); such a sequence is left unchanged.
    """
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    B, _, lmax, _ = k_cache.shape
    n = accepted_nodes.shape[1]
    new_lens = np.array(prefix_lens, dtype=np.int64, copy=True)
    bad = np.zeros(B, dtype=bool)
    for b in range(B):
        L, ln = int(prefix_lens[b]), int(accept_len[b])
        if ln < 0:
            continue
        if ln > n - 1 or L < 0 or L + 1 + ln > lmax or not valid_path(accepted_nodes[b], ln, n):
            bad[b] = True
            continue
        for k in range(ln):
            src = L + int(accepted_nodes[b, k])
            k_out[b, :, L + 1 + k, :] = k_cache[b, :, src, :]
            v_out[b, :, L + 1 + k, :] = v_cache[b, :, src, :]
        new_lens[b] = L + 1 + ln
    return k_out, v_out, new_lens, bad


def kv_compact_paged(k_pages, v_pages, block_table, page_size, prefix_lens, accept_len,
                     accepted_nodes):
    """Paged cache: the same moves, each slot reached through the table.  Returns
    (k_pages, v_pages, new_lens, bad); a sequence whose table maps a moved slot outside
    [0, num_pages) is bad and left unchanged."""
    k_out = np.array(k_pages, copy=True)
    v_out = np.array(v_pages, copy=True)
    num_pages = k_pages.shape[0]
    B, max_pages = block_table.shape
    n = accepted_nodes.shape[1]
    lmax = max_pages * page_size
    new_lens = np.array(prefix_lens, dtype=np.int64, copy=True)
    bad = np.zeros(B, dtype=bool)

    def where(b, s):
        page = int(block_table[b, s // page_size])
        return (page, s % page_size) if 0 <= page < num_pages else None

    for b in range(B):
        L, ln = int(prefix_lens[b]), int(accept_len[b])
        if ln < 0:
            continue
        if ln > n - 1 or L < 0 or L + 1 + ln > lmax or not valid_path(accepted_nodes[b], ln, n):
            bad[b] = True
            continue
        moves = [(where(b, L + int(accepted_nodes[b, k])), where(b, L + 1 + k)) for k in range(ln)]
        if any(src is None or dst is None for src, dst in moves):
            bad[b] = True
            continue
        for (sp, sr), (dp, dr) in moves:
            k_out[dp, :, dr, :] = k_pages[sp, :, sr, :]
            v_out[dp, :, dr, :] = v_pages[sp, :, sr, :]
        new_lens[b] = L + 1 + ln
    return k_out, v_out, new_lens, bad
