"""Seeded synthetic inputs for the token-tree verification step.

This module only *draws inputs*: draft trees, draft tokens, KV caches, queries, target logits,
draft-model probabilities and the uniforms the method consumes.  It holds none of the
verification arithmetic (no tree-attention, no accept/reject, no residual, no sampling of the
bonus token); both the CUDA path and the CPU oracle are fed from here.

Shapes follow the workloads of the EAGLE paper explainer ("Static tree" section: a 60-node tree of
depth 6 with at most 10 nodes per level, Vicuna-7B) and of the speculative-decoding survey explainer
("Formal Definition": drafts are sampled from the draft distribution, one uniform per test).  The
pages measure on MT-bench / Spec-Bench with real models; those are not available, so these seeded
tensors stand in for them by shape and value distribution only.

Everything is numpy (PCG64 through ``default_rng`` seeded with integer lists, which is identical on
x86_64 and aarch64).  bf16 tensors are returned as ``uint16`` bit patterns (round-to-nearest-even
from float32) so that both sides read exactly the same values.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

__all__ = [
    "AttnCase", "VerifyCase", "PagedAttnCase", "CompactCase", "CONFIGS", "make_tree",
    "chain_tree", "make_attention_case", "make_paged_attention_case", "make_compaction_case",
    "make_verify_case", "bf16_bits", "bf16_to_f64", "config", "attention_layout",
    "HeadVerifyCase", "make_head_verify_case", "tree_depth",
]


# ----------------------------------------------------------------------------------------------
# bf16 bit handling (input preparation only)
# ----------------------------------------------------------------------------------------------
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round to bf16 (nearest-even, via float32) and return the uint16 bit patterns."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    u = bits.astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------------------------
# draft trees
# ----------------------------------------------------------------------------------------------
def chain_tree(n: int) -> np.ndarray:
    """Parent array of a chain: node i's parent is i-1, node 0 is the root (parent -1)."""
    par = np.arange(-1, n - 1, dtype=np.int32)
    return par


def make_tree(rng: np.random.Generator, n: int, depth: int, width_cap: int) -> np.ndarray:
    """Random static draft tree: the root plus ``n-1`` draft nodes on levels 1..depth.

    Every level starts with one node; the remaining nodes are added one at a time to a uniformly
    random level that is still below ``width_cap``.  Each node picks a uniformly random parent on
    the previous level.  Nodes are numbered level by level, and within a level by parent, so the
    numbering is breadth-first and every parent index is smaller than its child's.
    """
    if n < 1:
        raise ValueError("n must be >= 1")
    drafts = n - 1
    if drafts == 0:
        return np.array([-1], dtype=np.int32)
    depth = min(depth, drafts)
    if drafts > depth * width_cap:
        raise ValueError("tree does not fit the depth/width caps")
    widths = [1] * depth
    for _ in range(drafts - depth):
        open_levels = [lv for lv in range(depth) if widths[lv] < width_cap]
        widths[open_levels[int(rng.integers(len(open_levels)))]] += 1
    parent = [-1]
    prev = [0]
    for lv in range(depth):
        pars = sorted(int(prev[int(rng.integers(len(prev)))]) for _ in range(widths[lv]))
        first = len(parent)
        parent.extend(pars)
        prev = list(range(first, first + widths[lv]))
    return np.asarray(parent, dtype=np.int32)


# ----------------------------------------------------------------------------------------------
# configurations
# ----------------------------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    prefix: tuple          # ("fixed", L) or ("uniform", lo, hi)
    N: int
    tree: str              # "chain" or "static"
    depth: int
    width: int
    V: int
    sigma_t: float
    sigma_d: float
    temperatures: tuple
    qkv_fp32: bool = False  # the tiny case draws fp32 Q/K/V (rounded to bf16 for the kernels)
    cfg_id: int = 0


CONFIGS = {
    # CPU-seconds case: chain of 5 nodes (depth 4), vocab 1000.
    "tiny": Config("tiny", 1, 4, 4, 64, ("fixed", 128), 5, "chain", 4, 1, 1000, 2.0, 0.5,
                   (1.0,), qkv_fp32=True, cfg_id=1),
    # EAGLE static tree (60 nodes, depth 6, width <= 10) on a Vicuna-7B attention shape.
    "eagle_vicuna7b": Config("eagle_vicuna7b", 1, 32, 32, 128, ("fixed", 1024), 60, "static", 6,
                             10, 32000, 3.0, 1.0, (0.0, 1.0), cfg_id=2),
    # Batched LLaMA-3-8B-like GQA, prefixes uniform in [512, 4096].
    "llama3_8b_gqa": Config("llama3_8b_gqa", 16, 32, 8, 128, ("uniform", 512, 4096), 60, "static",
                            6, 10, 128256, 3.0, 1.5, (0.7,), cfg_id=3),
    # Long-context 70B-like GQA.  The target-logit spread is not stated for this shape; the
    # batched GQA shape's 3.0 is used.
    "llama70b_longctx": Config("llama70b_longctx", 4, 64, 8, 128, ("fixed", 32768), 60, "static",
                               6, 10, 128256, 3.0, 1.0, (1.0,), cfg_id=4),
    # Verification stress sweep (tree size, temperature and draft noise vary per case).
    "stress": Config("stress", 64, 32, 32, 128, ("fixed", 2048), 60, "static", 6, 10, 32000, 3.0,
                     1.0, (0.0, 0.5, 1.0, 1.5), cfg_id=5),
}


def config(name: str, **overrides) -> Config:
    return dataclasses.replace(CONFIGS[name], **overrides)


def _rng(seed: int, cfg_id: int, b: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(cfg_id), int(b), int(stream)])


def _prefix_lens(cfg: Config, seed: int) -> np.ndarray:
    if cfg.prefix[0] == "fixed":
        return np.full(cfg.B, cfg.prefix[1], dtype=np.int32)
    lo, hi = cfg.prefix[1], cfg.prefix[2]
    rng = _rng(seed, cfg.cfg_id, 10_000, 7)
    return rng.integers(lo, hi + 1, size=cfg.B).astype(np.int32)


def _tree(cfg: Config, seed: int, b: int) -> np.ndarray:
    if cfg.tree == "chain":
        return chain_tree(cfg.N)
    return make_tree(_rng(seed, cfg.cfg_id, b, 1), cfg.N, cfg.depth, cfg.width)


def attention_layout(cfg: Config, seed: int = 0):
    """The prefix lengths [B], trees [B, N] and cache length Lmax that make_attention_case draws for
    (cfg, seed), without the Q / K / V tensors (for callers that draw those elsewhere)."""
    lens = _prefix_lens(cfg, seed)
    par = np.stack([_tree(cfg, seed, b) for b in range(cfg.B)]).astype(np.int32)
    return lens, par, int(lens.max()) + cfg.N


# ----------------------------------------------------------------------------------------------
# attention inputs
# ----------------------------------------------------------------------------------------------
@dataclasses.dataclass
class AttnCase:
    q: np.ndarray             # uint16 bf16 bits [B, N, Hq, D]
    k_cache: np.ndarray       # uint16 bf16 bits [B, Hkv, Lmax, D]; node i's key at slot L_b + i
    v_cache: np.ndarray       # uint16 bf16 bits [B, Hkv, Lmax, D]
    prefix_lens: np.ndarray   # int32 [B]
    tree_parent: np.ndarray   # int32 [B, N]
    scale: float
    Lmax: int

    @property
    def shape(self):
        B, N, Hq, D = self.q.shape
        return B, N, Hq, self.k_cache.shape[1], D


def make_attention_case(cfg: Config, seed: int = 0, lmax_pad: int = 0,
                        prefix_lens: Optional[Sequence[int]] = None) -> AttnCase:
    """Q, K, V ~ N(0, 1) rounded to bf16; the tree's own keys sit right after each prefix."""
    B, N, Hq, Hkv, D = cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D
    lens = (np.asarray(prefix_lens, dtype=np.int32) if prefix_lens is not None
            else _prefix_lens(cfg, seed))
    Lmax = int(lens.max()) + N + int(lmax_pad)
    q = np.empty((B, N, Hq, D), dtype=np.uint16)
    k = np.empty((B, Hkv, Lmax, D), dtype=np.uint16)
    v = np.empty((B, Hkv, Lmax, D), dtype=np.uint16)
    par = np.empty((B, N), dtype=np.int32)
    for b in range(B):
        rng = _rng(seed, cfg.cfg_id, b, 2)
        q[b] = bf16_bits(rng.standard_normal((N, Hq, D), dtype=np.float32))
        k[b] = bf16_bits(rng.standard_normal((Hkv, Lmax, D), dtype=np.float32))
        v[b] = bf16_bits(rng.standard_normal((Hkv, Lmax, D), dtype=np.float32))
        par[b] = _tree(cfg, seed, b)
    return AttnCase(q, k, v, lens, par, 1.0 / float(np.sqrt(D)), Lmax)


@dataclasses.dataclass
class PagedAttnCase:
    q: np.ndarray             # uint16 bf16 bits [B, N, Hq, D]
    k_pages: np.ndarray       # uint16 bf16 bits [num_pages, Hkv, page_size, D]
    v_pages: np.ndarray       # uint16 bf16 bits [num_pages, Hkv, page_size, D]
    block_table: np.ndarray   # int32 [B, max_pages]: physical page of each logical page
    page_size: int
    prefix_lens: np.ndarray   # int32 [B]
    tree_parent: np.ndarray   # int32 [B, N]
    scale: float


def make_paged_attention_case(cfg: Config, page_size: int, seed: int = 0, spare_pages: int = 3,
                              prefix_lens: Optional[Sequence[int]] = None) -> PagedAttnCase:
    """Pages of N(0, 1) bf16 values and a block table that hands every sequence distinct physical
    pages in a random order (plus a few pages nobody uses).  Table entries past the pages a
    sequence needs are -1."""
    B, N, Hq, Hkv, D = cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D
    lens = (np.asarray(prefix_lens, dtype=np.int32) if prefix_lens is not None
            else _prefix_lens(cfg, seed))
    need = [(int(L) + N + page_size - 1) // page_size for L in lens]
    max_pages = max(need) + 1
    num_pages = sum(need) + int(spare_pages)
    rng = _rng(seed, cfg.cfg_id, 20_000, 3)
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    at = 0
    for b in range(B):
        table[b, :need[b]] = perm[at:at + need[b]]
        at += need[b]
    k = bf16_bits(rng.standard_normal((num_pages, Hkv, page_size, D), dtype=np.float32))
    v = bf16_bits(rng.standard_normal((num_pages, Hkv, page_size, D), dtype=np.float32))
    q = np.empty((B, N, Hq, D), dtype=np.uint16)
    par = np.empty((B, N), dtype=np.int32)
    for b in range(B):
        q[b] = bf16_bits(_rng(seed, cfg.cfg_id, b, 2).standard_normal((N, Hq, D), dtype=np.float32))
        par[b] = _tree(cfg, seed, b)
    return PagedAttnCase(q, k, v, table, page_size, lens, par, 1.0 / float(np.sqrt(D)))


@dataclasses.dataclass
class CompactCase:
    k_cache: np.ndarray       # uint16 bf16 bits [B, Hkv, Lmax, D]
    v_cache: np.ndarray
    prefix_lens: np.ndarray   # int32 [B]
    accept_len: np.ndarray    # int32 [B]: -1 (verification failed), 0 .. N-1
    accepted_nodes: np.ndarray  # int32 [B, N]: the accepted node ids, -1 padded


def make_compaction_case(B: int, N: int, Hkv: int, D: int, seed: int = 0,
                         prefix_range=(0, 200), lmax_pad: int = 5,
                         lens: Optional[Sequence[int]] = None) -> CompactCase:
    """Random caches and random accepted paths: for each sequence a length in -1 .. N-1 (or the
    given ``lens``) and that many distinct node ids in 1 .. N-1, increasing (the numbering of a
    root-to-node path when parents precede children)."""
    rng = np.random.default_rng([int(seed), 30_000, B, N])
    prefix = rng.integers(prefix_range[0], prefix_range[1] + 1, size=B).astype(np.int32)
    Lmax = int(prefix.max()) + N + int(lmax_pad)
    k = bf16_bits(rng.standard_normal((B, Hkv, Lmax, D), dtype=np.float32))
    v = bf16_bits(rng.standard_normal((B, Hkv, Lmax, D), dtype=np.float32))
    acc = (np.asarray(lens, dtype=np.int32) if lens is not None
           else rng.integers(-1, N, size=B).astype(np.int32))
    nodes = np.full((B, N), -1, dtype=np.int32)
    for b in range(B):
        ln = int(acc[b])
        if ln > 0:
            nodes[b, :ln] = np.sort(rng.choice(np.arange(1, N), size=ln, replace=False))
    return CompactCase(k, v, prefix, acc, nodes)


# ----------------------------------------------------------------------------------------------
# verification inputs
# ----------------------------------------------------------------------------------------------
@dataclasses.dataclass
class VerifyCase:
    target_logits: np.ndarray  # float32 [B, N, V]: row j = target logits after node j's path
    draft_probs: np.ndarray    # float32 [B, N, V]: row j = draft distribution at node j
    tree_tokens: np.ndarray    # int32 [B, N]: token of node i (node 0 = last committed token)
    tree_parent: np.ndarray    # int32 [B, N]
    uniforms: np.ndarray       # float32 [B, N]: [b, i>=1] test uniform r_i, [b, 0] resample u
    temperature: float

    @property
    def shape(self):
        return self.target_logits.shape


def _draft_distribution(draft_logits: np.ndarray, T: float) -> np.ndarray:
    """The synthetic draft model's output distribution at temperature T (T=0 uses T=1)."""
    t = T if T > 0 else 1.0
    z = draft_logits.astype(np.float64) / t
    z -= z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def make_verify_case(cfg: Config, T: float, seed: int = 0, sigma_d: Optional[float] = None,
                     tree_parent: Optional[np.ndarray] = None) -> VerifyCase:
    """Target logits ~ N(0, sigma_t^2); draft logits = target + N(0, sigma_d^2).

    Draft tokens: for T > 0 each draft node's token is an independent draw from its parent's draft
    distribution (siblings are i.i.d., with replacement).  For T = 0 the children of a node take the
    top-k tokens of the parent's draft logits in descending order, so siblings are distinct (when a
    node has more children than the vocabulary has tokens, the ranking wraps around).
    Uniforms are k / 2^24 with integer k, exact in float32 and always below 1.
    """
    B, N, V = cfg.B, cfg.N, cfg.V
    sd = cfg.sigma_d if sigma_d is None else float(sigma_d)
    tl = np.empty((B, N, V), dtype=np.float32)
    dp = np.empty((B, N, V), dtype=np.float32)
    tok = np.empty((B, N), dtype=np.int32)
    par = np.empty((B, N), dtype=np.int32)
    uni = np.empty((B, N), dtype=np.float32)
    for b in range(B):
        rng = _rng(seed, cfg.cfg_id, b, 3)
        pb = (np.asarray(tree_parent[b], dtype=np.int32) if tree_parent is not None
              else _tree(cfg, seed, b))
        par[b] = pb
        target = rng.standard_normal((N, V), dtype=np.float32) * np.float32(cfg.sigma_t)
        draft = target + rng.standard_normal((N, V), dtype=np.float32) * np.float32(sd)
        tl[b] = target
        p64 = _draft_distribution(draft, T)
        dp[b] = p64.astype(np.float32)
        tok[b, 0] = int(rng.integers(V))
        rank = np.zeros(N, dtype=np.int64)
        order_cache = {}
        for i in range(1, N):
            j = int(pb[i])
            if T > 0:
                cdf = np.cumsum(p64[j])
                x = float(rng.random()) * cdf[-1]
                tok[b, i] = int(min(np.searchsorted(cdf, x, side="right"), V - 1))
            else:
                if j not in order_cache:
                    order_cache[j] = np.argsort(-draft[j].astype(np.float64), kind="stable")
                tok[b, i] = int(order_cache[j][rank[j] % V])
                rank[j] += 1
        uni[b] = rng.integers(0, 1 << 24, size=N).astype(np.float32) / np.float32(1 << 24)
    return VerifyCase(tl, dp, tok, par, uni, float(T))


@dataclasses.dataclass
class TreeBuildCase:
    """Inputs of a dynamic tree construction: every level's draft rows, in the order the levels
    consume them (row 0: the root's; row 1 + (d - 2) K + i: frontier slot i's at level d)."""
    draft_rows: np.ndarray   # fp32 [B, 1 + (D - 1) K, V]
    root_tokens: np.ndarray  # int32 [B]
    K: int
    D: int

    def level_rows(self, d: int) -> np.ndarray:
        """Level d's rows, [B, 1, V] at d = 1, else [B, K, V] (a contiguous copy)."""
        if d == 1:
            return np.ascontiguousarray(self.draft_rows[:, :1])
        s = 1 + (d - 2) * self.K
        return np.ascontiguousarray(self.draft_rows[:, s:s + self.K])


def make_tree_build_case(B: int, K: int, D: int, V: int, seed: int = 0,
                         sigma: float = 3.0) -> TreeBuildCase:
    """Draft logits ~ N(0, sigma^2) per row, independent across rows (the draft model's rows for
    the frontier nodes; the construction does not depend on where they come from)."""
    rows = np.empty((B, 1 + (D - 1) * K, V), dtype=np.float32)
    roots = np.empty(B, dtype=np.int32)
    for b in range(B):
        rng = _rng(seed, 7, b, 11)
        rows[b] = rng.standard_normal((rows.shape[1], V), dtype=np.float32) * np.float32(sigma)
        roots[b] = int(rng.integers(V))
    return TreeBuildCase(rows, roots, K, D)


@dataclasses.dataclass
class HeadVerifyCase:
    """Inputs of verification from the nodes' hidden states and the LM head."""
    hidden: np.ndarray       # bf16 bits [B, N, H]: node i's final hidden state
    head: np.ndarray         # bf16 bits [V, H]
    draft_probs: np.ndarray  # float32 [B, N, V]
    tree_tokens: np.ndarray  # int32 [B, N]
    tree_parent: np.ndarray  # int32 [B, N]
    uniforms: np.ndarray     # float32 [B, N]
    temperature: float
    max_depth: int           # the deepest node's depth over the batch (root: 0)


def tree_depth(parent_row) -> int:
    """Depth of the deepest node of a valid tree (parents precede their children)."""
    d = [0] * len(parent_row)
    for i in range(1, len(parent_row)):
        d[i] = d[int(parent_row[i])] + 1
    return max(d)


def make_head_verify_case(cfg: Config, H: int, T: float, seed: int = 0,
                          sigma_d: Optional[float] = None,
                          tree_parent: Optional[np.ndarray] = None) -> HeadVerifyCase:
    """Hidden states and head on a small lattice, so that every logit hidden . w is exact in fp32
    whatever the order of the sums: hidden = a / 4 with integers a in [-3, 3], head = c / 2^s with
    integers c in [-7, 7] (|sum| <= 21 H < 2^24 units of 2^-(2+s)); s puts the logits' spread near
    cfg.sigma_t.

    The draft model follows the EAGLE explainer's design (its own feature prediction, read out by
    the target's LM head): draft logits = (hidden + noise) @ head^T in float64, the noise scaled so
    that the draft logits stray from the target's by about sigma_d.  Draft tokens and uniforms as
    in make_verify_case.
    """
    B, N, V = cfg.B, cfg.N, cfg.V
    sd = cfg.sigma_d if sigma_d is None else float(sigma_d)
    rng = _rng(seed, cfg.cfg_id, 0, 17)
    s = int(np.clip(np.round(np.log2(np.sqrt(H * 4.0 * 18.67) / 4.0 / cfg.sigma_t)), 0, 20))
    a = rng.integers(-3, 4, size=(B, N, H), dtype=np.int8)
    c = rng.integers(-7, 8, size=(V, H), dtype=np.int8)
    hidden_f = a.astype(np.float32) * np.float32(0.25)
    head_f = c.astype(np.float32) * np.float32(2.0 ** -s)
    hidden, head = bf16_bits(hidden_f), bf16_bits(head_f)
    wnorm = float(np.sqrt(np.mean(np.sum(np.square(head_f, dtype=np.float64), axis=1))))
    sigma_h = sd / max(wnorm, 1e-30)
    dp = np.empty((B, N, V), dtype=np.float32)
    tok = np.empty((B, N), dtype=np.int32)
    par = np.empty((B, N), dtype=np.int32)
    uni = np.empty((B, N), dtype=np.float32)
    head64 = head_f.astype(np.float64)
    for b in range(B):
        rb = _rng(seed, cfg.cfg_id, b, 19)
        pb = (np.asarray(tree_parent[b], dtype=np.int32) if tree_parent is not None
              else _tree(cfg, seed, b))
        par[b] = pb
        feat = hidden_f[b].astype(np.float64) + rb.standard_normal((N, H)) * sigma_h
        draft = feat @ head64.T
        p64 = _draft_distribution(draft, T)
        dp[b] = p64.astype(np.float32)
        tok[b, 0] = int(rb.integers(V))
        rank = np.zeros(N, dtype=np.int64)
        order_cache = {}
        for i in range(1, N):
            j = int(pb[i])
            if T > 0:
                cdf = np.cumsum(p64[j])
                x = float(rb.random()) * cdf[-1]
                tok[b, i] = int(min(np.searchsorted(cdf, x, side="right"), V - 1))
            else:
                if j not in order_cache:
                    order_cache[j] = np.argsort(-draft[j], kind="stable")
                tok[b, i] = int(order_cache[j][rank[j] % V])
                rank[j] += 1
        uni[b] = rb.integers(0, 1 << 24, size=N).astype(np.float32) / np.float32(1 << 24)
    depth = 0
    for b in range(B):
        pb = par[b]
        if pb[0] == -1 and all(0 <= pb[i] < i for i in range(1, N)):
            depth = max(depth, tree_depth(pb))
    return HeadVerifyCase(hidden, head, dp, tok, par, uni, float(T), depth)


@dataclasses.dataclass
class LmHeadCase:
    hidden: np.ndarray      # bf16 bits [M, H]
    weight: np.ndarray      # bf16 bits [V, H]
    gather_idx: np.ndarray  # int32 [M, G] (-1: none)


def make_lm_head_case(M: int, H: int, V: int, G: int = 0, seed: int = 0,
                      sigma: float = 3.0) -> LmHeadCase:
    """hidden ~ N(0, 1), weight ~ N(0, sigma^2 / H) (logits ~ N(0, sigma^2)), both rounded to
    bf16; gather ids uniform in [0, V) with one in eight set to -1."""
    rng = _rng(seed, 9, 0, 13)
    hidden = bf16_bits(rng.standard_normal((M, H), dtype=np.float32))
    weight = bf16_bits(rng.standard_normal((V, H), dtype=np.float32)
                       * np.float32(sigma / np.sqrt(H)))
    gi = rng.integers(0, V, size=(M, G)).astype(np.int32)
    gi[rng.random((M, G)) < 0.125] = -1
    return LmHeadCase(hidden, weight, gi)
