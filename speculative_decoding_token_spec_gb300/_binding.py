"""Thin ctypes binding of libspectree (argument marshalling only).

Each function takes torch CUDA tensors, checks dtypes / contiguity, allocates the outputs it is
not given (torch owns device memory), and calls the C entry point of the same name with raw
device pointers and the current CUDA stream.  Every step of the computation runs in the library's
kernels; if the library is missing or fails to load, these functions raise -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

from . import build as _build

_LIB = None
_LOCK = threading.Lock()

SPEC_OK = 0
ERRORS = {-1: "SPEC_ERR_INVALID_ARG", -2: "SPEC_ERR_UNSUPPORTED", -3: "SPEC_ERR_WORKSPACE",
          -4: "SPEC_ERR_CUDA"}
ST_BAD_TREE, ST_BAD_LEN, ST_BAD_TOKEN, ST_NONFINITE, ST_TIMEOUT = 1, 2, 4, 8, 16
ST_BAD_PAGE, ST_BAD_PATH = 32, 64


class SpecError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} returned {code} ({ERRORS.get(code, '?')}): "
                         f"{spec_status_string(code)}")


_c_int, _c_size, _vp, _c_float = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float

_SIGNATURES = {
    "spec_tree_attention_workspace": (_c_size, [_c_int] * 6),
    "spec_tree_attention": (_c_int, [_vp] * 7 + [_c_int] * 6 + [_c_float, _vp, _c_size, _vp, _vp]),
    "spec_tree_verify_workspace": (_c_size, [_c_int] * 3),
    "spec_tree_verify": (_c_int, [_vp] * 5 + [_c_float] + [_c_int] * 3 + [_vp] * 5
                         + [_vp, _c_size, _vp, _vp]),
    "spec_tree_attention_paged": (_c_int, [_vp] * 4 + [_c_int] * 3 + [_vp] * 4 + [_c_int] * 5
                                  + [_c_float, _vp, _vp]),
    "spec_kv_compact": (_c_int, [_vp] * 6 + [_c_int] * 5 + [_vp, _vp]),
    "spec_kv_compact_paged": (_c_int, [_vp] * 3 + [_c_int] * 3 + [_vp] * 4 + [_c_int] * 4
                              + [_vp, _vp]),
    "spec_tree_verify_filtered_workspace": (_c_size, [_c_int] * 3),
    "spec_tree_verify_filtered": (_c_int, [_vp] * 5 + [_c_float, _c_int, _c_float] + [_c_int] * 3
                                  + [_vp] * 5 + [_vp, _c_size, _vp, _vp]),
    "spec_tree_build_workspace": (_c_size, [_c_int] * 3),
    "spec_tree_expand": (_c_int, [_vp] + [_c_int] * 5 + [_vp, _c_size] + [_vp] * 4),
    "spec_tree_finalize": (_c_int, [_vp, _c_size, _vp] + [_c_int] * 4 + [_vp] * 6),
    "spec_lm_head_stats_workspace": (_c_size, [_c_int] * 2),
    "spec_lm_head_stats": (_c_int, [_vp] * 3 + [_c_int] * 4 + [_c_float] + [_vp] * 5
                           + [_c_size, _vp, _vp]),
    "spec_lm_head_packed_bytes": (_c_size, [_c_int] * 2),
    "spec_lm_head_pack": (_c_int, [_vp, _c_int, _c_int, _vp, _c_size, _vp]),
    "spec_lm_head_stats_packed": (_c_int, [_vp] * 3 + [_c_int] * 4 + [_c_float] + [_vp] * 5
                                  + [_c_size, _vp, _vp]),
    "spec_tree_verify_greedy": (_c_int, [_vp] * 3 + [_c_int] * 3 + [_vp] * 6),
    "spec_tree_verify_head_workspace": (_c_size, [_c_int] * 5),
    "spec_tree_verify_head": (_c_int, [_vp, _vp, _c_int] + [_vp] * 4 + [_c_float] + [_c_int] * 5
                              + [_vp] * 5 + [_c_size, _vp, _vp]),
    "spec_status_string": (ctypes.c_char_p, [_c_int]),
    "spec_debug_set_verify_wait_polls": (_c_int, [ctypes.c_longlong]),
}


def lib_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = True):
    """Load libspectree.so (building it first if it is absent)."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = lib_path()
            if not os.path.exists(path):
                if not build_if_missing:
                    raise RuntimeError(f"libspectree not built ({path} missing)")
                _build.build()
            handle = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype, fn.argtypes = res, args
            _LIB = handle
    return _LIB


def spec_status_string(code: int) -> str:
    try:
        return lib().spec_status_string(int(code)).decode()
    except Exception:  # pragma: no cover - only used inside error messages
        return ERRORS.get(code, "unknown")


# ----------------------------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check(t, name, dtype, shape, device):
    torch = _torch()
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device or t.device.type != "cuda":
        raise ValueError(f"{name} must live on {device}")
    return torch


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def spec_tree_attention_workspace(B, N, Hq, Hkv, D, Lmax) -> int:
    return int(lib().spec_tree_attention_workspace(B, N, Hq, Hkv, D, Lmax))


def spec_tree_verify_workspace(B, N, V) -> int:
    return int(lib().spec_tree_verify_workspace(B, N, V))


def spec_tree_attention(q, k_cache, v_cache, prefix_lens, tree_parent, softmax_scale=None,
                        out=None, out_lse=None, want_lse=True, workspace=None, status=None,
                        stream=None):
    """Tree-masked attention; returns (out bf16 [B,N,Hq,D], lse fp32 [B,Hq,N] or None, status)."""
    torch = _torch()
    B, N, Hq, D = q.shape
    _, Hkv, Lmax, _ = k_cache.shape
    dev = q.device
    _check(q, "q", torch.bfloat16, (B, N, Hq, D), dev)
    _check(k_cache, "k_cache", torch.bfloat16, (B, Hkv, Lmax, D), dev)
    _check(v_cache, "v_cache", torch.bfloat16, (B, Hkv, Lmax, D), dev)
    _check(prefix_lens, "prefix_lens", torch.int32, (B,), dev)
    _check(tree_parent, "tree_parent", torch.int32, (B, N), dev)
    if out is None:
        out = torch.empty((B, N, Hq, D), dtype=torch.bfloat16, device=dev)
    if out_lse is None and want_lse:
        out_lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    if status is None:
        status = torch.zeros((B,), dtype=torch.int32, device=dev)  # bits are OR-ed in
    ws_bytes = spec_tree_attention_workspace(B, N, Hq, Hkv, D, Lmax)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty((ws_bytes,), dtype=torch.uint8, device=dev)
    scale = (1.0 / math.sqrt(D)) if softmax_scale is None else float(softmax_scale)
    rc = lib().spec_tree_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(prefix_lens), _ptr(tree_parent), _ptr(out),
        _ptr(out_lse), B, N, Hq, Hkv, D, Lmax, scale, _ptr(workspace),
        0 if workspace is None else workspace.numel(), _ptr(status), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError("spec_tree_attention", rc)
    return out, out_lse, status


def spec_tree_attention_paged(q, k_pages, v_pages, block_table, prefix_lens, tree_parent,
                              softmax_scale=None, out=None, out_lse=None, want_lse=True,
                              status=None, stream=None):
    """Tree attention over a paged cache (pages [num_pages, Hkv, P, D], block_table [B,
    max_pages]); returns (out, lse or None, status) like spec_tree_attention."""
    torch = _torch()
    B, N, Hq, D = q.shape
    num_pages, Hkv, P, _ = k_pages.shape
    max_pages = block_table.shape[1]
    dev = q.device
    _check(q, "q", torch.bfloat16, (B, N, Hq, D), dev)
    _check(k_pages, "k_pages", torch.bfloat16, (num_pages, Hkv, P, D), dev)
    _check(v_pages, "v_pages", torch.bfloat16, (num_pages, Hkv, P, D), dev)
    _check(block_table, "block_table", torch.int32, (B, max_pages), dev)
    _check(prefix_lens, "prefix_lens", torch.int32, (B,), dev)
    _check(tree_parent, "tree_parent", torch.int32, (B, N), dev)
    if out is None:
        out = torch.empty((B, N, Hq, D), dtype=torch.bfloat16, device=dev)
    if out_lse is None and want_lse:
        out_lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    if status is None:
        status = torch.zeros((B,), dtype=torch.int32, device=dev)
    scale = (1.0 / math.sqrt(D)) if softmax_scale is None else float(softmax_scale)
    rc = lib().spec_tree_attention_paged(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), P, max_pages, num_pages,
        _ptr(prefix_lens), _ptr(tree_parent), _ptr(out), _ptr(out_lse), B, N, Hq, Hkv, D, scale,
        _ptr(status), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError("spec_tree_attention_paged", rc)
    return out, out_lse, status


def spec_kv_compact(k_cache, v_cache, prefix_lens, accept_len, accepted_nodes,
                    new_prefix_lens=None, status=None, stream=None):
    """Commit the accepted path in place (contiguous cache); returns (new_prefix_lens, status)."""
    torch = _torch()
    B, Hkv, Lmax, D = k_cache.shape
    N = accepted_nodes.shape[1]
    dev = k_cache.device
    _check(k_cache, "k_cache", torch.bfloat16, (B, Hkv, Lmax, D), dev)
    _check(v_cache, "v_cache", torch.bfloat16, (B, Hkv, Lmax, D), dev)
    _check(prefix_lens, "prefix_lens", torch.int32, (B,), dev)
    _check(accept_len, "accept_len", torch.int32, (B,), dev)
    _check(accepted_nodes, "accepted_nodes", torch.int32, (B, N), dev)
    if new_prefix_lens is None:
        new_prefix_lens = torch.empty((B,), dtype=torch.int32, device=dev)
    if status is None:
        status = torch.zeros((B,), dtype=torch.int32, device=dev)
    rc = lib().spec_kv_compact(
        _ptr(k_cache), _ptr(v_cache), _ptr(prefix_lens), _ptr(accept_len), _ptr(accepted_nodes),
        _ptr(new_prefix_lens), B, N, Hkv, D, Lmax, _ptr(status), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError("spec_kv_compact", rc)
    return new_prefix_lens, status


def spec_kv_compact_paged(k_pages, v_pages, block_table, prefix_lens, accept_len, accepted_nodes,
                          new_prefix_lens=None, status=None, stream=None):
    """Commit the accepted path in place (paged cache); returns (new_prefix_lens, status)."""
    torch = _torch()
    num_pages, Hkv, P, D = k_pages.shape
    B, max_pages = block_table.shape
    N = accepted_nodes.shape[1]
    dev = k_pages.device
    _check(k_pages, "k_pages", torch.bfloat16, (num_pages, Hkv, P, D), dev)
    _check(v_pages, "v_pages", torch.bfloat16, (num_pages, Hkv, P, D), dev)
    _check(block_table, "block_table", torch.int32, (B, max_pages), dev)
    _check(prefix_lens, "prefix_lens", torch.int32, (B,), dev)
    _check(accept_len, "accept_len", torch.int32, (B,), dev)
    _check(accepted_nodes, "accepted_nodes", torch.int32, (B, N), dev)
    if new_prefix_lens is None:
        new_prefix_lens = torch.empty((B,), dtype=torch.int32, device=dev)
    if status is None:
        status = torch.zeros((B,), dtype=torch.int32, device=dev)
    rc = lib().spec_kv_compact_paged(
        _ptr(k_pages), _ptr(v_pages), _ptr(block_table), P, max_pages, num_pages,
        _ptr(prefix_lens), _ptr(accept_len), _ptr(accepted_nodes), _ptr(new_prefix_lens),
        B, N, Hkv, D, _ptr(status), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError("spec_kv_compact_paged", rc)
    return new_prefix_lens, status


def spec_tree_verify_filtered_workspace(B, N, V) -> int:
    return int(lib().spec_tree_verify_filtered_workspace(B, N, V))


def _verify_outputs(target_logits, draft_probs, tree_tokens, tree_parent, uniforms, outputs,
                    status, want_nodes, want_child_q):
    torch = _torch()
    B, N, V = target_logits.shape
    dev = target_logits.device
    _check(target_logits, "target_logits", torch.float32, (B, N, V), dev)
    if draft_probs is not None:
        _check(draft_probs, "draft_probs", torch.float32, (B, N, V), dev)
    _check(tree_tokens, "tree_tokens", torch.int32, (B, N), dev)
    _check(tree_parent, "tree_parent", torch.int32, (B, N), dev)
    _check(uniforms, "uniforms", torch.float32, (B, N), dev)
    o = dict(outputs or {})
    i32 = dict(dtype=torch.int32, device=dev)
    o.setdefault("accept_len", torch.empty((B,), **i32))
    o.setdefault("accepted_tokens", torch.empty((B, N), **i32))
    o.setdefault("bonus", torch.empty((B,), **i32))
    if want_nodes:
        o.setdefault("accepted_nodes", torch.empty((B, N), **i32))
    if want_child_q:
        o.setdefault("child_q", torch.empty((B, N), dtype=torch.float32, device=dev))
    o["status"] = status if status is not None else torch.zeros((B,), **i32)  # bits are OR-ed in
    return o


def spec_tree_verify(target_logits, draft_probs, tree_tokens, tree_parent, uniforms, temperature,
                     outputs=None, workspace=None, status=None, want_nodes=True,
                     want_child_q=False, stream=None):
    """Speculative-sampling verification; returns a dict of device tensors.

    Keys: accept_len [B], accepted_tokens [B,N], bonus [B], accepted_nodes [B,N] (if want_nodes),
    child_q [B,N] (if want_child_q), status [B].
    """
    torch = _torch()
    o = _verify_outputs(target_logits, draft_probs, tree_tokens, tree_parent, uniforms, outputs,
                        status, want_nodes, want_child_q)
    B, N, V = target_logits.shape
    dev = target_logits.device
    ws_bytes = spec_tree_verify_workspace(B, N, V)
    if workspace is None:
        workspace = torch.empty((max(ws_bytes, 16),), dtype=torch.uint8, device=dev)
    rc = lib().spec_tree_verify(
        _ptr(target_logits), _ptr(draft_probs), _ptr(tree_tokens), _ptr(tree_parent),
        _ptr(uniforms), float(temperature), B, N, V, _ptr(o["accept_len"]),
        _ptr(o["accepted_tokens"]), _ptr(o["bonus"]), _ptr(o.get("accepted_nodes")),
        _ptr(o.get("child_q")), _ptr(workspace), workspace.numel(), _ptr(o["status"]),
        _stream(stream))
    if rc != SPEC_OK:
        raise SpecError("spec_tree_verify", rc)
    return o


def spec_tree_verify_greedy(node_argmax, tree_tokens, tree_parent, V, outputs=None, status=None,
                            want_nodes=True, stream=None):
    """Greedy (T = 0) verification from each node's argmax token (node_argmax int32 [B, N], e.g.
    spec_lm_head_stats's argmax viewed as [B, N]); same outputs as spec_tree_verify."""
    torch = _torch()
    B, N = tree_tokens.shape
    dev = tree_tokens.device
    _check(node_argmax, "node_argmax", torch.int32, (B, N), dev)
    _check(tree_tokens, "tree_tokens", torch.int32, (B, N), dev)
    _check(tree_parent, "tree_parent", torch.int32, (B, N), dev)
    o = dict(outputs or {})
    i32 = dict(dtype=torch.int32, device=dev)
    o.setdefault("accept_len", torch.empty((B,), **i32))
    o.setdefault("accepted_tokens", torch.empty((B, N), **i32))
    o.setdefault("bonus", torch.empty((B,), **i32))
    if want_nodes:
        o.setdefault("accepted_nodes", torch.empty((B, N), **i32))
    o["status"] = status if status is not None else torch.zeros((B,), **i32)  # bits are OR-ed in
    rc = lib().spec_tree_verify_greedy(
        _ptr(node_argmax), _ptr(tree_tokens), _ptr(tree_parent), B, N, int(V),
        _ptr(o["accept_len"]), _ptr(o["accepted_tokens"]), _ptr(o["bonus"]),
        _ptr(o.get("accepted_nodes")), _ptr(o["status"]), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError("spec_tree_verify_greedy", rc)
    return o


def spec_tree_verify_head_workspace(B, N, H, V, max_depth) -> int:
    return int(lib().spec_tree_verify_head_workspace(int(B), int(N), int(H), int(V),
                                                     int(max_depth)))


def spec_tree_verify_head(hidden, head, draft_probs, tree_tokens, tree_parent, uniforms,
                          temperature, max_depth, packed_vocab=None, outputs=None, workspace=None,
                          status=None, want_nodes=True, stream=None):
    """Verification from each node's final hidden state (bf16 [B, N, H]) and the LM head (bf16
    [V, H], or spec_lm_head_pack's copy with packed_vocab = V) without the logit matrix; the trees'
    depth must not exceed max_depth.  Same outputs as spec_tree_verify (no per-child q)."""
    torch = _torch()
    B, N, H = hidden.shape
    dev = hidden.device
    _check(hidden, "hidden", torch.bfloat16, (B, N, H), dev)
    if packed_vocab is None:
        V = head.shape[0]
        _check(head, "head", torch.bfloat16, (V, H), dev)
    else:
        V = int(packed_vocab)
        if head.numel() * head.element_size() < spec_lm_head_packed_bytes(V, H):
            raise ValueError("packed head too small")
    T = float(temperature)
    if T > 0:
        _check(draft_probs, "draft_probs", torch.float32, (B, N, V), dev)
    _check(tree_tokens, "tree_tokens", torch.int32, (B, N), dev)
    _check(tree_parent, "tree_parent", torch.int32, (B, N), dev)
    _check(uniforms, "uniforms", torch.float32, (B, N), dev)
    o = dict(outputs or {})
    i32 = dict(dtype=torch.int32, device=dev)
    o.setdefault("accept_len", torch.empty((B,), **i32))
    o.setdefault("accepted_tokens", torch.empty((B, N), **i32))
    o.setdefault("bonus", torch.empty((B,), **i32))
    if want_nodes:
        o.setdefault("accepted_nodes", torch.empty((B, N), **i32))
    o["status"] = status if status is not None else torch.zeros((B,), **i32)  # bits are OR-ed in
    ws_bytes = spec_tree_verify_head_workspace(B, N, H, V, max_depth)
    if workspace is None:
        workspace = torch.empty((max(ws_bytes, 16),), dtype=torch.uint8, device=dev)
    rc = lib().spec_tree_verify_head(
        _ptr(hidden), _ptr(head), 0 if packed_vocab is None else 1,
        _ptr(draft_probs) if T > 0 else None, _ptr(tree_tokens), _ptr(tree_parent),
        _ptr(uniforms), T, B, N, H, V, int(max_depth), _ptr(o["accept_len"]),
        _ptr(o["accepted_tokens"]), _ptr(o["bonus"]), _ptr(o.get("accepted_nodes")),
        _ptr(workspace), workspace.numel(), _ptr(o["status"]), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError("spec_tree_verify_head", rc)
    return o


def spec_tree_verify_filtered(target_logits, draft_probs, tree_tokens, tree_parent, uniforms,
                              temperature, top_k=0, top_p=1.0, outputs=None, workspace=None,
                              status=None, want_nodes=True, want_child_q=False, stream=None):
    """Verification against the top-k / top-p filtered target distribution (top_k 0 and top_p 1
    switch a filter off); same outputs as spec_tree_verify."""
    torch = _torch()
    o = _verify_outputs(target_logits, draft_probs, tree_tokens, tree_parent, uniforms, outputs,
                        status, want_nodes, want_child_q)
    B, N, V = target_logits.shape
    dev = target_logits.device
    ws_bytes = spec_tree_verify_filtered_workspace(B, N, V)
    if workspace is None:
        workspace = torch.empty((max(ws_bytes, 16),), dtype=torch.uint8, device=dev)
    rc = lib().spec_tree_verify_filtered(
        _ptr(target_logits), _ptr(draft_probs), _ptr(tree_tokens), _ptr(tree_parent),
        _ptr(uniforms), float(temperature), int(top_k), float(top_p), B, N, V,
        _ptr(o["accept_len"]), _ptr(o["accepted_tokens"]), _ptr(o["bonus"]),
        _ptr(o.get("accepted_nodes")), _ptr(o.get("child_q")), _ptr(workspace),
        workspace.numel(), _ptr(o["status"]), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError("spec_tree_verify_filtered", rc)
    return o


# ----------------------------------------------------------------------------------------------
# verification without a workspace argument
# ----------------------------------------------------------------------------------------------
_NOALLOC_ARGS = [_vp] * 5 + [_c_float] + [_c_int] * 3 + [_vp] * 5 + [_vp, _vp]


def _header_define(name: str) -> int:
    """An integer #define of the C header (one source of truth for the library's limits)."""
    import re
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                        "spectree.h")
    with open(path) as f:
        m = re.search(r"^#define\s+" + name + r"\s+(\d+)", f.read(), flags=re.M)
    if m is None:
        raise RuntimeError(f"{name} not found in {path}")
    return int(m.group(1))


NOALLOC_MAX_NODES = _header_define("SPEC_NOALLOC_MAX_NODES")


def spec_tree_verify_noalloc(target_logits, draft_probs, tree_tokens, tree_parent, uniforms,
                             temperature, outputs=None, status=None, stream=None):
    """spec_tree_verify for callers that cannot provide device scratch memory.

    The library keeps the scratch in a fixed device array (B * N <= NOALLOC_MAX_NODES per call), so
    this path allocates nothing on the device besides outputs the caller did not pass.  Calls must
    not overlap on the GPU: they share that array.
    """
    torch = _torch()
    B, N, V = target_logits.shape
    dev = target_logits.device
    _check(target_logits, "target_logits", torch.float32, (B, N, V), dev)
    if draft_probs is not None:
        _check(draft_probs, "draft_probs", torch.float32, (B, N, V), dev)
    _check(tree_tokens, "tree_tokens", torch.int32, (B, N), dev)
    _check(tree_parent, "tree_parent", torch.int32, (B, N), dev)
    _check(uniforms, "uniforms", torch.float32, (B, N), dev)
    o = dict(outputs or {})
    i32 = dict(dtype=torch.int32, device=dev)
    o.setdefault("accept_len", torch.empty((B,), **i32))
    o.setdefault("accepted_tokens", torch.empty((B, N), **i32))
    o.setdefault("bonus", torch.empty((B,), **i32))
    o["status"] = status if status is not None else torch.zeros((B,), **i32)
    fn = lib().spec_tree_verify_noalloc
    fn.restype, fn.argtypes = _c_int, _NOALLOC_ARGS
    rc = fn(_ptr(target_logits), _ptr(draft_probs), _ptr(tree_tokens), _ptr(tree_parent),
            _ptr(uniforms), float(temperature), B, N, V, _ptr(o["accept_len"]),
            _ptr(o["accepted_tokens"]), _ptr(o["bonus"]), _ptr(o.get("accepted_nodes")),
            _ptr(o.get("child_q")), _ptr(o["status"]), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError("spec_tree_verify_noalloc", rc)
    return o


def spec_debug_set_verify_wait_polls(polls: int) -> None:
    """Debugging: the first-attempt poll limit of the verification kernels' bounded waits (0 makes
    every such wait give up at once and flag SPEC_ST_TIMEOUT; negative restores the default)."""
    lib().spec_debug_set_verify_wait_polls(int(polls))


# ----------------------------------------------------------------------------------------------
# dynamic tree construction
# ----------------------------------------------------------------------------------------------
def spec_tree_build_workspace(B, K, D) -> int:
    return int(lib().spec_tree_build_workspace(B, K, D))


def spec_tree_expand(draft_logits, K, D, level, workspace, frontier_tokens=None,
                     frontier_parent_slot=None, status=None, stream=None):
    """One level: draft_logits [B, 1, V] at level 1, else [B, K, V] (the frontier's draft rows).
    Returns (frontier_tokens [B, K], frontier_parent_slot [B, K], status [B])."""
    torch = _torch()
    B, R, V = draft_logits.shape
    dev = draft_logits.device
    _check(draft_logits, "draft_logits", torch.float32, (B, 1 if level == 1 else K, V), dev)
    i32 = dict(dtype=torch.int32, device=dev)
    if frontier_tokens is None:
        frontier_tokens = torch.empty((B, K), **i32)
    if frontier_parent_slot is None:
        frontier_parent_slot = torch.empty((B, K), **i32)
    if status is None:
        status = torch.zeros((B,), **i32)
    rc = lib().spec_tree_expand(_ptr(draft_logits), B, V, K, D, level, _ptr(workspace),
                                workspace.numel() * workspace.element_size(),
                                _ptr(frontier_tokens), _ptr(frontier_parent_slot), _ptr(status),
                                _stream(stream))
    if rc != SPEC_OK:
        raise SpecError("spec_tree_expand", rc)
    return frontier_tokens, frontier_parent_slot, status


def spec_tree_finalize(workspace, root_tokens, K, D, N, outputs=None, status=None, stream=None):
    """The tree of the root and the N - 1 best candidates; returns a dict of device tensors:
    tree_tokens, tree_parent, node_row [B, N] int32, node_value [B, N] fp32, status [B]."""
    torch = _torch()
    B = root_tokens.shape[0]
    dev = root_tokens.device
    _check(root_tokens, "root_tokens", torch.int32, (B,), dev)
    o = dict(outputs or {})
    i32 = dict(dtype=torch.int32, device=dev)
    for k in ("tree_tokens", "tree_parent", "node_row"):
        o.setdefault(k, torch.empty((B, N), **i32))
    o.setdefault("node_value", torch.empty((B, N), dtype=torch.float32, device=dev))
    o["status"] = status if status is not None else torch.zeros((B,), **i32)
    rc = lib().spec_tree_finalize(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _ptr(root_tokens), B, K, D, N, _ptr(o["tree_tokens"]),
                                  _ptr(o["tree_parent"]), _ptr(o["node_row"]),
                                  _ptr(o["node_value"]), _ptr(o["status"]), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError("spec_tree_finalize", rc)
    return o


# ----------------------------------------------------------------------------------------------
# LM head fused with the verification statistics
# ----------------------------------------------------------------------------------------------
def spec_lm_head_stats_workspace(M, V) -> int:
    return int(lib().spec_lm_head_stats_workspace(M, V))


def spec_lm_head_packed_bytes(V, H) -> int:
    return int(lib().spec_lm_head_packed_bytes(V, H))


def spec_lm_head_pack(weight, packed=None, stream=None):
    """The head [V, H] (bf16) in tile-major order (a uint8 device tensor)."""
    torch = _torch()
    V, H = weight.shape
    _check(weight, "weight", torch.bfloat16, (V, H), weight.device)
    nbytes = spec_lm_head_packed_bytes(V, H)
    if packed is None:
        packed = torch.empty((nbytes,), dtype=torch.uint8, device=weight.device)
    rc = lib().spec_lm_head_pack(_ptr(weight), V, H, _ptr(packed), packed.numel(),
                                 _stream(stream))
    if rc != SPEC_OK:
        raise SpecError("spec_lm_head_pack", rc)
    return packed


def spec_lm_head_stats(hidden, weight, temperature=1.0, gather_idx=None, outputs=None,
                       workspace=None, status=None, stream=None, packed_vocab=None):
    """Per row of hidden [M, H] @ weight [V, H]^T (bf16): max, sum of exp((l - max) / T), argmax
    and the logits at gather_idx [M, G]; returns a dict of device tensors.  With packed_vocab = V,
    `weight` is the head made by spec_lm_head_pack."""
    torch = _torch()
    M, H = hidden.shape
    dev = hidden.device
    _check(hidden, "hidden", torch.bfloat16, (M, H), dev)
    if packed_vocab is None:
        V = weight.shape[0]
        _check(weight, "weight", torch.bfloat16, (V, H), dev)
    else:
        V = int(packed_vocab)
        if weight.numel() * weight.element_size() < spec_lm_head_packed_bytes(V, H):
            raise ValueError("packed head too small")
    G = 0 if gather_idx is None else gather_idx.shape[1]
    if gather_idx is not None:
        _check(gather_idx, "gather_idx", torch.int32, (M, G), dev)
    o = dict(outputs or {})
    o.setdefault("max", torch.empty((M,), dtype=torch.float32, device=dev))
    o.setdefault("sumexp", torch.empty((M,), dtype=torch.float32, device=dev))
    o.setdefault("argmax", torch.empty((M,), dtype=torch.int32, device=dev))
    if G:
        o.setdefault("gather", torch.full((M, G), float("nan"), dtype=torch.float32, device=dev))
    o["status"] = status if status is not None else torch.zeros((1,), dtype=torch.int32,
                                                                 device=dev)
    if workspace is None:
        workspace = torch.empty((max(spec_lm_head_stats_workspace(M, V), 16),), dtype=torch.uint8,
                                device=dev)
    fn = lib().spec_lm_head_stats if packed_vocab is None else lib().spec_lm_head_stats_packed
    rc = fn(_ptr(hidden), _ptr(weight), _ptr(gather_idx), M, H, V, G, float(temperature),
            _ptr(o["max"]), _ptr(o["sumexp"]), _ptr(o["argmax"]), _ptr(o.get("gather")),
            _ptr(workspace), workspace.numel(), _ptr(o["status"]), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError("spec_lm_head_stats", rc)
    return o
