"""spec_tree_verify_noalloc: the verification entry point for callers that cannot allocate device
scratch memory (for example a serving engine that gives all free GPU memory to its KV cache at
start-up, or a plugin host that passes a kernel only its input and output buffers).

It is called here through the C ABI and must give the same results as spec_tree_verify with a
caller workspace, on two calls in a row (the fixed scratch keeps the previous call's contents).
This file sorts last so that a run stopping at its first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest

from speculative_decoding_token_spec_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu


def _noalloc_fn(lib):
    fn = lib.spec_tree_verify_noalloc
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.restype = ci
    fn.argtypes = [vp] * 5 + [cf] + [ci] * 3 + [vp] * 5 + [vp, vp]
    return fn


def _call_noalloc(fn, case, dev, child_q=True):
    import torch
    B, N, V = case.target_logits.shape
    t = lambda a: P.dev_tensor(a, dev)  # noqa: E731
    logits, probs = t(case.target_logits), t(case.draft_probs)
    toks, par, unif = t(case.tree_tokens), t(case.tree_parent), t(case.uniforms)
    i32 = dict(dtype=torch.int32, device=dev)
    out = {"accept_len": torch.full((B,), -7, **i32), "accepted_tokens": torch.full((B, N), -7, **i32),
           "bonus": torch.full((B,), -7, **i32), "accepted_nodes": torch.full((B, N), -7, **i32),
           "child_q": torch.full((B, N), -7.0, dtype=torch.float32, device=dev),
           "status": torch.zeros((B,), **i32)}
    rc = fn(logits.data_ptr(), probs.data_ptr(), toks.data_ptr(), par.data_ptr(), unif.data_ptr(),
            float(case.temperature), B, N, V, out["accept_len"].data_ptr(),
            out["accepted_tokens"].data_ptr(), out["bonus"].data_ptr(),
            out["accepted_nodes"].data_ptr(), out["child_q"].data_ptr() if child_q else None,
            out["status"].data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _same(a, ref, child_q=True):
    for k in ("accept_len", "accepted_tokens", "bonus", "accepted_nodes", "status"):
        np.testing.assert_array_equal(a[k], ref[k], err_msg=k)
    if child_q:
        assert np.abs(a["child_q"] - ref["child_q"]).max() <= P.CHILD_Q_ABS


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_noalloc_matches_workspace_entry_point_twice(cuda_lib, T):
    import torch
    dev = torch.device("cuda:0")
    fn = _noalloc_fn(cuda_lib)
    first = W.make_verify_case(W.config("eagle_vicuna7b", B=6), T, seed=31)
    second = W.make_verify_case(W.config("eagle_vicuna7b", B=6), T, seed=32)
    for case in (first, second):          # two calls in a row, different inputs
        ref = P.run_verify_gpu(case, dev, want_child_q=True)
        got = _call_noalloc(fn, case, dev)
        _same(got, ref)
    again = _call_noalloc(fn, first, dev)  # the scratch still holds the second call's data
    _same(again, P.run_verify_gpu(first, dev, want_child_q=True))


def test_noalloc_scratch_layout_changes_between_calls(cuda_lib):
    """B * N shrinks and grows between calls, so each call's arrival counters sit where an earlier
    call left node records (leaf records among them); then a large problem (more than 64 MiB of
    logits) with per-child q, the form in which leaves are not processed but still arrive."""
    import torch
    dev = torch.device("cuda:0")
    fn = _noalloc_fn(cuda_lib)
    cases = [W.make_verify_case(W.config("eagle_vicuna7b", B=B), 1.0, seed=40 + B)
             for B in (12, 5, 6, 1, 12)]
    cases.append(W.make_verify_case(W.config("eagle_vicuna7b", B=16), 1.0, seed=41))
    assert cases[-1].target_logits.nbytes > (64 << 20)
    for case in cases:
        _same(_call_noalloc(fn, case, dev), P.run_verify_gpu(case, dev, want_child_q=True))


def test_noalloc_without_child_q_walks_as_nodes_finish(cuda_lib):
    """Without per-child q small problems take the walk that follows the nodes as they finish
    (call tickets and hand-over words in the scratch); B * N shrinks and grows between calls, so
    those words sit where earlier calls left node records, counters and hand-over words."""
    import torch
    dev = torch.device("cuda:0")
    fn = _noalloc_fn(cuda_lib)
    for B, T in ((12, 1.0), (5, 1.0), (6, 0.0), (1, 1.0), (12, 0.7), (12, 1.0)):
        case = W.make_verify_case(W.config("eagle_vicuna7b", B=B), T, seed=50 + B)
        got = _call_noalloc(fn, case, dev, child_q=False)
        _same(got, P.run_verify_gpu(case, dev, want_child_q=False), child_q=False)


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_lib):
    import torch
    dev = torch.device("cuda:0")
    fn = _noalloc_fn(cuda_lib)
    from speculative_decoding_token_spec_gb300 import _binding
    limit = _binding.NOALLOC_MAX_NODES
    B, N, V = limit // 32 + 1, 32, 8   # B * N = 4128 > limit
    z = torch.zeros((B * N * V + 16,), dtype=torch.float32, device=dev)
    i = torch.zeros((B * N + 16,), dtype=torch.int32, device=dev)
    rc = fn(z.data_ptr(), z.data_ptr(), i.data_ptr(), i.data_ptr(), z.data_ptr(), 1.0, B, N, V,
            i.data_ptr(), i.data_ptr(), i.data_ptr(), None, None, None,
            torch.cuda.current_stream().cuda_stream)
    assert rc == -5
    assert b"SPEC_NOALLOC_MAX_NODES" in cuda_lib.spec_status_string(rc)
