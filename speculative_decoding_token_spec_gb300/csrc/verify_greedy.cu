// Greedy (T = 0) tree verification from each node's argmax token (sm_103a).
//
// Method: survey explainer, Formal Definition, 検証フェーズ, at temperature 0: starting at the root,
// the walk moves to the first child (ascending index) whose draft token equals the argmax of the
// current node's target logits, and stops where no child does; the bonus token is the argmax at
// the node where it stopped.  The argmax per node is all the walk reads, so with the fused LM head
// (spec_lm_head_stats) greedy verification never materialises a logit row.
//
// One warp per sequence (N <= 64): lane l holds nodes l and l + 32 (parent, token, argmax) in
// registers; each step of the walk is two ballots and a shuffle.
#include "common.cuh"
#include "internal.h"

namespace spectree {
namespace {

constexpr int kGreedyWarps = 8;  // sequences per 256-thread block

__global__ void __launch_bounds__(32 * kGreedyWarps)
    verify_greedy_kernel(const int32_t* __restrict__ node_argmax,
                         const int32_t* __restrict__ tokens, const int32_t* __restrict__ parent,
                         int B, int N, int V, int32_t* __restrict__ accept_len,
                         int32_t* __restrict__ acc_tokens, int32_t* __restrict__ bonus,
                         int32_t* __restrict__ acc_nodes, int32_t* __restrict__ status) {
  griddep_wait();  // the argmax may come from the preceding kernel
  griddep_launch_dependents();
  const int b = blockIdx.x * kGreedyWarps + (threadIdx.x >> 5), l = threadIdx.x & 31;
  if (b >= B) return;  // whole warps leave together
  const size_t base = (size_t)b * N;
  const bool h0 = l < N, h1 = l + 32 < N;
  const int p0 = h0 ? __ldg(parent + base + l) : -2, p1 = h1 ? __ldg(parent + base + l + 32) : -2;
  const int t0 = h0 ? __ldg(tokens + base + l) : -1, t1 = h1 ? __ldg(tokens + base + l + 32) : -1;
  const int a0 = h0 ? __ldg(node_argmax + base + l) : -1;
  const int a1 = h1 ? __ldg(node_argmax + base + l + 32) : -1;
  // the tree's checks, as in every verification entry
  bool bt = false, bk = false;
  if (h0) {
    bt |= l == 0 ? p0 != -1 : (p0 < 0 || p0 >= l);
    bk |= l > 0 && (t0 < 0 || t0 >= V);
  }
  if (h1) {
    bt |= p1 < 0 || p1 >= l + 32;
    bk |= t1 < 0 || t1 >= V;
  }
  int flags = (__any_sync(0xffffffffu, bt) ? SPEC_ST_BAD_TREE : 0) |
              (__any_sync(0xffffffffu, bk) ? SPEC_ST_BAD_TOKEN : 0);
  // the walk; path[k] (k < len) is the k-th accepted node, held by lane k & 31 in slot k >> 5
  int c = 0, len = 0, path0 = -1, path1 = -1, am = -1;
  if (!flags) {
    for (;;) {
      const int src = c & 31;
      const int x0 = __shfl_sync(0xffffffffu, a0, src), x1 = __shfl_sync(0xffffffffu, a1, src);
      am = c < 32 ? x0 : x1;
      if (am < 0 || am >= V) {  // the node's logits had no maximum (NaN or -inf throughout)
        flags = SPEC_ST_NONFINITE;
        break;
      }
      const unsigned m0 = __ballot_sync(0xffffffffu, h0 && p0 == c && t0 == am);
      const unsigned m1 = __ballot_sync(0xffffffffu, h1 && p1 == c && t1 == am);
      if (!(m0 | m1)) break;  // no child carries the argmax: c is the terminal node
      c = m0 ? __ffs(m0) - 1 : 32 + __ffs(m1) - 1;  // the lowest-index such child
      if (l == (len & 31)) {
        if (len < 32)
          path0 = c;
        else
          path1 = c;
      }
      ++len;  // children have larger indices than their parents: at most N - 1 steps
    }
  }
  const bool ok = flags == 0;
  if (l == 0) {
    accept_len[b] = ok ? len : -1;
    bonus[b] = ok ? am : -1;
    if (status && flags) atomicOr(status + b, flags);
  }
  // accepted tokens in path order, -1 past the path (and everywhere for a flagged sequence)
  if (h0) {
    const int node = ok && l < len ? path0 : -1;
    acc_tokens[base + l] = node >= 0 ? __ldg(tokens + base + node) : -1;
    if (acc_nodes) acc_nodes[base + l] = node;
  }
  if (h1) {
    const int node = ok && l + 32 < len ? path1 : -1;
    acc_tokens[base + l + 32] = node >= 0 ? __ldg(tokens + base + node) : -1;
    if (acc_nodes) acc_nodes[base + l + 32] = node;
  }
}

}  // namespace

cudaError_t launch_verify_greedy(const int32_t* node_argmax, const int32_t* tokens,
                                 const int32_t* parent, int B, int N, int V, int32_t* accept_len,
                                 int32_t* acc_tokens, int32_t* bonus, int32_t* acc_nodes,
                                 int32_t* status, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((B + kGreedyWarps - 1) / kGreedyWarps));
  cfg.blockDim = dim3(32 * kGreedyWarps);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_greedy_kernel, node_argmax, tokens, parent, B, N, V,
                            accept_len, acc_tokens, bonus, acc_nodes, status);
}

}  // namespace spectree
