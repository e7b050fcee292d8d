// The statistics walk of verification driven by the LM head (shared by verify_head.cu, which
// starts it, and the node step in tree_verify.cu, which continues it after an accepted child).
//
// Survey explainer, Formal Definition, 検証フェーズ: child x~ of node c is accepted iff
// r p_c(x~) < q_c(x~), and q_c(x~) = exp((l_x~ - m) / T) / S needs only the row's max m, its sum S
// and the logit of x~.  From node c the walk accepts first children while that test accepts; the
// node where it stops (its first child rejected, or a leaf) needs its full row.
#pragma once

#include <cfloat>

#include "common.cuh"
#include "internal.h"

namespace spectree {

// One thread.  Moves the walk state of sequence b from node c (its first child not yet tested)
// and returns the node where it stops, marked pending with its row slot and the next pass's flag
// set; or -1 with `flags` set when a value the test reads is not finite (nothing marked).
__device__ inline int head_stats_walk(const HeadWalkIn& w, const float* probs,
                                      const int32_t* tokens, const float* uniforms, int b, int N,
                                      int V, int c, HeadWalk* hw, int& flags) {
  int len = hw->len;
  for (;;) {  // at most one step per level: first children have larger indices
    const size_t r = (size_t)b * N + c;
    const int fc = w.fchild[r];
    if (fc <= c || fc >= N) break;  // a leaf: the bonus draw needs the row
    const float m = w.stat_m[r], S = w.stat_s[r], lx = w.gath[r];
    if (!(m <= FLT_MAX) || !(S > 0.f && S <= FLT_MAX) || !(lx <= FLT_MAX)) {
      flags |= SPEC_ST_NONFINITE;  // +Inf or NaN in the row (or no finite logit at all)
      return -1;
    }
    const int x = tokens[(size_t)b * N + fc];
    const float p = probs[r * (size_t)V + x];
    const float u = uniforms[(size_t)b * N + fc];
    if (!(p >= 0.f && p <= FLT_MAX)) {
      flags |= SPEC_ST_NONFINITE;
      return -1;
    }
    // r p(x~) S < exp((l_x~ - m) / T): the test r < q(x~) / p(x~) without the division
    const double n = exp(((double)lx - (double)m) * w.invT);
    if (!((double)u * (double)p * (double)S < n)) break;  // rejected: residual rounds follow
    if (len < kHeadMaxNodes) hw->path[len] = fc;
    ++len;
    c = fc;
  }
  hw->cur = c;
  hw->len = len;
  hw->pending = c;
  w.row_dst[b] = head_row_offset(b, c, N, V);
  *w.active = 1;
  return c;
}

// The pending node's hidden state into the row pass's input (threads t of nt; 16-byte pieces:
// H % 8 == 0 and both buffers 16-byte aligned).
__device__ inline void head_copy_hidden(const HeadWalkIn& w, int b, int N, int node, int t,
                                        int nt) {
  const uint4* src = reinterpret_cast<const uint4*>(w.hidden + ((size_t)b * N + node) * w.H);
  uint4* dst = reinterpret_cast<uint4*>(w.hrow + (size_t)b * w.H);
  for (int k = t; k < w.H / 8; k += nt) dst[k] = src[k];
}

}  // namespace spectree
