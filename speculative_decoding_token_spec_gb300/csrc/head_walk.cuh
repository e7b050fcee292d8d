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

// One warp (every lane calls it).  Moves the walk state of sequence b from node c (its first
// child not yet tested) and returns the node where it stops, marked pending with its row slot and
// the next pass's flag set; or -1 with `flags` set when a value the test reads is not finite
// (nothing marked).  Every node's first-child test is evaluated at once (lane l: nodes l and
// l + 32, three rounds of independent loads); the walk then follows them through shuffles, and
// only the nodes it visits decide (a non-finite value elsewhere is never looked at).
__device__ inline int head_stats_walk(const HeadWalkIn& w, const float* probs,
                                      const int32_t* tokens, const float* uniforms, int b, int N,
                                      int V, int c, HeadWalk* hw, int& flags) {
  const int lane = threadIdx.x & 31;
  int nxt[2], bad[2];  // per node: the first child if the statistics accept it, else -1
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = lane + 32 * h;
    nxt[h] = -1;
    bad[h] = 0;
    const size_t r = (size_t)b * N + j;
    const int fc = j < N ? w.fchild[r] : -1;
    if (fc > j && fc < N) {
      const float m = w.stat_m[r], S = w.stat_s[r], lx = w.gath[r];
      const int x = tokens[(size_t)b * N + fc];
      const float u = uniforms[(size_t)b * N + fc];
      const float p = probs[r * (size_t)V + x];
      if (!(m <= FLT_MAX) || !(S > 0.f && S <= FLT_MAX) || !(lx <= FLT_MAX) ||
          !(p >= 0.f && p <= FLT_MAX)) {
        bad[h] = SPEC_ST_NONFINITE;  // +Inf or NaN in the row, or a bad draft probability
      } else {
        // r p(x~) S < exp((l_x~ - m) / T): the test r < q(x~) / p(x~) without the division
        const double n = exp(((double)lx - (double)m) * w.invT);
        if ((double)u * (double)p * (double)S < n) nxt[h] = fc;
      }
    }
  }
  int len = hw->len;  // every lane reads the same value
  for (;;) {  // at most one step per level: first children have larger indices
    const int src = c & 31, hi = c >> 5;
    const int n0 = __shfl_sync(0xffffffffu, nxt[0], src), n1 = __shfl_sync(0xffffffffu, nxt[1], src);
    const int b0 = __shfl_sync(0xffffffffu, bad[0], src), b1 = __shfl_sync(0xffffffffu, bad[1], src);
    const int f = hi ? b1 : b0, n = hi ? n1 : n0;
    if (f) {
      flags |= f;
      return -1;
    }
    if (n <= c || n >= N) break;  // a leaf, or the first child rejected: the row is needed
    if (lane == 0 && len < kHeadMaxNodes) hw->path[len] = n;
    ++len;
    c = n;
  }
  if (lane == 0) {
    hw->cur = c;
    hw->len = len;
    hw->pending = c;
    w.row_dst[b] = head_row_offset(b, c, N, V);
    *w.active = 1;
  }
  return c;
}

// The pending node's hidden state into the row pass's input (threads t of nt; 16-byte pieces:
// H % 8 == 0 and both buffers 16-byte aligned).
// Eight loads in flight per thread before their stores (a plain copy loop waits for each load:
// the compiler cannot move a load above the previous store to a possibly aliasing buffer).
__device__ inline void head_copy_hidden(const HeadWalkIn& w, int b, int N, int node, int t,
                                        int nt) {
  constexpr int kBatch = 8;
  const uint4* src = reinterpret_cast<const uint4*>(w.hidden + ((size_t)b * N + node) * w.H);
  uint4* dst = reinterpret_cast<uint4*>(w.hrow + (size_t)b * w.H);
  const int n = w.H / 8;
  for (int k0 = t; k0 < n; k0 += nt * kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (k0 + i * nt < n) v[i] = src[k0 + i * nt];
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (k0 + i * nt < n) dst[k0 + i * nt] = v[i];
  }
}

}  // namespace spectree
