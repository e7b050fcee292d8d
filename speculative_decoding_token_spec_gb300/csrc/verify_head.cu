// Tree verification driven by the target LM head's per-row statistics (sm_103a).
//
// Method: survey explainer, Formal Definition, 検証フェーズ -- child x~ of node c is accepted iff
// r < min(1, q_c(x~) / p_c(x~)); after a rejection the next sibling is tested against
// norm(max(0, q - p_c)); the bonus token is drawn where the walk stops.  EAGLE explainer: q_c comes
// from the target's LM head applied to node c's final hidden state.
//
// Only two kinds of step need more than q_c(x~) = exp((l_x~ - m) / T) / S: the residual rounds
// after a node's first child is rejected, and the bonus draw.  A walk can therefore follow first
// children that are accepted using each row's (m, S) and the first child's logit, which the fused
// LM head produces without writing any logit row, and it needs a full row only at the node where
// it stops following first children.  The walk:
//   1. head_prep_kernel: validate each tree, find every node's first child and its token, check
//      the depth against the caller's bound;
//   2. the LM head over every node's hidden state (lm_head.cu): m, S and the first child's logit;
//   3. head_walk_kernel: from the root, accept first children while the test from the statistics
//      accepts them (head_walk.cuh); the node where it stops is pending (its first child was
//      rejected, or it is a leaf); its hidden state is copied out;
//   4. per row pass (max_depth + 1 of them):
//      a. the LM head over the pending nodes' hidden states writes their full logit rows;
//      b. verify_head_step_kernel (tree_verify.cu): the per-node step of spec_tree_verify on that
//         row -- sibling tests from the first child, residual rounds, the bonus draw; an accepted
//         child becomes the walk's position and the walk continues from it as in 3 (marking the
//         next pass's row), otherwise the outputs are written;
//   5. head_finish_kernel: flags what no pass finished (cannot happen after the depth check).
// Each pass moves a sequence down at least one level or finishes it, so max_depth + 1 passes
// suffice; passes with no pending node leave after one flag read.
#include <cfloat>

#include "common.cuh"
#include "head_walk.cuh"
#include "internal.h"
#include "spectree.h"

namespace spectree {

static_assert(kHeadMaxNodes == kMaxNodes, "walk state holds a whole path");

namespace {

constexpr int kWalkWarps = 4;  // sequences per 128-thread block

// Launch with programmatic stream serialisation, like every kernel of the library.
template <class... Params, class... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, cudaStream_t s,
                       Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

struct Outs {
  int32_t* accept_len;
  int32_t* acc_tokens;
  int32_t* bonus;
  int32_t* acc_nodes;
  int32_t* status;
};

// A flagged sequence: accept_len = bonus = -1, -1 rows (one warp or block writes the rows).
__device__ void flag_sequence(const Outs& o, int b, int N, int flags, int lane, int width) {
  if (lane == 0) {
    o.accept_len[b] = -1;
    o.bonus[b] = -1;
    if (o.status && flags) atomicOr(o.status + b, flags);
  }
  for (int k = lane; k < N; k += width) {
    o.acc_tokens[(size_t)b * N + k] = -1;
    if (o.acc_nodes) o.acc_nodes[(size_t)b * N + k] = -1;
  }
}

// One block of 64 threads per sequence (node i: thread i).  depth_limit > N - 1 disables the
// depth check.
__global__ void __launch_bounds__(kMaxNodes)
    head_prep_kernel(const int32_t* __restrict__ tokens, const int32_t* __restrict__ parent, int B,
                     int N, int V, int depth_limit, int32_t* __restrict__ gidx,
                     int32_t* __restrict__ fchild, HeadWalk* __restrict__ state,
                     int32_t* __restrict__ active, int n_active, int32_t* __restrict__ lmflag,
                     Outs o) {
  __shared__ int par[kMaxNodes];
  __shared__ int maxd;
  const int b = blockIdx.x, i = threadIdx.x;
  griddep_wait();  // the tree may come from the preceding kernel
  griddep_launch_dependents();
  if (b == 0) {
    for (int k = i; k < n_active; k += blockDim.x) active[k] = 0;
    if (i == 0) *lmflag = 0;
  }
  if (i == 0) maxd = 0;
  int st = 0;
  if (i < N) {
    const int p = __ldg(parent + (size_t)b * N + i);
    const int t = __ldg(tokens + (size_t)b * N + i);
    par[i] = p;
    if (i == 0 ? p != -1 : (p < 0 || p >= i)) st |= SPEC_ST_BAD_TREE;
    if (i > 0 && (t < 0 || t >= V)) st |= SPEC_ST_BAD_TOKEN;
  }
  const int bt = __syncthreads_or(st & SPEC_ST_BAD_TREE) ? SPEC_ST_BAD_TREE : 0;
  const int bk = __syncthreads_or(st & SPEC_ST_BAD_TOKEN) ? SPEC_ST_BAD_TOKEN : 0;
  const int bad = bt | bk;
  if (i < N) {
    int fc = -1;
    if (!bad) {
      int d = 0;
      for (int k = i; k > 0; k = par[k]) ++d;  // parents strictly decrease: at most i steps
      atomicMax(&maxd, d);
      for (int c = i + 1; c < N; ++c)
        if (par[c] == i) {
          fc = c;
          break;
        }
    }
    fchild[(size_t)b * N + i] = fc;
    gidx[(size_t)b * N + i] = fc >= 0 ? __ldg(tokens + (size_t)b * N + fc) : -1;
  }
  __syncthreads();
  const int flags = bad | ((!bad && maxd > depth_limit) ? SPEC_ST_BAD_TREE : 0);
  if (i == 0) {
    HeadWalk* w = state + b;
    w->cur = 0;
    w->pending = -1;
    w->len = 0;
    w->done = flags ? 1 : 0;
  }
  if (flags) flag_sequence(o, b, N, flags, i, blockDim.x);
}

struct WalkArgs {
  HeadWalkIn in;
  const float* probs;  // [B, N, V]
  const int32_t* tokens;
  const float* uniforms;
  const int32_t* lmflag;
  HeadWalk* state;
  int B, N, V;
  Outs o;
};

// The walk's first stretch, after the statistics pass: one warp per sequence; lane 0 walks, the
// warp copies the pending node's hidden state.  Later stretches run in the node step's tail.
__global__ void __launch_bounds__(32 * kWalkWarps) head_walk_kernel(const WalkArgs w) {
  const int b = blockIdx.x * kWalkWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  griddep_wait();  // the statistics and the walk state come from the preceding kernels
  griddep_launch_dependents();
  if (b >= w.B) return;  // whole warps leave together
  const int N = w.N;
  HeadWalk* hw = w.state + b;
  int pend = -1;  // >= 0: pending node; -2: flagged here
  int flags = 0;
  if (lane == 0) w.in.row_dst[b] = -1;
  __syncwarp();
  if (!hw->done) {  // the same value in every lane (written by an earlier kernel)
    if (*reinterpret_cast<const volatile int32_t*>(w.lmflag)) flags |= SPEC_ST_TIMEOUT;
    if (!flags)
      pend = head_stats_walk(w.in, w.probs, w.tokens, w.uniforms, b, N, w.V, hw->cur, hw, flags);
    if (flags) {
      if (lane == 0) {
        hw->done = 1;
        hw->pending = -1;
      }
      pend = -2;
    }
  }
  if (pend == -2)
    flag_sequence(w.o, b, N, flags, lane, 32);
  else if (pend >= 0)
    head_copy_hidden(w.in, b, N, pend, lane, 32);
}

// What no pass finished, and LM-head passes that gave up (every sequence flagged).
__global__ void __launch_bounds__(32 * kWalkWarps)
    head_finish_kernel(const HeadWalk* __restrict__ state, const int32_t* __restrict__ lmflag,
                       int B, int N, Outs o) {
  const int b = blockIdx.x * kWalkWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  griddep_wait();
  griddep_launch_dependents();
  if (b >= B) return;
  const bool timeout = *reinterpret_cast<const volatile int32_t*>(lmflag) != 0;
  const bool open = state && !reinterpret_cast<const volatile HeadWalk*>(state + b)->done;
  if (timeout || open)
    flag_sequence(o, b, N, (timeout ? SPEC_ST_TIMEOUT : 0) | (open ? SPEC_ST_BAD_TREE : 0), lane,
                  32);
}

constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

struct HeadLayout {
  size_t part, stat_m, stat_s, gath, gidx, fchild, argmax, row_dst, active, lmflag, state, hrow,
      rows, total;
};

HeadLayout head_layout(int B, int N, int H, int V, int max_depth) {
  const size_t M = (size_t)B * N;
  HeadLayout L;
  size_t o = 0;
  L.part = o;
  o += up(lm_head_workspace_bytes((int)M, V));
  L.stat_m = o;
  o += up(M * 4);
  L.stat_s = o;
  o += up(M * 4);
  L.gath = o;
  o += up(M * 4);
  L.gidx = o;
  o += up(M * 4);
  L.fchild = o;
  o += up(M * 4);
  L.argmax = o;
  o += up(M * 4);
  L.row_dst = o;
  o += up((size_t)B * 8);
  L.active = o;
  o += up((size_t)(max_depth + 1) * 4);
  L.lmflag = o;
  o += up(4);
  L.state = o;
  o += up((size_t)B * sizeof(HeadWalk));
  L.hrow = o;
  o += up((size_t)B * H * 2);
  L.rows = o;
  o += up((size_t)B * (V + 4) * 4);
  L.total = o;
  return L;
}

}  // namespace

size_t verify_head_workspace_bytes(int B, int N, int H, int V, int max_depth) {
  return head_layout(B, N, H, V, max_depth).total;
}

cudaError_t launch_verify_head(const HeadVerifyArgs& a, int num_sms, cudaStream_t s) {
  const HeadLayout L = head_layout(a.B, a.N, a.H, a.V, a.max_depth);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  auto at = [&](size_t off) { return static_cast<void*>(ws + off); };
  int32_t* gidx = static_cast<int32_t*>(at(L.gidx));
  int32_t* fchild = static_cast<int32_t*>(at(L.fchild));
  int32_t* active = static_cast<int32_t*>(at(L.active));
  int32_t* lmflag = static_cast<int32_t*>(at(L.lmflag));
  HeadWalk* state = static_cast<HeadWalk*>(at(L.state));
  const Outs o{a.accept_len, a.acc_tokens, a.bonus, a.acc_nodes, a.status};
  const bool sampling = a.T > 0.f;
  const int M = a.B * a.N;
  const dim3 wgrid((unsigned)((a.B + kWalkWarps - 1) / kWalkWarps)), wblock(32 * kWalkWarps);

  cudaError_t e = launch_pdl(head_prep_kernel, dim3(a.B), dim3(kMaxNodes), s, a.tokens, a.parent,
                             a.B, a.N, a.V, sampling ? a.max_depth : kMaxNodes, gidx, fchild,
                             state, active, a.max_depth + 1, lmflag, o);
  if (e != cudaSuccess) return e;
  if (!sampling) {  // greedy: the argmax of every row, then the argmax walk
    int32_t* argmax = static_cast<int32_t*>(at(L.argmax));
    e = launch_lm_head(a.hidden, a.head, nullptr, M, a.H, a.V, 0, 1.f, nullptr, nullptr, argmax,
                       nullptr, at(L.part), lmflag, num_sms, a.packed, s);
    if (e != cudaSuccess) return e;
    e = launch_verify_greedy(argmax, a.tokens, a.parent, a.B, a.N, a.V, a.accept_len,
                             a.acc_tokens, a.bonus, a.acc_nodes, a.status, s);
    if (e != cudaSuccess) return e;
    return launch_pdl(head_finish_kernel, wgrid, wblock, s, (const HeadWalk*)nullptr,
                      (const int32_t*)lmflag, a.B, a.N, o);
  }
  float* stat_m = static_cast<float*>(at(L.stat_m));
  float* stat_s = static_cast<float*>(at(L.stat_s));
  float* gath = static_cast<float*>(at(L.gath));
  e = launch_lm_head(a.hidden, a.head, gidx, M, a.H, a.V, 1, a.T, stat_m, stat_s, nullptr, gath,
                     at(L.part), lmflag, num_sms, a.packed, s);
  if (e != cudaSuccess) return e;

  HeadWalkIn in;
  in.hidden = static_cast<const uint16_t*>(a.hidden);
  in.fchild = fchild;
  in.stat_m = stat_m;
  in.stat_s = stat_s;
  in.gath = gath;
  in.row_dst = static_cast<long long*>(at(L.row_dst));
  in.active = active;  // pass 0
  in.hrow = static_cast<uint16_t*>(at(L.hrow));
  in.invT = 1.0 / (double)a.T;
  in.H = a.H;
  WalkArgs w;
  w.in = in;
  w.probs = a.probs;
  w.tokens = a.tokens;
  w.uniforms = a.uniforms;
  w.lmflag = lmflag;
  w.state = state;
  w.B = a.B;
  w.N = a.N;
  w.V = a.V;
  w.o = o;
  e = launch_pdl(head_walk_kernel, wgrid, wblock, s, w);
  if (e != cudaSuccess) return e;

  VerifyArgs va;
  va.logits = nullptr;
  va.probs = a.probs;
  va.tokens = a.tokens;
  va.parent = a.parent;
  va.uniforms = a.uniforms;
  va.T = a.T;
  va.B = a.B;
  va.N = a.N;
  va.V = a.V;
  va.accept_len = a.accept_len;
  va.acc_tokens = a.acc_tokens;
  va.bonus = a.bonus;
  va.acc_nodes = a.acc_nodes;
  va.child_q = nullptr;
  va.status = a.status;
  va.stats = nullptr;
  va.counters = nullptr;
  va.handover = nullptr;
  va.walk_done = nullptr;
  va.gen = 0;
  va.first_polls = a.first_polls;
  va.head_rows = static_cast<const float*>(at(L.rows));
  va.head_state = state;
  va.head_flag = lmflag;
  va.head_walk = in;

  for (int it = 0; it <= a.max_depth; ++it) {
    e = launch_lm_head_rows(at(L.hrow), a.head, a.B, a.H, a.V, in.row_dst,
                            static_cast<float*>(at(L.rows)), active + it, lmflag, a.packed, s);
    if (e != cudaSuccess) return e;
    // the step continues the walk after an accepted child and marks the next pass's rows
    va.head_walk.active = it < a.max_depth ? active + it + 1 : nullptr;
    e = launch_verify_head_step(va, num_sms, s);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(head_finish_kernel, wgrid, wblock, s, (const HeadWalk*)state,
                    (const int32_t*)lmflag, a.B, a.N, o);
}

}  // namespace spectree
