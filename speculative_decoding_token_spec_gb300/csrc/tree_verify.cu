// Speculative-sampling verification of a draft token tree (sm_103a).
//
// Method: speculative-decoding survey explainer, "Formal Definition" -- draft x~_i ~ p_i is accepted
// if r < min(1, q_i(x~_i) / p_i(x~_i)); at the first rejection c the next token is drawn from
// norm(max(0, q_c - p_c)); greedy verification (taxonomy table) accepts a draft equal to the target's
// argmax.  Tree form: children of the current node are tried in ascending index against the current
// target distribution, which becomes its normalised residual after every rejection.
//
// Two kernels:
//   node kernel  grid (CL, N, B), one thread-block cluster of CL CTAs per (sequence, node).  Leaves
//                exit at once.  For an internal node j the cluster sweeps target row j once
//                (128-bit loads, online max / compensated sum, or the argmax at T = 0), reduces the
//                per-CTA partials through distributed shared memory, then runs the sibling-ordered
//                tests of j's children; each rejection that leaves a sibling to test costs one more
//                sweep (target row + draft row) for the residual's normaliser beta.
//   walk kernel  grid (CL, B), one cluster per sequence.  Follows the accepted child of every node
//                from the root, writes the accepted path, and draws the bonus token at the node
//                where the walk stopped: argmax (T = 0), q_c (leaf) or the last residual (all
//                children rejected), by inverse CDF over the cluster's slices.
//
// Precision: element terms are fp32 (expf); sums use TwoSum-compensated fp32 per thread and fp64
// across threads / CTAs; the few gathered q(x~) values and every accept test are evaluated in fp64.
#include <cooperative_groups.h>
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace spectree {

constexpr int kVThreads = 256;
constexpr int kVWarps = kVThreads / 32;

struct ClusterPart {
  float m;
  int idx;
  double s;
  int flags;
  int last_nz;
};

struct VerifySmem {
  int parent[kMaxNodes];
  int tokens[kMaxNodes];
  int kids[kMaxNodes];
  int nk;
  int bad;
  int decision;
  int terminal;
  int path[kMaxNodes];
  int path_len;
  int flags;
  float red_f[kVWarps];
  int red_i[kVWarps];
  double red_d[kVWarps];
  double scan_d[kVThreads];
  ClusterPart part[2];  // ping-pong slots read by the other CTAs of the cluster
  double beta[kMaxNodes];
};

__device__ __forceinline__ bool bad_value(float v) { return !(v <= FLT_MAX); }  // NaN or +Inf

// The CTA's slice of a row in float4 units.  Elements [0, a0) and [a0 + 4 * nvec, V) are the
// unaligned head / tail (at most 3 each), swept by rank 0.
struct RowSlice {
  const float* row;
  int a0, nvec, v_lo, v_hi, tail_lo, V;
  __device__ RowSlice(const float* r, int V_, int rank, int cl) : row(r), V(V_) {
    uintptr_t mis = (reinterpret_cast<uintptr_t>(r) >> 2) & 3u;
    a0 = mis ? int(4 - mis) : 0;
    if (a0 > V) a0 = V;
    nvec = (V - a0) >> 2;
    v_lo = int((long long)nvec * rank / cl);
    v_hi = int((long long)nvec * (rank + 1) / cl);
    tail_lo = a0 + 4 * nvec;
  }
  __device__ float4 vec(int i) const {
    return __ldg(reinterpret_cast<const float4*>(row + a0) + i);
  }
};

// ------------------------------------------------------------------------------------------------
// block / cluster reductions (fixed association order: deterministic)
// ------------------------------------------------------------------------------------------------
__device__ float block_max(float v, VerifySmem& sm) {
  v = warp_max_f(v);
  int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sm.red_f[w] = v;
  __syncthreads();
  float r = sm.red_f[0];
  for (int i = 1; i < kVWarps; ++i) r = fmaxf(r, sm.red_f[i]);
  return r;
}

__device__ double block_sum(double v, VerifySmem& sm) {
  v = warp_sum_d(v);
  int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sm.red_d[w] = v;
  __syncthreads();
  double r = 0.0;
  for (int i = 0; i < kVWarps; ++i) r += sm.red_d[i];
  return r;
}

__device__ int block_or(int v, VerifySmem& sm) { return __syncthreads_or(v); }

// argmax with lowest index on ties; NaN never wins.
__device__ __forceinline__ void argmax_merge(float& bv, int& bi, float v, int i) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

__device__ void block_argmax(float& bv, int& bi, VerifySmem& sm) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    argmax_merge(bv, bi, ov, oi);
  }
  int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) {
    sm.red_f[w] = bv;
    sm.red_i[w] = bi;
  }
  __syncthreads();
  bv = sm.red_f[0];
  bi = sm.red_i[0];
  for (int i = 1; i < kVWarps; ++i) argmax_merge(bv, bi, sm.red_f[i], sm.red_i[i]);
}

// Publish this CTA's partial in slot `slot`, make it visible cluster-wide, and return a pointer
// for reading rank r's copy.
template <int CL>
__device__ __forceinline__ void cluster_publish(VerifySmem& sm, int slot, const ClusterPart& p) {
  if (threadIdx.x == 0) sm.part[slot] = p;
  if constexpr (CL > 1) {
    cg::this_cluster().sync();
  } else {
    __syncthreads();
  }
}

template <int CL>
__device__ __forceinline__ ClusterPart cluster_read(VerifySmem& sm, int slot, int r) {
  if constexpr (CL > 1) {
    ClusterPart* p = cg::this_cluster().map_shared_rank(&sm.part[slot], r);
    return *p;
  } else {
    return sm.part[slot];
  }
}

// ------------------------------------------------------------------------------------------------
// sweeps over this CTA's slice of a row
// ------------------------------------------------------------------------------------------------
// Online max / compensated sum of exp((l - m) * invT) over the CTA's slice.
__device__ void slice_stats(const RowSlice& rs, int rank, float invT, float& m_out, double& s_out,
                            int& bad_out, VerifySmem& sm) {
  float m = -INFINITY;
  CompSum s;
  bool bad = false;
  auto add = [&](float x) {
    bad |= bad_value(x);
    if (x > m) {
      float f = (m == -INFINITY) ? 0.f : expf((m - x) * invT);
      s.hi *= f;
      s.lo *= f;
      m = x;
    }
    if (m != -INFINITY) s.add(expf((x - m) * invT));
  };
  for (int i = rs.v_lo + threadIdx.x; i < rs.v_hi; i += kVThreads) {
    float4 v = rs.vec(i);
    bad |= bad_value(v.x) | bad_value(v.y) | bad_value(v.z) | bad_value(v.w);
    float mx = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
    if (mx > m) {
      float f = (m == -INFINITY) ? 0.f : expf((m - mx) * invT);
      s.hi *= f;
      s.lo *= f;
      m = mx;
    }
    if (m != -INFINITY) {
      float e = (expf((v.x - m) * invT) + expf((v.y - m) * invT)) +
                (expf((v.z - m) * invT) + expf((v.w - m) * invT));
      s.add(e);
    }
  }
  if (rank == 0) {
    if (threadIdx.x < rs.a0) add(__ldg(rs.row + threadIdx.x));
    int t = rs.tail_lo + threadIdx.x;
    if (threadIdx.x < 4 && t < rs.V) add(__ldg(rs.row + t));
  }
  float M = block_max(m, sm);
  double c = (m == -INFINITY) ? 0.0 : s.value() * (double)expf((m - M) * invT);
  s_out = block_sum(c, sm);
  m_out = M;
  bad_out = block_or(bad ? 1 : 0, sm);
}

__device__ void slice_argmax(const RowSlice& rs, int rank, float& bv_out, int& bi_out,
                             int& bad_out, VerifySmem& sm) {
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  bool bad = false;
  for (int i = rs.v_lo + threadIdx.x; i < rs.v_hi; i += kVThreads) {
    float4 v = rs.vec(i);
    int y = rs.a0 + 4 * i;
    bad |= bad_value(v.x) | bad_value(v.y) | bad_value(v.z) | bad_value(v.w);
    argmax_merge(bv, bi, v.x, y);
    argmax_merge(bv, bi, v.y, y + 1);
    argmax_merge(bv, bi, v.z, y + 2);
    argmax_merge(bv, bi, v.w, y + 3);
  }
  if (rank == 0) {
    if (threadIdx.x < rs.a0) {
      float x = __ldg(rs.row + threadIdx.x);
      bad |= bad_value(x);
      argmax_merge(bv, bi, x, threadIdx.x);
    }
    int t = rs.tail_lo + threadIdx.x;
    if (threadIdx.x < 4 && t < rs.V) {
      float x = __ldg(rs.row + t);
      bad |= bad_value(x);
      argmax_merge(bv, bi, x, t);
    }
  }
  block_argmax(bv, bi, sm);
  bv_out = bv;
  bi_out = bi;
  bad_out = block_or(bad ? 1 : 0, sm);
}

// Residual-chain value of element y: q^(t)(y) from q^(0)(y) = exp((l - M) invT) / S.
__device__ __forceinline__ float residual_chain(float l, float p, float M, float invT, float invS,
                                                const float* inv_beta, int t) {
  float q = expf((l - M) * invT) * invS;
  for (int i = 0; i < t; ++i)
    if (inv_beta[i] > 0.f) q = fmaxf(q - p, 0.f) * inv_beta[i];
  return q;
}

// sum_y max(0, q^(t)(y) - p(y)) over the CTA's slice.
__device__ void slice_beta(const RowSlice& rl, const RowSlice& rp, int rank, float M, float invT,
                           float invS, const float* inv_beta, int t, double& out, int& bad_out,
                           VerifySmem& sm) {
  CompSum s;
  bool bad = false;
  auto term = [&](float l, float p) {
    bad |= !(p >= 0.f && p <= FLT_MAX);
    return fmaxf(residual_chain(l, p, M, invT, invS, inv_beta, t) - p, 0.f);
  };
  for (int i = rl.v_lo + threadIdx.x; i < rl.v_hi; i += kVThreads) {
    float4 l = rl.vec(i);
    float4 p = rp.vec(i);
    float e = (term(l.x, p.x) + term(l.y, p.y)) + (term(l.z, p.z) + term(l.w, p.w));
    s.add(e);
  }
  if (rank == 0) {
    if (threadIdx.x < rl.a0) s.add(term(__ldg(rl.row + threadIdx.x), __ldg(rp.row + threadIdx.x)));
    int t2 = rl.tail_lo + threadIdx.x;
    if (threadIdx.x < 4 && t2 < rl.V) s.add(term(__ldg(rl.row + t2), __ldg(rp.row + t2)));
  }
  out = block_sum(s.value(), sm);
  bad_out = block_or(bad ? 1 : 0, sm);
}

// ------------------------------------------------------------------------------------------------
// shared prologue: load and validate the tree of sequence b
// ------------------------------------------------------------------------------------------------
__device__ int load_tree(const VerifyArgs& a, int b, VerifySmem& sm) {
  const int N = a.N;
  if (threadIdx.x < N) {
    sm.parent[threadIdx.x] = __ldg(a.parent + (size_t)b * N + threadIdx.x);
    sm.tokens[threadIdx.x] = __ldg(a.tokens + (size_t)b * N + threadIdx.x);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int st = 0;
    if (sm.parent[0] != -1) st |= SPEC_ST_BAD_TREE;
    for (int i = 1; i < N; ++i) {
      int p = sm.parent[i];
      if (p < 0 || p >= i) st |= SPEC_ST_BAD_TREE;
      int t = sm.tokens[i];
      if (t < 0 || t >= a.V) st |= SPEC_ST_BAD_TOKEN;
    }
    sm.bad = st;
  }
  __syncthreads();
  return sm.bad;
}

__device__ void list_children(int j, int N, VerifySmem& sm) {
  if (threadIdx.x == 0) {
    int n = 0;
    for (int i = j + 1; i < N; ++i)
      if (sm.parent[i] == j) sm.kids[n++] = i;
    sm.nk = n;
  }
  __syncthreads();
}

// ------------------------------------------------------------------------------------------------
// node kernel
// ------------------------------------------------------------------------------------------------
template <int CL>
__global__ void __launch_bounds__(kVThreads) verify_node_kernel(const VerifyArgs a) {
  __shared__ VerifySmem sm;
  const int rank = (CL > 1) ? int(cg::this_cluster().block_rank()) : 0;
  const int j = blockIdx.y, b = blockIdx.z;
  const int N = a.N, V = a.V;
  if (load_tree(a, b, sm)) return;  // uniform across the cluster: same data everywhere
  list_children(j, N, sm);
  const int nk = sm.nk;
  if (nk == 0) return;

  const size_t row_off = ((size_t)b * N + j) * (size_t)V;
  RowSlice rl(a.logits + row_off, V, rank, CL);
  NodeStat st;
  st.pad = 0;
  int slot = 0;

  if (a.T == 0.f) {
    float bv;
    int bi, bad;
    slice_argmax(rl, rank, bv, bi, bad, sm);
    ClusterPart p{bv, bi, 0.0, bad ? SPEC_ST_NONFINITE : 0, 0};
    cluster_publish<CL>(sm, slot, p);
    float gv = -INFINITY;
    int gi = 0x7fffffff, flags = 0;
    for (int r = 0; r < CL; ++r) {
      ClusterPart o = cluster_read<CL>(sm, slot, r);
      argmax_merge(gv, gi, o.m, o.idx);
      flags |= o.flags;
    }
    if (gi == 0x7fffffff) gi = 0;  // every value NaN: flagged below
    int first = -1, nrej = nk;
    for (int t = 0; t < nk; ++t)
      if (sm.tokens[sm.kids[t]] == gi) {
        first = sm.kids[t];
        nrej = t;
        break;
      }
    if (rank == 0 && threadIdx.x == 0) {
      st.m = gv;
      st.argmax = gi;
      st.s = 0.0;
      st.first_acc = first;
      st.nrej = nrej;
      st.flags = flags;
      a.stats[(size_t)b * N + j] = st;
    }
    if (rank == 0 && a.child_q && threadIdx.x < nk) {
      int k = sm.kids[threadIdx.x];
      float v = threadIdx.x <= nrej ? (sm.tokens[k] == gi ? 1.f : 0.f) : -1.f;
      a.child_q[(size_t)b * N + k] = v;
    }
    if constexpr (CL > 1) cg::this_cluster().sync();  // keep smem alive for remote readers
    return;
  }

  // ---- T > 0: statistics of q_j = softmax(l_j / T)
  const float invT = 1.f / a.T;
  float mloc;
  double sloc;
  int bad;
  slice_stats(rl, rank, invT, mloc, sloc, bad, sm);
  cluster_publish<CL>(sm, slot, ClusterPart{mloc, 0, sloc, bad ? SPEC_ST_NONFINITE : 0, 0});
  float M = -INFINITY;
  int flags = 0;
  for (int r = 0; r < CL; ++r) M = fmaxf(M, cluster_read<CL>(sm, slot, r).m);
  double S = 0.0;
  for (int r = 0; r < CL; ++r) {
    ClusterPart o = cluster_read<CL>(sm, slot, r);
    flags |= o.flags;
    if (o.m != -INFINITY) S += o.s * (double)expf((o.m - M) * invT);
  }
  if (!(S > 0.0) || !(S <= DBL_MAX)) flags |= SPEC_ST_NONFINITE;
  slot ^= 1;

  RowSlice rp(a.probs + row_off, V, rank, CL);
  __shared__ float inv_beta[kMaxNodes];
  const float invS = (float)(1.0 / S);
  const double dT = (double)a.T;
  int first = -1, nrej = nk;
  for (int t = 0; t < nk; ++t) {
    const int k = sm.kids[t];
    if (threadIdx.x == 0) {
      const int x = sm.tokens[k];
      const float lx = __ldg(rl.row + x);
      const float px = __ldg(rp.row + x);
      double q = exp(((double)lx - (double)M) / dT) / S;
      for (int i = 0; i < t; ++i)
        if (sm.beta[i] > 0.0) q = fmax(q - (double)px, 0.0) / sm.beta[i];
      const double r = (double)__ldg(a.uniforms + (size_t)b * N + k);
      const bool acc = r * (double)px < q;  // r < min(1, q/p), division-free
      if (!(px >= 0.f && px <= FLT_MAX)) flags |= SPEC_ST_NONFINITE;
      sm.decision = acc ? 1 : 0;
      if (rank == 0 && a.child_q) a.child_q[(size_t)b * N + k] = (float)q;
    }
    __syncthreads();
    if (sm.decision) {
      first = k;
      nrej = t;
      break;
    }
    if (t == nk - 1) break;  // every child rejected: the walk kernel samples the residual
    // residual normaliser beta_{t+1} = sum_y max(0, q^(t)(y) - p_j(y))
    double bl;
    int bb;
    slice_beta(rl, rp, rank, M, invT, invS, inv_beta, t, bl, bb, sm);
    cluster_publish<CL>(sm, slot, ClusterPart{0.f, 0, bl, bb ? SPEC_ST_NONFINITE : 0, 0});
    double beta = 0.0;
    for (int r = 0; r < CL; ++r) {
      ClusterPart o = cluster_read<CL>(sm, slot, r);
      beta += o.s;
      flags |= o.flags;
    }
    slot ^= 1;
    if (threadIdx.x == 0) {
      sm.beta[t] = beta;
      inv_beta[t] = beta > 0.0 ? (float)(1.0 / beta) : 0.f;
    }
    __syncthreads();
  }
  if (rank == 0) {
    if (threadIdx.x == 0) {
      st.m = M;
      st.argmax = -1;
      st.s = S;
      st.first_acc = first;
      st.nrej = nrej;
      st.flags = flags;
      a.stats[(size_t)b * N + j] = st;
    }
    if (threadIdx.x < nrej && threadIdx.x < nk - 1)
      a.beta[((size_t)b * N + j) * kMaxNodes + threadIdx.x] = sm.beta[threadIdx.x];
    if (a.child_q && threadIdx.x > nrej && threadIdx.x < nk)
      a.child_q[(size_t)b * N + sm.kids[threadIdx.x]] = -1.f;
  }
  if constexpr (CL > 1) cg::this_cluster().sync();
}

// ------------------------------------------------------------------------------------------------
// walk kernel
// ------------------------------------------------------------------------------------------------
// Inclusive block scan (fixed order) of per-thread doubles; fills sm.scan_d.
__device__ void block_scan_inclusive(double v, VerifySmem& sm) {
  const int l = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    double n = __shfl_up_sync(0xffffffffu, v, o);
    if (l >= o) v += n;
  }
  __syncthreads();
  if (l == 31) sm.red_d[w] = v;
  __syncthreads();
  double off = 0.0;
  for (int i = 0; i < w; ++i) off += sm.red_d[i];
  sm.scan_d[threadIdx.x] = off + v;
  __syncthreads();
}

// Weights of the bonus draw at the terminal node c.
//   leaf:                 w(y) = exp((l_y - M) invT)                       (t = 0, sub = false)
//   all children rejected: w(y) = max(0, q^(t)(y) - p_c(y)), t = rejections - 1  (sub = true)
//   zero-residual fallback: w(y) = q^(t)(y)                                 (sub = false)
struct TerminalWeights {
  const float* lrow;
  const float* prow;
  float M, invT, invS;
  const float* inv_beta;
  int t;
  bool sub;
  __device__ __forceinline__ float operator()(int y) const {
    float l = __ldg(lrow + y);
    if (!sub && t == 0) return expf((l - M) * invT) * invS;
    float p = __ldg(prow + y);
    float q = residual_chain(l, p, M, invT, invS, inv_beta, t);
    return sub ? fmaxf(q - p, 0.f) : q;
  }
};

// Inverse-CDF draw y = min{y : C(y) > u * S} over the whole row, each CTA owning a contiguous
// slice and each thread a contiguous chunk of it.  Returns the token (identical in every CTA of
// the cluster), or -1 when the weights sum to zero.
template <int CL>
__device__ int cluster_sample(const TerminalWeights& w, int V, int rank, double u, int& slot,
                              int& flags, VerifySmem& sm) {
  __shared__ int found;
  const int lo = int((long long)V * rank / CL), hi = int((long long)V * (rank + 1) / CL);
  const int chunk = (hi - lo + kVThreads - 1) / kVThreads;
  const int c_lo = min(lo + (int)threadIdx.x * chunk, hi), c_hi = min(c_lo + chunk, hi);
  CompSum s;
  int last_nz = -1;
  bool bad = false;
  for (int y = c_lo; y < c_hi; ++y) {
    float x = w(y);
    bad |= !(x >= 0.f && x <= FLT_MAX);
    if (x > 0.f) last_nz = y;
    s.add(x);
  }
  block_scan_inclusive(s.value(), sm);
  const double W = sm.scan_d[kVThreads - 1];
  int lnz = last_nz;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lnz = max(lnz, __shfl_xor_sync(0xffffffffu, lnz, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.red_i[threadIdx.x >> 5] = lnz;
  __syncthreads();
  int blk_lnz = sm.red_i[0];
  for (int i = 1; i < kVWarps; ++i) blk_lnz = max(blk_lnz, sm.red_i[i]);
  const int blk_bad = block_or(bad ? 1 : 0, sm);

  cluster_publish<CL>(sm, slot, ClusterPart{0.f, blk_lnz, W, blk_bad ? SPEC_ST_NONFINITE : 0, 0});
  double Wr[CL];
  int g_lnz = -1;
  for (int r = 0; r < CL; ++r) {
    ClusterPart o = cluster_read<CL>(sm, slot, r);
    Wr[r] = o.s;
    g_lnz = max(g_lnz, o.idx);
    flags |= o.flags;
  }
  slot ^= 1;
  double Stot = 0.0;
  for (int r = 0; r < CL; ++r) Stot += Wr[r];
  if (!(Stot > 0.0)) return -1;
  const double tgt = u * Stot;
  int rstar = -1;
  double P = 0.0, Pstar = 0.0;
  for (int r = 0; r < CL; ++r) {
    if (P + Wr[r] > tgt) {
      rstar = r;
      Pstar = P;
      break;
    }
    P += Wr[r];
  }
  if (rstar < 0) return g_lnz;  // rounding left no crossing: last positive weight

  if (threadIdx.x == 0) found = -1;
  __syncthreads();
  if (rank == rstar) {
    const double t_loc = tgt - Pstar;
    const double incl = sm.scan_d[threadIdx.x];
    const double excl = threadIdx.x ? sm.scan_d[threadIdx.x - 1] : 0.0;
    if (incl > t_loc && excl <= t_loc) {  // exactly one thread: the scan is non-decreasing
      double acc = excl;
      int y_hit = -1;
      for (int y = c_lo; y < c_hi; ++y) {
        acc += (double)w(y);
        if (acc > t_loc) {
          y_hit = y;
          break;
        }
      }
      found = (y_hit >= 0) ? y_hit : last_nz;
    }
  }
  __syncthreads();
  // broadcast the winner from rank rstar
  if (threadIdx.x == 0) {
    ClusterPart p{0.f, (found >= 0) ? found : blk_lnz, 0.0, 0, 0};
    sm.part[slot] = p;
  }
  if constexpr (CL > 1) {
    cg::this_cluster().sync();
  } else {
    __syncthreads();
  }
  const int y = cluster_read<CL>(sm, slot, rstar).idx;
  slot ^= 1;
  return y;
}

template <int CL>
__global__ void __launch_bounds__(kVThreads) verify_walk_kernel(const VerifyArgs a) {
  __shared__ VerifySmem sm;
  __shared__ float inv_beta[kMaxNodes];
  const int rank = (CL > 1) ? int(cg::this_cluster().block_rank()) : 0;
  const int b = blockIdx.y;
  const int N = a.N, V = a.V;
  const int bad_tree = load_tree(a, b, sm);
  const bool writer = (rank == 0);
  if (bad_tree) {
    if (writer) {
      if (threadIdx.x == 0) {
        a.accept_len[b] = -1;
        a.bonus[b] = -1;
        if (a.status) atomicOr(a.status + b, bad_tree);
      }
      for (int i = threadIdx.x; i < N; i += kVThreads) {
        a.acc_tokens[(size_t)b * N + i] = -1;
        if (a.acc_nodes) a.acc_nodes[(size_t)b * N + i] = -1;
        if (a.child_q) a.child_q[(size_t)b * N + i] = -1.f;
      }
    }
    return;
  }
  // walk from the root along the accepted children
  if (threadIdx.x == 0) {
    int flags = 0;
    bool internal[kMaxNodes];
    for (int i = 0; i < N; ++i) internal[i] = false;
    for (int i = 1; i < N; ++i) internal[sm.parent[i]] = true;
    for (int i = 0; i < N; ++i)
      if (internal[i]) flags |= a.stats[(size_t)b * N + i].flags;
    int c = 0, len = 0;
    while (internal[c]) {
      int fa = a.stats[(size_t)b * N + c].first_acc;
      if (fa <= c || fa >= N || sm.parent[fa] != c) break;  // -1: every child rejected
      sm.path[len++] = fa;
      c = fa;
    }
    sm.path_len = len;
    sm.terminal = c;
    sm.flags = flags;
    sm.nk = internal[c] ? 1 : 0;
  }
  __syncthreads();
  const int c = sm.terminal;
  const bool c_internal = sm.nk != 0;
  int flags = sm.flags;
  int slot = 0;
  int bonus = -1;
  const size_t row_off = ((size_t)b * N + c) * (size_t)V;

  if (a.T == 0.f) {
    if (c_internal) {
      bonus = a.stats[(size_t)b * N + c].argmax;
    } else {
      RowSlice rl(a.logits + row_off, V, rank, CL);
      float bv;
      int bi, bad;
      slice_argmax(rl, rank, bv, bi, bad, sm);
      cluster_publish<CL>(sm, slot, ClusterPart{bv, bi, 0.0, bad ? SPEC_ST_NONFINITE : 0, 0});
      float gv = -INFINITY;
      int gi = 0x7fffffff;
      for (int r = 0; r < CL; ++r) {
        ClusterPart o = cluster_read<CL>(sm, slot, r);
        argmax_merge(gv, gi, o.m, o.idx);
        flags |= o.flags;
      }
      slot ^= 1;
      bonus = (gi == 0x7fffffff) ? 0 : gi;
    }
  } else {
    const float invT = 1.f / a.T;
    TerminalWeights tw;
    tw.lrow = a.logits + row_off;
    tw.prow = a.probs + row_off;
    tw.invT = invT;
    tw.inv_beta = inv_beta;
    if (c_internal) {
      const NodeStat st = a.stats[(size_t)b * N + c];
      const int nrej = st.nrej;  // every child was rejected
      if ((int)threadIdx.x < nrej - 1) {
        double bt = a.beta[((size_t)b * N + c) * kMaxNodes + threadIdx.x];
        inv_beta[threadIdx.x] = bt > 0.0 ? (float)(1.0 / bt) : 0.f;
      }
      __syncthreads();
      tw.M = st.m;
      tw.invS = (float)(1.0 / st.s);
      tw.t = nrej - 1;
      tw.sub = true;
    } else {
      RowSlice rl(tw.lrow, V, rank, CL);
      float mloc;
      double sloc;
      int bad;
      slice_stats(rl, rank, invT, mloc, sloc, bad, sm);
      cluster_publish<CL>(sm, slot, ClusterPart{mloc, 0, sloc, bad ? SPEC_ST_NONFINITE : 0, 0});
      float M = -INFINITY;
      for (int r = 0; r < CL; ++r) {
        ClusterPart o = cluster_read<CL>(sm, slot, r);
        M = fmaxf(M, o.m);
        flags |= o.flags;
      }
      slot ^= 1;
      tw.M = M;
      tw.invS = 1.f;
      tw.t = 0;
      tw.sub = false;
    }
    const double u = (double)__ldg(a.uniforms + (size_t)b * N);
    if (!(flags & SPEC_ST_NONFINITE)) {
      bonus = cluster_sample<CL>(tw, V, rank, u, slot, flags, sm);
      if (bonus < 0 && tw.sub) {
        // the last residual is identically zero: keep the distribution it came from
        tw.sub = false;
        bonus = cluster_sample<CL>(tw, V, rank, u, slot, flags, sm);
      }
    }
  }
  if (flags & SPEC_ST_NONFINITE) bonus = -1;

  if (writer) {
    const int len = sm.path_len;
    const bool ok = bonus >= 0;
    if (threadIdx.x == 0) {
      a.accept_len[b] = ok ? len : -1;
      a.bonus[b] = ok ? bonus : -1;
      if (a.status && flags) atomicOr(a.status + b, flags);
      if (a.child_q) a.child_q[(size_t)b * N] = -1.f;
    }
    for (int i = threadIdx.x; i < N; i += kVThreads) {
      int node = (ok && i < len) ? sm.path[i] : -1;
      a.acc_tokens[(size_t)b * N + i] = node >= 0 ? sm.tokens[node] : -1;
      if (a.acc_nodes) a.acc_nodes[(size_t)b * N + i] = node;
    }
  }
  if constexpr (CL > 1) cg::this_cluster().sync();
}

// ------------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------------
size_t verify_workspace_bytes(int B, int N, int V) {
  (void)V;
  size_t stats = (size_t)B * N * sizeof(NodeStat);
  size_t beta = (size_t)B * N * kMaxNodes * sizeof(double);
  return stats + beta;
}

template <int CL>
static cudaError_t launch_cl(const VerifyArgs& a, dim3 grid, void (*kern)(const VerifyArgs),
                             cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kVThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

static int pick_cluster(long long units, int V, int num_sms) {
  // aim for about one wave of CTAs, and keep each CTA's slice of the row >= 2048 elements
  int cl = 1;
  while (cl < 8 && units * (cl * 2) <= (long long)num_sms * 3 / 2 && V / (cl * 2) >= 2048) cl *= 2;
  return cl;
}

cudaError_t launch_verify(const VerifyArgs& a, int num_sms, cudaStream_t s) {
  const int cl_node = pick_cluster((long long)a.B * a.N / 2, a.V, num_sms);
  const int cl_walk = pick_cluster((long long)a.B, a.V, num_sms);
  cudaError_t e;
  dim3 g1(cl_node, a.N, a.B);
  switch (cl_node) {
    case 1: e = launch_cl<1>(a, g1, verify_node_kernel<1>, s); break;
    case 2: e = launch_cl<2>(a, g1, verify_node_kernel<2>, s); break;
    case 4: e = launch_cl<4>(a, g1, verify_node_kernel<4>, s); break;
    default: e = launch_cl<8>(a, g1, verify_node_kernel<8>, s); break;
  }
  if (e != cudaSuccess) return e;
  dim3 g2(cl_walk, a.B, 1);
  switch (cl_walk) {
    case 1: e = launch_cl<1>(a, g2, verify_walk_kernel<1>, s); break;
    case 2: e = launch_cl<2>(a, g2, verify_walk_kernel<2>, s); break;
    case 4: e = launch_cl<4>(a, g2, verify_walk_kernel<4>, s); break;
    default: e = launch_cl<8>(a, g2, verify_walk_kernel<8>, s); break;
  }
  return e;
}

}  // namespace spectree
