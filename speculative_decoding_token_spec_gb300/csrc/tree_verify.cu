// Speculative-sampling verification of a draft token tree (sm_103a).
//
// Method: speculative-decoding survey explainer, "Formal Definition" -- draft x~_i ~ p_i is accepted
// if r < min(1, q_i(x~_i) / p_i(x~_i)); at the first rejection c the next token is drawn from
// norm(max(0, q_c - p_c)); greedy verification (taxonomy table) accepts a draft equal to the target's
// argmax.  Tree form: children of the current node are tried in ascending index against the current
// target distribution, which becomes its normalised residual after every rejection.
//
// One kernel, grid (CL, N, B): a thread-block cluster of CL CTAs per (sequence, node).
//   * Each CTA of an internal node's cluster copies its slice of the node's target-logit row into
//     shared memory with bulk async copies (all bytes in flight at once).  At T > 0 the cluster
//     reduces the row max M, then every logit is replaced by e(y) = exp((l_y - M)/T) in place and
//     summed; at T = 0 it takes the argmax.  Every warp pushes its partial into every CTA of the
//     cluster (remote stores) and, after one cluster barrier, each warp combines all partials.
//   * The children are tested in index order with the division-free test r * p * D < n (q = n / D,
//     see "Precision"); each rejection builds the next residual in a shared-memory buffer (one
//     multiply-subtract per element) and reduces its normaliser beta.  A node whose children are all
//     rejected draws its own bonus token from the last residual, since the walk stops there
//     whenever it reaches it.  For small problems leaves are processed too (bonus from q_leaf or the
//     argmax).
//   * The last cluster of a sequence to finish (a per-sequence arrival counter in the workspace,
//     reset by that cluster) walks the tree from the root along the accepted children and writes
//     the outputs; for large problems it also draws the bonus at a leaf terminal.
//
// Precision.  Element terms are fp32 (expf once per element).  Every sum is a compensated fp32 sum
// per thread and a double-float (pair of fp32) sum across threads and CTAs: on this part a dependent
// fp64 operation costs 64 cycles and an fp64 division or exp about 1000, so fp64 stays off the
// sequential chains.  The accept decisions compare in fp64 without division: with q^(0)(x) =
// e(x)/S, e(x) = exp((l_x - M)/T), each child keeps a numerator n(x) and the node a common
// denominator D; after a rejection n <- max(0, n - p(x) D) and D <- D beta, so q^(t)(x) = n/D and
// r * p(x) < q(x) becomes r * p(x) * D < n.  e(x) is expf of an argument computed exactly as a
// double-float, times (1 + its low part): relative error within expf's 2 ulp.
#include <cooperative_groups.h>
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace spectree {

constexpr int kVThreads = 256;
constexpr int kVWarps = kVThreads / 32;
constexpr uint32_t kBulkChunk = 32768;  // bytes per bulk copy instruction

// One warp's partial result, published to the whole cluster (32 bytes: two 16-byte stores).
struct __align__(16) WarpPart {
  float m;     // max (stats) / value (argmax)
  int idx;     // argmax index / last positive weight
  float s_hi;  // sum (double-float)
  float s_lo;
  int flags;
  int pad[3];
};
static_assert(sizeof(WarpPart) == 32, "WarpPart layout");

struct VerifySmem {
  int parent[kMaxNodes];
  int tokens[kMaxNodes];
  int kids[kMaxNodes];
  int path[kMaxNodes];
  int internal[kMaxNodes];
  int nk;
  int decision;
  int path_len;
  int terminal;
  int flags;
  int is_last;
  int found[2];
  float red_f[kVWarps];
  float g_r[kMaxNodes];         // children's test uniforms
  WarpPart wp[2][8 * kVWarps];  // ping-pong: every warp partial of the cluster, pushed here
  float inv_beta[kMaxNodes];
  float g_lx[kMaxNodes];  // gathered target logit / draft probability of each child's token
  float g_px[kMaxNodes];
  double g_n[kMaxNodes];  // numerators n(x~) of the children's current q values
  NodeStat st[kMaxNodes];
};

__device__ __forceinline__ bool bad_value(float v) { return !(v <= FLT_MAX); }  // NaN or +Inf

__device__ __forceinline__ float scaled_exp(float l, float M, float invT) {
  return expf(__fmul_rn(__fsub_rn(l, M), invT));
}

// ------------------------------------------------------------------------------------------------
// a CTA's slice of a row, staged in shared memory
// ------------------------------------------------------------------------------------------------
// Elements [lo, hi) of the row belong to this CTA.  [blo, bhi) is the 16-byte aligned part that is
// bulk-copied; the rest (at most 3 elements at each end of the row) is loaded with plain loads.
// Element e sits at buf[e - sbase]; sbase keeps the bulk part 16-byte aligned in shared memory.
struct Slice {
  int lo, hi, blo, bhi, sbase;
};

__device__ __forceinline__ Slice make_slice(const float* row, int V, int rank, int cl) {
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(row) >> 2) & 3u;
  int a0 = mis ? int(4 - mis) : 0;
  if (a0 > V) a0 = V;
  const int nvec = (V - a0) >> 2;
  Slice s;
  s.blo = a0 + 4 * int((long long)nvec * rank / cl);
  s.bhi = a0 + 4 * int((long long)nvec * (rank + 1) / cl);
  s.lo = (rank == 0) ? 0 : s.blo;
  s.hi = (rank == cl - 1) ? V : s.bhi;
  s.sbase = (rank == 0 && a0 > 0) ? a0 - 4 : s.lo;
  return s;
}

// Floats of shared memory one slice buffer needs for (V, CL).
static inline int slice_capacity(int V, int cl) {
  const int nvec = V / 4 + 1;
  return 4 * ((nvec + cl - 1) / cl) + 16;
}

// Issue the copies of the slice into buf (thread 0 issues the bulk part; the ragged ends are
// loaded by the first threads).  Completion: the barrier's phase, then __syncthreads().
__device__ __forceinline__ void stage_slice(const float* row, const Slice& s, float* buf,
                                            uint32_t bar) {
  if (threadIdx.x == 0) {
    const uint32_t bytes = uint32_t(s.bhi - s.blo) * 4u;
    mbar_arrive_expect_tx(bar, bytes);
    const uint32_t dst = smem_u32(buf + (s.blo - s.sbase));
    for (uint32_t off = 0; off < bytes; off += kBulkChunk)
      bulk_load(dst + off, row + s.blo + off / 4, min(kBulkChunk, bytes - off), bar);
  }
  const int head = s.blo - s.lo, tail = s.hi - s.bhi;
  if ((int)threadIdx.x < head) buf[s.lo + threadIdx.x - s.sbase] = __ldg(row + s.lo + threadIdx.x);
  if ((int)threadIdx.x < tail) buf[s.bhi + threadIdx.x - s.sbase] = __ldg(row + s.bhi + threadIdx.x);
}

// Wait for a staged slice (phase `parity` of its barrier: 0 for the barrier's first use in this
// launch, 1 for its second); returns SPEC_ST_TIMEOUT if the copy did not land in time.
__device__ __forceinline__ int wait_slice(uint32_t bar, uint32_t parity = 0) {
  int st = 0;
  if (!mbar_wait(bar, parity)) {
    st = SPEC_ST_TIMEOUT;
    mbar_wait(bar, parity);  // give copies still in flight a second bounded chance
  }
  __syncthreads();
  return st;
}

// Calls f(idx, n) for every element run of the slice (idx = element - sbase): n = 4 over the
// aligned body (16-byte aligned in shared memory), then n = 1 for the ragged ends.
template <class F>
__device__ __forceinline__ void for_slice4(const Slice& s, F&& f) {
  const int off = s.blo - s.sbase;
  const int nv = (s.bhi - s.blo) >> 2;
  for (int i = threadIdx.x; i < nv; i += kVThreads) f(off + 4 * i, 4);
  const int head = s.blo - s.lo, tail = s.hi - s.bhi;
  if ((int)threadIdx.x < head) f(s.lo + threadIdx.x - s.sbase, 1);
  if ((int)threadIdx.x < tail) f(s.bhi + threadIdx.x - s.sbase, 1);
}

__device__ __forceinline__ void load_run(const float* buf, int idx, int n, float (&v)[4]) {
  if (n == 4) {
    const float4 q = *reinterpret_cast<const float4*>(buf + idx);
    v[0] = q.x;
    v[1] = q.y;
    v[2] = q.z;
    v[3] = q.w;
  } else {
    v[0] = buf[idx];
  }
}

__device__ __forceinline__ void store_run(float* buf, int idx, int n, const float (&v)[4]) {
  if (n == 4) {
    *reinterpret_cast<float4*>(buf + idx) = make_float4(v[0], v[1], v[2], v[3]);
  } else {
    buf[idx] = v[0];
  }
}

// ------------------------------------------------------------------------------------------------
// cluster-wide reductions: warp partial -> every warp combines all CL * 8 partials
// ------------------------------------------------------------------------------------------------
template <int CL>
__device__ __forceinline__ void cluster_barrier() {
  if constexpr (CL > 1) {
    cg::this_cluster().sync();
  } else {
    __syncthreads();
  }
}

// p must be warp-uniform.  Lane L < CL of every warp pushes it into CTA L's copy of the partial
// table (entry rank * 8 + warp); after the barrier every CTA holds all CL * 8 partials locally.
template <int CL>
__device__ __forceinline__ void publish(VerifySmem& sm, int slot, int rank, const WarpPart& p) {
  const int lane = threadIdx.x & 31;
  WarpPart* dst = &sm.wp[slot][rank * kVWarps + (threadIdx.x >> 5)];
  if constexpr (CL > 1) {
    if (lane < CL) {
      const uint32_t a = dsmem_addr(dst, lane);
      const uint4* v = reinterpret_cast<const uint4*>(&p);
      dsmem_store_v4(a, v[0]);
      dsmem_store_v4(a + 16, v[1]);
    }
  } else {
    if (lane == 0) *dst = p;
  }
  cluster_barrier<CL>();
}

// Partial e (= rank * 8 + warp) of the cluster, or `fill` past the end (local read).
template <int CL>
__device__ __forceinline__ WarpPart entry(VerifySmem& sm, int slot, int e, const WarpPart& fill) {
  return (e < CL * kVWarps) ? sm.wp[slot][e] : fill;
}

template <int CL>
__device__ DF reduce_sum(VerifySmem& sm, int slot, int& flags) {
  const int l = threadIdx.x & 31;
  const WarpPart fill{0.f, 0, 0.f, 0.f, 0, {0, 0, 0}};
  const WarpPart a = entry<CL>(sm, slot, 2 * l, fill), b = entry<CL>(sm, slot, 2 * l + 1, fill);
  flags |= __reduce_or_sync(0xffffffffu, a.flags | b.flags);
  return warp_sum_df(df_add(DF{a.s_hi, a.s_lo}, DF{b.s_hi, b.s_lo}));
}

// argmax with lowest index on ties; NaN never wins.
__device__ __forceinline__ void argmax_merge(float& bv, int& bi, float v, int i) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

__device__ __forceinline__ void warp_argmax(float& bv, int& bi) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    argmax_merge(bv, bi, ov, oi);
  }
}

template <int CL>
__device__ void reduce_argmax(VerifySmem& sm, int slot, float& gv, int& gi, int& flags) {
  const int l = threadIdx.x & 31;
  const WarpPart fill{-INFINITY, 0x7fffffff, 0.f, 0.f, 0, {0, 0, 0}};
  const WarpPart a = entry<CL>(sm, slot, 2 * l, fill), b = entry<CL>(sm, slot, 2 * l + 1, fill);
  gv = a.m;
  gi = a.idx;
  argmax_merge(gv, gi, b.m, b.idx);
  warp_argmax(gv, gi);
  flags |= __reduce_or_sync(0xffffffffu, a.flags | b.flags);
}

// ------------------------------------------------------------------------------------------------
// sweeps over staged slices
// ------------------------------------------------------------------------------------------------
// Slice max -> warp partial (the cluster max M is reduced from these first).
__device__ WarpPart slice_max(const Slice& s, const float* lbuf, int lflags) {
  float m = -INFINITY;
  bool bad = false;
  for_slice4(s, [&](int idx, int n) {
    float v[4];
    load_run(lbuf, idx, n, v);
    for (int k = 0; k < n; ++k) {
      bad |= bad_value(v[k]);
      m = fmaxf(m, v[k]);
    }
  });
  m = warp_max_f(m);
  const int f = __reduce_or_sync(0xffffffffu, bad ? SPEC_ST_NONFINITE : 0) | lflags;
  return WarpPart{m, 0, 0.f, 0.f, f, {0, 0, 0}};
}

// e(y) = exp((l_y - M) / T) written over the logits, and summed -> warp partial.
__device__ WarpPart slice_exp_sum(const Slice& s, float* lbuf, float M, float invT) {
  CompSum acc;
  for_slice4(s, [&](int idx, int n) {
    float v[4];
    load_run(lbuf, idx, n, v);
    float sum = 0.f;
    for (int k = 0; k < n; ++k) {
      v[k] = (M == -INFINITY) ? 0.f : scaled_exp(v[k], M, invT);
      sum = __fadd_rn(sum, v[k]);
    }
    store_run(lbuf, idx, n, v);
    acc.add(sum);
  });
  const DF S = warp_sum_df(df_from(acc));
  return WarpPart{M, 0, S.hi, S.lo, 0, {0, 0, 0}};
}

// Cluster max of the published slice maxima.
template <int CL>
__device__ float reduce_max(VerifySmem& sm, int slot, int& flags) {
  const int l = threadIdx.x & 31;
  const WarpPart fill{-INFINITY, 0, 0.f, 0.f, 0, {0, 0, 0}};
  const WarpPart a = entry<CL>(sm, slot, 2 * l, fill), b = entry<CL>(sm, slot, 2 * l + 1, fill);
  flags |= __reduce_or_sync(0xffffffffu, a.flags | b.flags);
  return warp_max_f(fmaxf(a.m, b.m));
}

// Statistics of softmax(l / T) over the cluster's row: M = max, S = sum exp((l - M)/T); e(y)
// replaces the logits in lbuf.  Two cluster exchanges (max, then sum).
template <int CL>
__device__ void cluster_exp_stats(const Slice& s, float* lbuf, float invT, int lflags, int rank,
                                  int& slot, float& M, DF& S, int& flags, VerifySmem& sm) {
  publish<CL>(sm, slot, rank, slice_max(s, lbuf, lflags));
  M = reduce_max<CL>(sm, slot, flags);
  slot ^= 1;
  publish<CL>(sm, slot, rank, slice_exp_sum(s, lbuf, M, invT));
  S = reduce_sum<CL>(sm, slot, flags);
  slot ^= 1;
}

__device__ WarpPart slice_argmax(const Slice& s, const float* lbuf, int lflags) {
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  bool bad = false;
  for_slice4(s, [&](int idx, int n) {
    float v[4];
    load_run(lbuf, idx, n, v);
    for (int k = 0; k < n; ++k) {
      bad |= bad_value(v[k]);
      argmax_merge(bv, bi, v[k], idx + k + s.sbase);
    }
  });
  warp_argmax(bv, bi);
  const int f = __reduce_or_sync(0xffffffffu, bad ? SPEC_ST_NONFINITE : 0) | lflags;
  return WarpPart{bv, bi, 0.f, 0.f, f, {0, 0, 0}};
}

// q^(t)(y) from scratch: q^(0) = e(y) * c0 (c0 = 1/S), then t residual rounds (rounds whose
// normaliser was zero keep q).  Used only after a zero normaliser.
__device__ __forceinline__ float chain_q(float e, float p, float c0, const float* inv_beta, int t) {
  float q = __fmul_rn(e, c0);
  for (int i = 0; i < t; ++i)
    if (inv_beta[i] > 0.f) q = __fmul_rn(fmaxf(__fsub_rn(q, p), 0.f), inv_beta[i]);
  return q;
}

struct RoundArgs {
  float c0;               // 1 / S: q^(0) = e * c0
  const float* inv_beta;  // [rounds so far]
  int k;                  // this round (1-based): residual of q^(k-1)
  bool chain;             // a normaliser was zero: recompute q^(k-1) from e
};

// Residual round k: rbuf[y] = max(0, q^(k-1)(y) - p(y)) -> warp partial of sum_y rbuf[y].
// q^(0) = e * c0; q^(k-1) for k > 1 is the previous residual times 1/beta_{k-1}.
__device__ WarpPart residual_round(const Slice& s, const float* ebuf, const float* pbuf,
                                   float* rbuf, const RoundArgs& ra, int lflags) {
  CompSum acc;
  bool bad = false;
  const float invb = (ra.k > 1) ? ra.inv_beta[ra.k - 2] : 0.f;
  for_slice4(s, [&](int idx, int n) {
    float p[4], q[4];
    load_run(pbuf, idx, n, p);
    if (ra.k == 1 || ra.chain) {
      load_run(ebuf, idx, n, q);
    } else {
      load_run(rbuf, idx, n, q);
    }
    float sum = 0.f;
    for (int k = 0; k < n; ++k) {
      bad |= !(p[k] >= 0.f && p[k] <= FLT_MAX);
      float qq;
      if (ra.chain) {
        qq = chain_q(q[k], p[k], ra.c0, ra.inv_beta, ra.k - 1);
      } else {
        qq = __fmul_rn(q[k], ra.k == 1 ? ra.c0 : invb);
      }
      q[k] = fmaxf(__fsub_rn(qq, p[k]), 0.f);
      sum = __fadd_rn(sum, q[k]);
    }
    store_run(rbuf, idx, n, q);
    acc.add(sum);
  });
  const DF S = warp_sum_df(df_from(acc));
  const int f = __reduce_or_sync(0xffffffffu, bad ? SPEC_ST_NONFINITE : 0) | lflags;
  return WarpPart{0.f, 0, S.hi, S.lo, f, {0, 0, 0}};
}

// ------------------------------------------------------------------------------------------------
// inverse-CDF draw across the cluster
// ------------------------------------------------------------------------------------------------
// Weights of the bonus draw, read from the staged buffers (element index idx = y - sbase).
struct Weights {
  enum Kind { kExp, kBuffer, kChain } kind;
  const float* ebuf;  // e(y)
  const float* pbuf;
  const float* rbuf;
  float c;            // kExp: 1 (weights e(y)); kChain: 1/S
  const float* inv_beta;
  int t;
  __device__ __forceinline__ float operator()(int idx) const {
    if (kind == kExp) return ebuf[idx];
    if (kind == kBuffer) return rbuf[idx];
    return chain_q(ebuf[idx], pbuf[idx], c, inv_beta, t);
  }
};

// y = min{y : C(y) > u * S} over the whole row.  Each CTA owns its slice, each thread a contiguous
// chunk of it, so (rank, warp, lane) order is element order.  Returns the token (the same in every
// CTA of the cluster), or -1 when the weights sum to zero.  If rounding leaves no crossing, the
// last positive weight is taken.
template <int CL>
__device__ int cluster_sample(const Weights& w, const Slice& s, int rank, float u, int& slot,
                              int& flags, VerifySmem& sm) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int chunk = (s.hi - s.lo + kVThreads - 1) / kVThreads;
  const int c_lo = min(s.lo + (int)threadIdx.x * chunk, s.hi), c_hi = min(c_lo + chunk, s.hi);
  CompSum acc;
  int last_nz = -1;
  bool bad = false;
  for (int y = c_lo; y < c_hi; ++y) {
    const float x = w(y - s.sbase);
    bad |= !(x >= 0.f && x <= FLT_MAX);
    if (x > 0.f) last_nz = y;
    acc.add(x);
  }
  const DF lane_incl = warp_scan_df(df_from(acc));
  const DF wtot{__shfl_sync(0xffffffffu, lane_incl.hi, 31),
                __shfl_sync(0xffffffffu, lane_incl.lo, 31)};
  int wlnz = last_nz;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wlnz = max(wlnz, __shfl_xor_sync(0xffffffffu, wlnz, o));
  const int wf = __reduce_or_sync(0xffffffffu, bad ? SPEC_ST_NONFINITE : 0);
  publish<CL>(sm, slot, rank, WarpPart{0.f, wlnz, wtot.hi, wtot.lo, wf, {0, 0, 0}});

  // every warp: prefix over the CL * 8 warp totals in element order (lane l: entries 2l, 2l + 1)
  const WarpPart fill{0.f, -1, 0.f, 0.f, 0, {0, 0, 0}};
  const WarpPart ea = entry<CL>(sm, slot, 2 * lane, fill);
  const WarpPart eb = entry<CL>(sm, slot, 2 * lane + 1, fill);
  slot ^= 1;
  flags |= __reduce_or_sync(0xffffffffu, ea.flags | eb.flags);
  int g_lnz = max(ea.idx, eb.idx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) g_lnz = max(g_lnz, __shfl_xor_sync(0xffffffffu, g_lnz, o));
  const DF a{ea.s_hi, ea.s_lo}, b{eb.s_hi, eb.s_lo};
  const DF pincl = warp_scan_df(df_add(a, b));
  DF pexcl{__shfl_up_sync(0xffffffffu, pincl.hi, 1), __shfl_up_sync(0xffffffffu, pincl.lo, 1)};
  if (lane == 0) pexcl = DF{0.f, 0.f};
  const DF Stot{__shfl_sync(0xffffffffu, pincl.hi, 31), __shfl_sync(0xffffffffu, pincl.lo, 31)};
  if (!(Stot.hi > 0.f)) return -1;
  const DF tgt = df_scale(Stot, u);
  const DF incl_a = df_add(pexcl, a);
  const bool ca = df_gt(incl_a, tgt);
  const bool cb = !ca && df_gt(pincl, tgt);
  const unsigned cross = __ballot_sync(0xffffffffu, ca || cb);
  if (cross == 0) return g_lnz;  // rounding left no crossing
  const int L = __ffs(cross) - 1;
  const bool at_a = __shfl_sync(0xffffffffu, ca, L);
  const int estar = 2 * L + (at_a ? 0 : 1);
  const DF pe{__shfl_sync(0xffffffffu, pexcl.hi, L), __shfl_sync(0xffffffffu, pexcl.lo, L)};
  const DF pa{__shfl_sync(0xffffffffu, incl_a.hi, L), __shfl_sync(0xffffffffu, incl_a.lo, L)};
  const DF before = at_a ? pe : pa;
  const int rstar = estar / kVWarps, wstar = estar % kVWarps;

  if (rank == rstar && wid == wstar) {
    // the crossing warp: find the crossing lane, then rescan that lane's chunk 32 at a time
    const DF t_loc = df_add(tgt, DF{-before.hi, -before.lo});
    DF lexcl{__shfl_up_sync(0xffffffffu, lane_incl.hi, 1),
             __shfl_up_sync(0xffffffffu, lane_incl.lo, 1)};
    if (lane == 0) lexcl = DF{0.f, 0.f};
    const unsigned lb = __ballot_sync(0xffffffffu, df_gt(lane_incl, t_loc));
    int y = wlnz;
    if (lb) {
      const int Lc = __ffs(lb) - 1;
      const int tc = wid * 32 + Lc;
      const int r_lo = min(s.lo + tc * chunk, s.hi), r_hi = min(r_lo + chunk, s.hi);
      DF carry{__shfl_sync(0xffffffffu, lexcl.hi, Lc), __shfl_sync(0xffffffffu, lexcl.lo, Lc)};
      y = __shfl_sync(0xffffffffu, last_nz, Lc);
      for (int base = r_lo; base < r_hi; base += 32) {
        const int yy = base + lane;
        const float x = (yy < r_hi) ? w(yy - s.sbase) : 0.f;
        const DF run = df_add(carry, warp_scan_df(DF{x, 0.f}));
        const unsigned hb = __ballot_sync(0xffffffffu, yy < r_hi && df_gt(run, t_loc));
        if (hb) {
          y = base + __ffs(hb) - 1;
          break;
        }
        carry = DF{__shfl_sync(0xffffffffu, run.hi, 31), __shfl_sync(0xffffffffu, run.lo, 31)};
      }
    }
    if constexpr (CL > 1) {
      if (lane < CL) dsmem_store_u32(dsmem_addr(&sm.found[slot], lane), (uint32_t)y);
    } else {
      if (lane == 0) sm.found[slot] = y;
    }
  }
  cluster_barrier<CL>();
  const int y = sm.found[slot];
  slot ^= 1;
  return y;
}

// ------------------------------------------------------------------------------------------------
// tree prologue
// ------------------------------------------------------------------------------------------------
// Loads and validates the tree of sequence b; marks internal nodes.  Returns the status bits.
__device__ int load_tree(const VerifyArgs& a, int b, VerifySmem& sm) {
  const int N = a.N;
  const int i = threadIdx.x;
  int st = 0;
  if (i < N) {
    const int p = __ldg(a.parent + (size_t)b * N + i);
    const int t = __ldg(a.tokens + (size_t)b * N + i);
    sm.parent[i] = p;
    sm.tokens[i] = t;
    sm.internal[i] = 0;
    if (i == 0 ? p != -1 : (p < 0 || p >= i)) st |= SPEC_ST_BAD_TREE;
    if (i > 0 && (t < 0 || t >= a.V)) st |= SPEC_ST_BAD_TOKEN;
  }
  if (i == 0) sm.flags = 0;
  const int bt = __syncthreads_or(st & SPEC_ST_BAD_TREE) ? SPEC_ST_BAD_TREE : 0;
  const int bk = __syncthreads_or(st & SPEC_ST_BAD_TOKEN) ? SPEC_ST_BAD_TOKEN : 0;
  if (bt | bk) return bt | bk;
  if (i > 0 && i < N) sm.internal[sm.parent[i]] = 1;
  __syncthreads();
  return 0;
}

// Children of node j in ascending index (one warp; lane l looks at nodes l and l + 32).
__device__ void list_children(int j, int N, VerifySmem& sm) {
  if (threadIdx.x < 32) {
    const int l = threadIdx.x;
    const bool a = l < N && l > j && sm.parent[l] == j;
    const bool b = l + 32 < N && l + 32 > j && sm.parent[l + 32] == j;
    const unsigned m0 = __ballot_sync(0xffffffffu, a), m1 = __ballot_sync(0xffffffffu, b);
    const unsigned lt = (1u << l) - 1u;
    if (a) sm.kids[__popc(m0 & lt)] = l;
    if (b) sm.kids[__popc(m0) + __popc(m1 & lt)] = l + 32;
    if (l == 0) sm.nk = __popc(m0) + __popc(m1);
  }
  __syncthreads();
}

// Numerator e(x) = exp((l_x - M) / T) of a child's q^(0): the argument is formed exactly as a
// double-float, exponentiated by expf on its high part and corrected by (1 + low part).
__device__ __forceinline__ double child_numerator(float lx, float M, DF invT) {
  const DF d = df_two_sum(lx, -M);
  const DF a = df_mul(d, invT);
  if (a.hi < -80.f) return exp((double)a.hi + (double)a.lo);  // outside expf's normal range
  const double e = (double)expf(a.hi);
  return fma(e, (double)a.lo, e);
}

struct NodeBufs {
  float* lbuf;  // logits, then e(y) at T > 0
  float* pbuf;  // draft probabilities
  float* rbuf;  // residual
  uint32_t bar_l, bar_p;
};

// ------------------------------------------------------------------------------------------------
// one node: statistics, sibling tests, residual rounds, bonus if the walk can stop here
// ------------------------------------------------------------------------------------------------
// logits_staged: the kernel already issued the copy of this node's logit slice into nb.lbuf.
template <int CL>
__device__ NodeStat process_node(const VerifyArgs& a, int b, int j, int rank, const NodeBufs& nb,
                                 bool eager_probs, bool logits_staged, DF invT_df, int& slot,
                                 VerifySmem& sm) {
  const int N = a.N, V = a.V;
  list_children(j, N, sm);
  const int nk = sm.nk;
  const size_t row_off = ((size_t)b * N + j) * (size_t)V;
  const float* lrow = a.logits + row_off;
  const float* prow = a.probs ? a.probs + row_off : nullptr;
  const Slice s = make_slice(lrow, V, rank, CL);  // the draft row has the same alignment
  const bool sampling = a.T > 0.f;
  if (!logits_staged) stage_slice(lrow, s, nb.lbuf, nb.bar_l);
  bool probs_staged = false, probs_ready = false;
  if (sampling && nk > 0 && eager_probs) {
    stage_slice(prow, s, nb.pbuf, nb.bar_p);
    probs_staged = true;
  }
  if ((int)threadIdx.x < nk) {  // gathers for the tests, overlapping the bulk copies
    const int k = sm.kids[threadIdx.x];
    const int x = sm.tokens[k];
    sm.g_lx[threadIdx.x] = __ldg(lrow + x);
    sm.g_px[threadIdx.x] = sampling ? __ldg(prow + x) : 0.f;
    sm.g_r[threadIdx.x] = __ldg(a.uniforms + (size_t)b * N + k);
  }
  const float u_bonus = __ldg(a.uniforms + (size_t)b * N);
  const int lflags0 = wait_slice(nb.bar_l);
  int flags = 0;  // cluster-uniform: only ever updated from published partials
  NodeStat st;
  st.bonus = -1;
  st.s = 0.0;

  if (!sampling) {
    publish<CL>(sm, slot, rank, slice_argmax(s, nb.lbuf, lflags0));
    float gv;
    int gi;
    reduce_argmax<CL>(sm, slot, gv, gi, flags);
    slot ^= 1;
    if (gi == 0x7fffffff) gi = 0;  // every value NaN: flagged
    int first = -1, nrej = nk;
    for (int t = 0; t < nk; ++t)
      if (sm.tokens[sm.kids[t]] == gi) {
        first = sm.kids[t];
        nrej = t;
        break;
      }
    if (rank == 0 && a.child_q && (int)threadIdx.x < nk) {
      const int k = sm.kids[threadIdx.x];
      a.child_q[(size_t)b * N + k] =
          (int)threadIdx.x <= nrej ? (sm.tokens[k] == gi ? 1.f : 0.f) : -1.f;
    }
    st.m = gv;
    st.argmax = gi;
    st.first_acc = first;
    st.nrej = nrej;
    st.flags = flags;
    st.bonus = gi;  // the bonus wherever the walk stops here
    return st;
  }

  // ---- T > 0: statistics of q_j = softmax(l_j / T); e(y) replaces the logits in lbuf
  const float invT = 1.f / a.T;
  float M;
  DF S;
  cluster_exp_stats<CL>(s, nb.lbuf, invT, lflags0, rank, slot, M, S, flags, sm);
  if (!(S.hi > 0.f) || !(S.hi <= FLT_MAX)) flags |= SPEC_ST_NONFINITE;
  const float invS = __fdiv_rn(1.f, S.hi);
  const float c0 = invS;
  double D = df_to_double(S);
  if ((int)threadIdx.x < nk)
    sm.g_n[threadIdx.x] = child_numerator(sm.g_lx[threadIdx.x], M, invT_df);
  if (__syncthreads_or((int)threadIdx.x < nk && !(sm.g_px[threadIdx.x] >= 0.f &&
                                                   sm.g_px[threadIdx.x] <= FLT_MAX)))
    flags |= SPEC_ST_NONFINITE;

  int first = -1, nrej = nk;
  bool chain = false;
  Weights wt;
  wt.ebuf = nb.lbuf;
  wt.pbuf = nb.pbuf;
  wt.rbuf = nb.rbuf;
  wt.inv_beta = sm.inv_beta;
  wt.t = 0;
  if (nk == 0 && !(flags & (SPEC_ST_NONFINITE | SPEC_ST_TIMEOUT))) {
    // leaf (small problems): the bonus when the walk ends here is drawn from q_j
    wt.kind = Weights::kExp;
    wt.c = 1.f;
    st.bonus = cluster_sample<CL>(wt, s, rank, u_bonus, slot, flags, sm);
  }
  for (int t = 0; t < nk; ++t) {
    const int k = sm.kids[t];
    if ((int)threadIdx.x == t) {
      const double px = (double)sm.g_px[t];
      const double r = (double)sm.g_r[t];
      const double n = sm.g_n[t];
      sm.decision = (r * px * D < n) ? 1 : 0;  // r < min(1, q/p) with q = n / D
      if (rank == 0 && a.child_q) {
        const float df = (float)D;
        a.child_q[(size_t)b * N + k] = df > 1e-30f ? __fdiv_rn((float)n, df) : (float)(n / D);
      }
    }
    __syncthreads();
    if (sm.decision) {
      first = k;
      nrej = t;
      break;
    }
    // rejected: residual round t + 1 (needed by the next sibling or by the bonus draw)
    int lflags = 0;  // CTA-local events; they reach every CTA through the published partial
    if (!probs_ready) {
      if (!probs_staged) stage_slice(prow, s, nb.pbuf, nb.bar_p);
      lflags |= wait_slice(nb.bar_p);
      probs_staged = probs_ready = true;
    }
    const RoundArgs ra{c0, sm.inv_beta, t + 1, chain};
    publish<CL>(sm, slot, rank, residual_round(s, nb.lbuf, nb.pbuf, nb.rbuf, ra, lflags));
    const DF beta = reduce_sum<CL>(sm, slot, flags);
    slot ^= 1;
    const double beta_d = df_to_double(beta);
    if (threadIdx.x == 0) {
      sm.inv_beta[t] = beta.hi > 0.f ? __fdiv_rn(1.f, beta.hi) : 0.f;
      if (rank == 0) a.beta[((size_t)b * N + j) * kMaxNodes + t] = beta_d;
    }
    if (t == nk - 1) {  // every child rejected: the bonus comes from the last residual
      __syncthreads();
      if (!(flags & (SPEC_ST_NONFINITE | SPEC_ST_TIMEOUT))) {
        wt.kind = Weights::kBuffer;
        st.bonus = cluster_sample<CL>(wt, s, rank, u_bonus, slot, flags, sm);
        if (st.bonus < 0) {  // the last residual is all zero: keep the distribution it came from
          wt.kind = Weights::kChain;
          wt.c = c0;
          wt.t = t;
          st.bonus = cluster_sample<CL>(wt, s, rank, u_bonus, slot, flags, sm);
        }
      }
      break;
    }
    if (beta_d > 0.0) {
      if ((int)threadIdx.x > t && (int)threadIdx.x < nk)
        sm.g_n[threadIdx.x] = fmax(fma(-(double)sm.g_px[threadIdx.x], D, sm.g_n[threadIdx.x]), 0.0);
      D *= beta_d;
    } else {
      chain = true;  // q stays: later rounds recompute it from e
    }
    __syncthreads();
  }
  if (probs_staged && !probs_ready) flags |= wait_slice(nb.bar_p);  // no copy left in flight
  if (rank == 0 && a.child_q && (int)threadIdx.x > nrej && (int)threadIdx.x < nk)
    a.child_q[(size_t)b * N + sm.kids[threadIdx.x]] = -1.f;
  st.m = M;
  st.argmax = -1;
  st.s = df_to_double(S);
  st.first_acc = first;
  st.nrej = nrej;
  st.flags = flags;
  if (flags & (SPEC_ST_NONFINITE | SPEC_ST_TIMEOUT)) st.bonus = -1;
  return st;
}

// ------------------------------------------------------------------------------------------------
// the walk (run by the last cluster of the sequence to finish)
// ------------------------------------------------------------------------------------------------
// bar_l_used: whether this CTA already staged a row on nb.bar_l in this launch.
template <int CL>
__device__ void walk_sequence(const VerifyArgs& a, int b, int rank, const NodeBufs& nb,
                              bool leaves_done, bool bar_l_used, int& slot, VerifySmem& sm) {
  const int N = a.N, V = a.V;
  // every node record written in this call (L2: bypass L1), flags of the internal rows
  int f = 0;
  if ((int)threadIdx.x < N) {
    const int i = threadIdx.x;
    if (sm.internal[i] || leaves_done) {
      const NodeStat* src = a.stats + (size_t)b * N + i;
      NodeStat st;
      st.m = __ldcg(&src->m);
      st.argmax = __ldcg(&src->argmax);
      st.s = __ldcg(&src->s);
      st.first_acc = __ldcg(&src->first_acc);
      st.nrej = __ldcg(&src->nrej);
      st.flags = __ldcg(&src->flags);
      st.bonus = __ldcg(&src->bonus);
      sm.st[i] = st;
      if (sm.internal[i]) f = st.flags;
    }
  }
  f = __reduce_or_sync(0xffffffffu, f);
  if ((threadIdx.x & 31) == 0 && f) atomicOr(&sm.flags, f);
  __syncthreads();
  if (threadIdx.x == 0) {
    int c = 0, len = 0;
    while (sm.internal[c]) {
      const int fa = sm.st[c].first_acc;
      if (fa <= c || fa >= N || sm.parent[fa] != c) break;  // -1: every child rejected
      sm.path[len++] = fa;
      c = fa;
    }
    sm.path_len = len;
    sm.terminal = c;
  }
  __syncthreads();
  const int c = sm.terminal;
  int flags = sm.flags;
  int bonus = -1;
  if (sm.internal[c]) {
    bonus = sm.st[c].bonus;
  } else if (leaves_done) {
    flags |= sm.st[c].flags;
    bonus = sm.st[c].bonus;
  } else {
    // leaf terminal of a large problem: sweep its row here
    const size_t row_off = ((size_t)b * N + c) * (size_t)V;
    const float* lrow = a.logits + row_off;
    const Slice s = make_slice(lrow, V, rank, CL);
    stage_slice(lrow, s, nb.lbuf, nb.bar_l);
    const int lflags = wait_slice(nb.bar_l, bar_l_used ? 1 : 0);  // CTA-local: published below
    if (a.T == 0.f) {
      publish<CL>(sm, slot, rank, slice_argmax(s, nb.lbuf, lflags));
      float gv;
      int gi;
      reduce_argmax<CL>(sm, slot, gv, gi, flags);
      slot ^= 1;
      bonus = (gi == 0x7fffffff) ? 0 : gi;
    } else {
      const float invT = 1.f / a.T;
      float M;
      DF S;
      cluster_exp_stats<CL>(s, nb.lbuf, invT, lflags, rank, slot, M, S, flags, sm);
      Weights wt;
      wt.kind = Weights::kExp;
      wt.ebuf = nb.lbuf;
      wt.c = 1.f;
      const float u = __ldg(a.uniforms + (size_t)b * N);
      if (!(flags & (SPEC_ST_NONFINITE | SPEC_ST_TIMEOUT)))
        bonus = cluster_sample<CL>(wt, s, rank, u, slot, flags, sm);
    }
  }
  if (flags & (SPEC_ST_NONFINITE | SPEC_ST_TIMEOUT)) bonus = -1;

  if (rank == 0) {
    const int len = sm.path_len;
    const bool ok = bonus >= 0;
    if (threadIdx.x == 0) {
      a.accept_len[b] = ok ? len : -1;
      a.bonus[b] = ok ? bonus : -1;
      if (a.status && flags) atomicOr(a.status + b, flags);
      if (a.child_q) a.child_q[(size_t)b * N] = -1.f;
    }
    for (int i = threadIdx.x; i < N; i += kVThreads) {
      const int node = (ok && i < len) ? sm.path[i] : -1;
      a.acc_tokens[(size_t)b * N + i] = node >= 0 ? sm.tokens[node] : -1;
      if (a.acc_nodes) a.acc_nodes[(size_t)b * N + i] = node;
    }
  }
}

// ------------------------------------------------------------------------------------------------
// per-sequence arrival counter
// ------------------------------------------------------------------------------------------------
// The counter word holds (call generation << 16) | arrivals.  A word carrying another
// generation (left by another call, or never initialised) is claimed for this call -- reset to
// (gen, 0) -- by whichever cluster of the sequence starts first, so no zero-filled workspace is
// needed; every cluster claims before it can arrive, and the last arrival only comes after all of
// them started.  Arrivals are plain atomic adds; the last one resets the count, which keeps
// CUDA-graph replays (same generation) correct.
__device__ __forceinline__ void claim_counter(unsigned long long* ctr, unsigned long long gen) {
  const unsigned long long g = gen & 0xFFFFFFFFFFFFull;
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(ctr);
  for (int it = 0; it < 4 && (old >> 16) != g; ++it) old = atomicCAS(ctr, old, g << 16);
}

// Returns true for the last of the N arrivals.
__device__ __forceinline__ bool arrive(unsigned long long* ctr, unsigned long long gen, int N) {
  const unsigned long long g = gen & 0xFFFFFFFFFFFFull;
  const unsigned long long old = atomicAdd(ctr, 1ull);
  if ((old >> 16) == g && (old & 0xFFFFull) + 1 == (unsigned long long)N) {
    atomicExch(ctr, g << 16);
    return true;
  }
  return false;
}

// ------------------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------------------
template <int CL>
__global__ void __launch_bounds__(kVThreads)
    verify_kernel(const VerifyArgs a, int cap, int eager_probs, int do_leaves, float invT_hi,
                  float invT_lo) {
  extern __shared__ __align__(16) float dyn[];
  __shared__ VerifySmem sm;
  __shared__ __align__(8) uint64_t bars[2];
  const NodeBufs nb{dyn, dyn + cap, dyn + 2 * cap, smem_u32(&bars[0]), smem_u32(&bars[1])};
  const int rank = (CL > 1) ? int(cg::this_cluster().block_rank()) : 0;
  const int j = blockIdx.y, b = blockIdx.z;
  const int N = a.N;
  if (threadIdx.x == 0) {
    mbar_init(nb.bar_l, 1);
    mbar_init(nb.bar_p, 1);
    mbar_fence_init();
  }
  griddep_wait();  // the inputs may be produced by the preceding kernel in the stream
  griddep_launch_dependents();
  // small problems process every node: its logit row is needed whatever the tree looks like, so
  // the copy goes out before anything else
  const bool early = do_leaves != 0;
  if (early) {
    const float* lrow = a.logits + ((size_t)b * N + j) * (size_t)a.V;
    stage_slice(lrow, make_slice(lrow, a.V, rank, CL), nb.lbuf, nb.bar_l);
  }
  if (rank == 0 && threadIdx.x == 0) claim_counter(a.counters + b, a.gen);
  const int bad = load_tree(a, b, sm);  // uniform across the cluster: same tree everywhere
  if (bad) {
    if (j == 0 && rank == 0) {  // one writer per sequence
      if (threadIdx.x == 0) {
        a.accept_len[b] = -1;
        a.bonus[b] = -1;
        if (a.status) atomicOr(a.status + b, bad);
      }
      for (int i = threadIdx.x; i < N; i += kVThreads) {
        a.acc_tokens[(size_t)b * N + i] = -1;
        if (a.acc_nodes) a.acc_nodes[(size_t)b * N + i] = -1;
        if (a.child_q) a.child_q[(size_t)b * N + i] = -1.f;
      }
    }
    if (early) wait_slice(nb.bar_l);  // no copy left in flight
    return;
  }
  int slot = 0;
  const bool work = sm.internal[j] || do_leaves;
  NodeStat st;
  if (work)
    st = process_node<CL>(a, b, j, rank, nb, eager_probs != 0, early, DF{invT_hi, invT_lo}, slot,
                          sm);

  // arrival: the last cluster of the sequence walks the tree
  if (rank == 0 && threadIdx.x == 0) {
    if (work) a.stats[(size_t)b * N + j] = st;
    __threadfence();
    const int last = arrive(a.counters + b, a.gen, N) ? 1 : 0;
    __threadfence();
    if constexpr (CL > 1) {
      for (int r = 0; r < CL; ++r) dsmem_store_u32(dsmem_addr(&sm.is_last, r), (uint32_t)last);
    } else {
      sm.is_last = last;
    }
  }
  cluster_barrier<CL>();
  if (!sm.is_last) return;
  walk_sequence<CL>(a, b, rank, nb, do_leaves != 0, work, slot, sm);
  cluster_barrier<CL>();  // keep shared memory alive for remote stores
}

// ------------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------------
size_t verify_workspace_bytes(int B, int N, int V) {
  (void)V;
  return (size_t)B * N * sizeof(NodeStat) + (size_t)B * N * kMaxNodes * sizeof(double) +
         (size_t)B * sizeof(unsigned long long);
}

template <class... Params, class... Args>
static cudaError_t launch_ex(void (*kern)(Params...), dim3 grid, int cl, size_t smem,
                             cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kVThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Per-buffer slice limit (floats): three buffers plus the static state must fit in a CTA's 227 KB.
constexpr int kMaxSliceFloats = 16 * 1024 + 64;

// Cluster size: large enough that the slice buffers fit; for latency-bound (small) problems as
// large as slices of >= 1024 elements allow; otherwise aim for about one wave of CTAs.
static int pick_cluster(long long units, int V, int num_sms, bool small) {
  int cl = 1;
  while (cl < 8 && slice_capacity(V, cl) > kMaxSliceFloats) cl *= 2;
  if (small) {
    while (cl < 8 && V / (cl * 2) >= 1024) cl *= 2;
    return cl;
  }
  while (cl < 8 && units * (cl * 2) <= (long long)num_sms * 3 / 2 && V / (cl * 2) >= 2048) cl *= 2;
  return cl;
}

bool verify_supported(int V) { return slice_capacity(V, 8) <= kMaxSliceFloats; }

cudaError_t launch_verify(const VerifyArgs& a, int num_sms, cudaStream_t s) {
  const bool small = (long long)a.B * a.N * a.V * 4 <= (64ll << 20);
  // small problems are latency-bound: stage the draft rows eagerly and process leaves speculatively
  const int eager = small ? 1 : 0;
  const int leaves = small ? 1 : 0;
  const long long units = (long long)a.B * (leaves ? a.N : (a.N + 1) / 2);
  const int cl = pick_cluster(units, a.V, num_sms, small);
  const int cap = slice_capacity(a.V, cl);
  const size_t smem = (size_t)(a.T > 0.f ? 3 : 1) * cap * sizeof(float);
  const double invTd = a.T > 0.f ? 1.0 / (double)a.T : 0.0;
  const float invT_hi = (float)invTd, invT_lo = (float)(invTd - (double)invT_hi);
  const dim3 g(cl, a.N, a.B);
  switch (cl) {
    case 1: return launch_ex(verify_kernel<1>, g, 1, smem, s, a, cap, eager, leaves, invT_hi, invT_lo);
    case 2: return launch_ex(verify_kernel<2>, g, 2, smem, s, a, cap, eager, leaves, invT_hi, invT_lo);
    case 4: return launch_ex(verify_kernel<4>, g, 4, smem, s, a, cap, eager, leaves, invT_hi, invT_lo);
    default: return launch_ex(verify_kernel<8>, g, 8, smem, s, a, cap, eager, leaves, invT_hi, invT_lo);
  }
}

}  // namespace spectree
