// Speculative-sampling verification of a draft token tree (sm_103a).
//
// Method: speculative-decoding survey explainer, "Formal Definition" -- draft x~_i ~ p_i is accepted
// if r < min(1, q_i(x~_i) / p_i(x~_i)); at the first rejection c the next token is drawn from
// norm(max(0, q_c - p_c)); greedy verification (taxonomy table) accepts a draft equal to the target's
// argmax.  Tree form: children of the current node are tried in ascending index against the current
// target distribution, which becomes its normalised residual after every rejection (and stays as it
// is when that residual sums to zero).
//
// verify_kernel, grid (CL, N, B): a thread-block cluster of CL CTAs per (sequence, node).
// verify_path_kernel, grid (CL, 1, B), for large problems: one cluster per sequence runs the same
// per-node step on the nodes its walk reaches, in turn (the root, then each accepted child).
//   * Each CTA copies its slice of the node's target-logit row (and, for an internal node at T > 0,
//     of the draft row) into shared memory with bulk async copies, padded with neutral values so
//     that every thread owns a run of `ch` consecutive elements (a multiple of 4).  Runs are in
//     element order across (rank, warp, lane), so per-thread totals give the row's CDF at run
//     boundaries.
//   * T > 0, statistics: each thread takes the max m_t of its run, replaces its logits by
//     e_t(y) = 2^((l_y - m_t) k), k = log2(e) / T, and sums them; warps combine (m, s) pairs, and
//     one cluster exchange of the warp pairs gives M and S = sum_y exp((l_y - M) / T).  The thread
//     keeps f_t = 2^((m_t - M) k), so e(y) = e_t(y) f_t.
//   * Residual rounds in closed form: with w_0 = e, D_0 = S and after rejections 1..k,
//     w_k(y) = max(0, e(y) - c_k p(y)), c_k = D_0 + ... + D_{k-1}, D_k = sum_y w_k(y), and the
//     current distribution is w_k / D_k.  A round is one pass (one FMA per element) and one cluster
//     exchange; a zero D_k freezes the distribution, and nothing after it needs a pass.
//   * Each child is tested with the division-free r * p(x) * D < n(x), n(x) = w(x) tracked in fp64
//     from an exactly formed exp argument; see "Precision".
//   * Bonus draw (inverse CDF, y = min{y : C(y) > u * total}): the CTA totals of the current
//     weights are known from the last exchange, the thread totals from the last pass, so only the
//     crossing CTA scans its warps' and threads' totals and the crossing thread's run (by its
//     warp) -- no extra pass over the row.
//   * The walk.  Small problems without per-child q: each node hands its outcome over in a
//     per-node word as soon as it is done, the walk starts at the root and follows the accepted
//     children as their outcomes appear, and nodes still in their residual rounds stop once the
//     walk cannot reach them (see "walk hand-over").  Otherwise the last cluster of a sequence to
//     finish (a per-sequence arrival counter in the workspace) walks the tree from the root along
//     the accepted children and writes the outputs; when leaves were not processed (large
//     problems) it draws the bonus at a leaf terminal itself.
//
// Precision.  Element weights are fp32 (hardware 2^x on an argument formed as (l - m) * k).  Every
// sum is a compensated fp32 sum per thread and a double-float (pair of fp32) sum across threads and
// CTAs.  No fp64 arithmetic: this part's fp64 pipe is narrow (a dependent operation costs 64
// cycles, a division about 1 us) and shared by every CTA on the SM.
// The accept decisions compare double-floats: n(x) starts as exp((l_x - M)/T) with the argument
// formed exactly as a double-float and exponentiated by expf (a few ulp, about 1e-7 relative), and
// after a rejection n <- max(0, n - p(x) D), D <- D_k.  The double-float products and sums carry
// about 2^-44 themselves; expf's error and that of the fp32 element weights (ex2.approx) summed
// into S and D bound a decision's accuracy at a few 1e-7 relative -- inside the 1e-6 band in which
// decisions are counted, not compared.
#include <cooperative_groups.h>
#include <float.h>

#include "common.cuh"
#include "head_walk.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace spectree {

constexpr int kVThreads = 256;
constexpr int kVWarps = kVThreads / 32;
static_assert(kVWarps == 8, "exchanges and draws combine 8 warps (and at most 8 CTAs) in 8 lanes");
constexpr uint32_t kBulkChunk = 32768;  // bytes per bulk copy instruction

// A warp's or a CTA's partial result in an exchange (32 bytes: two 16-byte stores).
struct __align__(16) Entry {
  float m;     // max (statistics) / value (argmax)
  int idx;     // argmax index
  float s_hi;  // sum (double-float)
  float s_lo;
  int flags;
  int pad[3];
};
static_assert(sizeof(Entry) == 32, "Entry layout");

constexpr int kMaxCluster = 8;  // the portable cluster size

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
  int found;
  uint32_t ticket;       // rank 0: this node's call ticket (online walk); sent with each exchange
  uint32_t ticket_c;     // rank 0's ticket, as received through the exchanges
  unsigned long long hv_guess;  // the node's hand-over word as read at the start (online walk)
  unsigned long long hv_snap[kMaxNodes];  // every node's hand-over word, read when walking
  uint32_t hv_lo;                         // low half of the word the walk continues from
  uint32_t first_polls;  // first-attempt polls of the bounded waits (VerifyArgs::first_polls)
  float g_r[kMaxNodes];         // children's test uniforms
  float g_lx[kMaxNodes];        // gathered target logit / draft probability of each child's token
  float g_px[kMaxNodes];
  DF g_n[kMaxNodes];            // numerators n(x~) of the children's current q values
  Entry wpart[kVWarps];         // this CTA's warp entries of the current exchange
  Entry cpart[2][kMaxCluster];  // every CTA's entry, per exchange slot (sent here by st.async)
  DF wcur[kVWarps];             // totals of the current sampling weights: this CTA's warps,
  DF ccur[kMaxCluster];         // and every CTA of the cluster (e(y) scale)
  NodeStat st[kMaxNodes];
  Entry xres;                     // result of the current exchange (written by warp 0)
  __align__(8) uint64_t xbar[2];  // transaction barriers of the exchange slots
};

__device__ __forceinline__ float ex2f(float x) {  // hardware 2^x
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------------------------------------
// a CTA's slice of a row, staged in shared memory
// ------------------------------------------------------------------------------------------------
// Elements [lo, hi) of the row belong to this CTA.  [blo, bhi) is the 16-byte aligned part that is
// bulk-copied; the rest (at most 3 elements at each end of the row) is loaded with plain loads.
// Element y sits at buf[y - sbase]; sbase keeps the bulk part 16-byte aligned in shared memory.
// Thread t owns buffer positions [t ch, (t + 1) ch); positions outside [lo, hi) - sbase are pads.
struct Slice {
  int lo, hi, blo, bhi, sbase, ch;
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
  const int nbuf = s.hi - s.sbase;
  s.ch = 4 * ((nbuf + 4 * kVThreads - 1) / (4 * kVThreads));
  return s;
}

// The draft probabilities of a slice, at the positions of the logit buffer: either staged in
// shared memory (sbuf) or read from the row in global memory (through L2) -- positions outside
// [lo, hi) - sbase are pads and read as 0, as the staged pads do.  row + sbase is 16-byte aligned
// (make_slice keeps it so), so whole float4s inside the slice load as float4.
template <bool GLOBAL>
struct DraftSlice;

template <>
struct DraftSlice<false> {  // staged
  const float* sbuf;
  __device__ __forceinline__ float4 load4(int pos) const {
    return *reinterpret_cast<const float4*>(sbuf + pos);
  }
  __device__ __forceinline__ float at(int pos) const { return sbuf[pos]; }
};

template <>
struct DraftSlice<true> {  // read from the row in global memory
  const float* grow;
  int sbase, lo, hi;
  __device__ __forceinline__ float at(int pos) const {
    const int y = sbase + pos;
    return (y >= lo && y < hi) ? __ldg(grow + y) : 0.f;
  }
  __device__ __forceinline__ float4 load4(int pos) const {
    const int y = sbase + pos;
    if (y >= lo && y + 4 <= hi) return __ldg(reinterpret_cast<const float4*>(grow + y));
    return make_float4(at(pos), at(pos + 1), at(pos + 2), at(pos + 3));
  }
};

// Floats of shared memory one slice buffer needs for (V, CL): the widest slice (with its ragged
// ends) rounded up to whole runs.
static inline int slice_capacity(int V, int cl) {
  const int nbuf = 4 * ((V / 4 + 1 + cl - 1) / cl) + 8;
  return kVThreads * 4 * ((nbuf + 4 * kVThreads - 1) / (4 * kVThreads));
}

// Issue the copies of the slice into buf (thread 0 issues the bulk part; the ragged ends are
// loaded by the first threads) and fill the pads with `pad`.  Completion: the barrier's phase,
// then __syncthreads().
__device__ __forceinline__ void stage_slice(const float* row, const Slice& s, float* buf,
                                            uint32_t bar, float pad) {
  if (threadIdx.x == 0) {
    const uint32_t bytes = uint32_t(s.bhi - s.blo) * 4u;
    mbar_arrive_expect_tx(bar, bytes);
    const uint32_t dst = smem_u32(buf + (s.blo - s.sbase));
    for (uint32_t off = 0; off < bytes; off += kBulkChunk)
      bulk_load(dst + off, row + s.blo + off / 4, min(kBulkChunk, bytes - off), bar);
  }
  const int t = threadIdx.x;
  const int head = s.blo - s.lo, tail = s.hi - s.bhi;
  if (t < head) buf[s.lo + t - s.sbase] = __ldg(row + s.lo + t);
  if (t < tail) buf[s.bhi + t - s.sbase] = __ldg(row + s.bhi + t);
  const int pre = s.lo - s.sbase, post0 = s.hi - s.sbase, post1 = kVThreads * s.ch;
  if (t < pre) buf[t] = pad;
  for (int i = post0 + t; i < post1; i += kVThreads) buf[i] = pad;
}

// Wait for a staged slice (phase `parity` of its barrier: 0 for the barrier's first use in this
// launch, 1 for its second); returns SPEC_ST_TIMEOUT if the copy did not land within `polls`
// polls, after giving copies still in flight a second wait with the full limit (so that no copy
// is left in flight when the CTA moves on).
__device__ __forceinline__ int wait_slice(uint32_t bar, uint32_t parity, uint32_t polls) {
  int st = 0;
  if (!mbar_wait(bar, parity, polls)) {
    st = SPEC_ST_TIMEOUT;
    mbar_wait(bar, parity);
  }
  __syncthreads();
  return st;
}

// argmax with lowest index on ties (indices compared unsigned); NaN never wins.
__device__ __forceinline__ void argmax_merge(float& bv, int& bi, float v, int i) {
  if (v > bv || (v == bv && (unsigned)i < (unsigned)bi)) {
    bv = v;
    bi = i;
  }
}

template <int CL>
__device__ __forceinline__ void cluster_barrier() {
  if constexpr (CL > 1) {
    cg::this_cluster().sync();
  } else {
    __syncthreads();
  }
}

// ------------------------------------------------------------------------------------------------
// cluster exchanges
// ------------------------------------------------------------------------------------------------
// An exchange combines one entry per warp into a cluster-wide result.  The warps' entries are first
// combined inside the CTA; warp 0 then sends the CTA's entry to every CTA of the cluster with
// st.async, whose completion is counted on the receiver's transaction mbarrier (a one-way trip,
// no cluster barrier).  Every CTA then combines the CL entries in rank order.  Two slots alternate;
// slot s of exchange x waits for phase (x / 2) & 1 of its barrier.  A CTA can send exchange x + 2
// only after exchange x + 1 completed everywhere it reads from, and every CTA passes a
// __syncthreads (step 1) after reading exchange x, so slots are never overwritten early.
enum XKind { kXSum = 0, kXMaxSum = 1, kXArgmax = 2 };

template <int KIND>
__device__ __forceinline__ Entry entry_identity() {
  return KIND == kXArgmax ? Entry{-INFINITY, 0x7fffffff, 0.f, 0.f, 0, {0, 0, 0}}
                          : Entry{-INFINITY, 0, 0.f, 0.f, 0, {0, 0, 0}};
}

// Combination of the entries held by lanes 0..7 (in lane order; the other lanes hold the identity),
// in every lane: sums in lane order, max-sums rescaled to the largest max first (k = log2(e) / T),
// argmax with the lower index on ties.  One code path per kind and no divergence: at every level
// of the butterfly both lanes of a pair take the lower lane's operand first (selects), so every
// lane ends with the same bits.
template <int KIND>
__device__ __forceinline__ Entry lanes_combine8(Entry e, float k) {
  const int lane = threadIdx.x & 31;
  e.flags = __reduce_or_sync(0xffffffffu, e.flags);
  if constexpr (KIND == kXArgmax) {
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, e.m, o);
      const int oi = __shfl_xor_sync(0xffffffffu, e.idx, o);
      const bool upper = (lane & o) != 0;
      float am = upper ? ov : e.m;
      int ai = upper ? oi : e.idx;
      argmax_merge(am, ai, upper ? e.m : ov, upper ? e.idx : oi);
      e.m = am;
      e.idx = ai;
    }
  } else {
    if constexpr (KIND == kXMaxSum) {
      float M = e.m;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float f = (e.m == -INFINITY) ? 0.f : ex2f(__fmul_rn(__fsub_rn(e.m, M), k));
      const DF sc = df_scale(DF{e.s_hi, e.s_lo}, f);
      e.m = M;
      e.s_hi = sc.hi;
      e.s_lo = sc.lo;
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
      const DF w{__shfl_xor_sync(0xffffffffu, e.s_hi, o), __shfl_xor_sync(0xffffffffu, e.s_lo, o)};
      const DF v{e.s_hi, e.s_lo};
      const bool upper = (lane & o) != 0;
      const DF s = df_add(upper ? w : v, upper ? v : w);
      e.s_hi = s.hi;
      e.s_lo = s.lo;
    }
  }
  return e;
}

// One exchange; returns the cluster-wide combination (in every thread).  `mine` is this warp's
// entry (warp-uniform).  Warp 0 combines the CTA's warps, sends, waits for the CL entries and
// combines them; the others meet it at a __syncthreads.  After it, sm.cpart[slot][r] holds CTA
// r's entry (slot returned through xslot).  A wait that gives up sets SPEC_ST_TIMEOUT.
template <int CL, int KIND>
__device__ Entry exchange(VerifySmem& sm, int& xk, const Entry& mine, float k, int rank,
                          int& xslot) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) sm.wpart[wid] = mine;
  __syncthreads();
  const int slot = xk & 1;
  const uint32_t parity = (xk >> 1) & 1;
  ++xk;
  xslot = slot;
  if (wid == 0) {
    const uint32_t bar = smem_u32(&sm.xbar[slot]);
    Entry c = lanes_combine8<KIND>(lane < kVWarps ? sm.wpart[lane] : entry_identity<KIND>(), k);
    c.pad[0] = (int)sm.ticket;  // rank 0's reaches every CTA (the online walk's call ticket)
    if (lane == 0) mbar_arrive_expect_tx(bar, CL * (uint32_t)sizeof(Entry));
    if (lane < CL) {
      const uint32_t dst = dsmem_addr(&sm.cpart[slot][rank], lane);
      const uint32_t rbar = dsmem_addr(&sm.xbar[slot], lane);
      const uint4* v = reinterpret_cast<const uint4*>(&c);
      st_async_v4(dst, v[0], rbar);
      st_async_v4(dst + 16, v[1], rbar);
    }
    // a first attempt that gives up flags the exchange, then the peers' stores are waited for
    // with the full limit: no CTA moves on (or exits) with a store into it still in flight
    const bool ok = __all_sync(0xffffffffu, mbar_wait_acq_cluster(bar, parity, sm.first_polls));
    if (!ok) mbar_wait_acq_cluster(bar, parity);
    Entry r = lanes_combine8<KIND>(lane < CL ? sm.cpart[slot][lane] : entry_identity<KIND>(), k);
    if (lane == 0) {
      sm.ticket_c = (uint32_t)sm.cpart[slot][0].pad[0];
      r.flags |= ok ? 0 : SPEC_ST_TIMEOUT;
      sm.xres = r;
    }
  }
  __syncthreads();
  return sm.xres;
}

// ------------------------------------------------------------------------------------------------
// passes over a thread's run
// ------------------------------------------------------------------------------------------------
// A run of n4 = ch / 4 float4s starting at lane-dependent offsets: read in place order, the eight
// lanes of a quarter-warp would hit the same banks whenever n4 is even.  Each thread visits its
// float4s rotated by rot(lane) (c -> (c + rot) mod n4), which spreads every quarter-warp over all
// 32 banks: with d = gcd(n4, 8), lane * n4 mod 8 repeats every 8 / d lanes and rot adds
// (lane mod 8) * d / 8 to tell the repeats apart.
struct RunWalk {
  int n4, rot;
  __device__ __forceinline__ explicit RunWalk(int ch) {
    n4 = ch >> 2;
    const int d = min(n4 & -n4, 8);
    rot = ((threadIdx.x & 7) * d) >> 3;
  }
  __device__ __forceinline__ int at(int c) const {  // c-th visited float4 of the run
    const int cc = c + rot;
    return cc >= n4 ? cc - n4 : cc;
  }
};

__device__ __forceinline__ void warp_argmax(float& bv, int& bi) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    argmax_merge(bv, bi, ov, oi);
  }
}

// T = 0: argmax of the row (cluster-wide), NaN / +Inf flagged.
template <int CL>
__device__ void cluster_argmax(const Slice& s, const float* lbuf, int lflags, int rank, int& xk,
                               float& gv, int& gi, int& flags, VerifySmem& sm) {
  const float4* L4 = reinterpret_cast<const float4*>(lbuf + threadIdx.x * s.ch);
  const int y0 = threadIdx.x * s.ch + s.sbase;  // element of the run's first position
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  bool bad = false;
  const RunWalk rw(s.ch);
  for (int c = 0; c < rw.n4; ++c) {
    const int q = rw.at(c);
    const float4 v = L4[q];
    bad |= !(v.x <= FLT_MAX) | !(v.y <= FLT_MAX) | !(v.z <= FLT_MAX) | !(v.w <= FLT_MAX);
    argmax_merge(bv, bi, v.x, y0 + 4 * q);  // index tie-break: the visiting order is rotated
    argmax_merge(bv, bi, v.y, y0 + 4 * q + 1);
    argmax_merge(bv, bi, v.z, y0 + 4 * q + 2);
    argmax_merge(bv, bi, v.w, y0 + 4 * q + 3);
  }
  if (bi == 0x7fffffff) {  // nothing above -inf: the run's first real element (pads are -inf)
    const int first = max(y0, s.lo);
    bi = first < min(y0 + s.ch, s.hi) ? first : 0x7fffffff;
  }
  warp_argmax(bv, bi);
  const int f = __reduce_or_sync(0xffffffffu, bad ? SPEC_ST_NONFINITE : 0) | lflags;
  int xs;
  const Entry r =
      exchange<CL, kXArgmax>(sm, xk, Entry{bv, bi, 0.f, 0.f, f, {0, 0, 0}}, 0.f, rank, xs);
  gv = r.m;
  gi = r.idx;
  flags |= r.flags;
}

// Per-thread state of a node at T > 0.
struct RunState {
  float f;    // 2^((m_t - M) k): e(y) = e_t(y) f over the thread's run
  DF tot;     // the thread's total of the current sampling weights (e(y) scale)
  float cw;   // current weights max(0, e_t(y) - cw p(y)) f; cw = 0: w = e (p not read)
};

// T > 0: e_t(y) replaces the logits; returns M, S (cluster-wide) and the thread's state.  The
// totals of e(y) per CTA of the cluster go to sm.ccur.
template <int CL>
__device__ void cluster_stats(const Slice& s, float* lbuf, float k, int lflags, int rank, int& xk,
                              float& M, DF& S, RunState& rs, int& flags, VerifySmem& sm) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  float4* L4 = reinterpret_cast<float4*>(lbuf + threadIdx.x * s.ch);
  const RunWalk rw(s.ch);
  float m = -INFINITY;
  for (int c = 0; c < rw.n4; ++c) {
    const float4 v = L4[rw.at(c)];
    m = fmaxf(m, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
  }
  const float mm = (m == -INFINITY) ? 0.f : m;  // NaN / +Inf reach S and are flagged there
  CompSum acc;
  for (int c = 0; c < rw.n4; ++c) {
    const int q = rw.at(c);
    float4 v = L4[q];
    v.x = ex2f(__fmul_rn(__fsub_rn(v.x, mm), k));
    v.y = ex2f(__fmul_rn(__fsub_rn(v.y, mm), k));
    v.z = ex2f(__fmul_rn(__fsub_rn(v.z, mm), k));
    v.w = ex2f(__fmul_rn(__fsub_rn(v.w, mm), k));
    L4[q] = v;
    acc.add(__fadd_rn(__fadd_rn(v.x, v.y), __fadd_rn(v.z, v.w)));
  }
  const DF st = df_from(acc);
  const float mw = warp_max_f(m);
  const float g = (m == -INFINITY) ? 0.f : ex2f(__fmul_rn(__fsub_rn(m, mw), k));
  const DF sw = warp_sum_df(df_scale(st, g));
  int xs;
  const Entry r =
      exchange<CL, kXMaxSum>(sm, xk, Entry{mw, 0, sw.hi, sw.lo, lflags, {0, 0, 0}}, k, rank, xs);
  M = r.m;
  S = DF{r.s_hi, r.s_lo};
  flags |= r.flags;
  // sampling state of q^(0): thread, warp and CTA totals of e(y)
  rs.f = (m == -INFINITY) ? 0.f : ex2f(__fmul_rn(__fsub_rn(m, M), k));
  rs.tot = df_scale(st, rs.f);
  rs.cw = 0.f;
  if (wid == 0 && lane < CL) {
    const Entry& c = sm.cpart[xs][lane];
    const float fc = (c.m == -INFINITY) ? 0.f : ex2f(__fmul_rn(__fsub_rn(c.m, M), k));
    sm.ccur[lane] = df_scale(DF{c.s_hi, c.s_lo}, fc);
  }
  if (!(S.hi > 0.f) || !(S.hi <= FLT_MAX)) flags |= SPEC_ST_NONFINITE;
}

// Residual round: returns D = sum_y max(0, e(y) - c p(y)) (cluster-wide; c_t = c / f).  check_p:
// flag bad draft values.  The thread's total of the new weights goes to `tot`, the warp's to
// `wt`; `xs` is the slot whose sm.cpart holds the CTA totals.
// `late()`: more flags of this thread, taken after its pass over the slice (the results of loads
// issued before the call, whose round trips the pass hides).
struct NoLateFlags {
  __device__ __forceinline__ int operator()() const { return 0; }
};
template <int CL, class PD, class Late = NoLateFlags>
__device__ DF cluster_residual(const Slice& s, const float* ebuf, const PD& pd, float c_t,
                               float f, bool check_p, int lflags, int rank, int& xk, DF& tot,
                               DF& wt, int& xs, int& flags, VerifySmem& sm, Late late = Late()) {
  const float4* E4 = reinterpret_cast<const float4*>(ebuf + threadIdx.x * s.ch);
  const int p0 = threadIdx.x * s.ch;
  CompSum acc;
  float pmin = 0.f, psum = 0.f;
  const RunWalk rw(s.ch);
  for (int c = 0; c < rw.n4; ++c) {
    const int q = rw.at(c);
    const float4 e = E4[q], p = pd.load4(p0 + 4 * q);
    const float r0 = fmaxf(fmaf(-c_t, p.x, e.x), 0.f);
    const float r1 = fmaxf(fmaf(-c_t, p.y, e.y), 0.f);
    const float r2 = fmaxf(fmaf(-c_t, p.z, e.z), 0.f);
    const float r3 = fmaxf(fmaf(-c_t, p.w, e.w), 0.f);
    acc.add(__fadd_rn(__fadd_rn(r0, r1), __fadd_rn(r2, r3)));
    if (check_p) {
      pmin = fminf(pmin, fminf(fminf(p.x, p.y), fminf(p.z, p.w)));
      psum += (p.x + p.y) + (p.z + p.w);
    }
  }
  const bool bad = check_p && (pmin < 0.f || !(psum <= FLT_MAX));  // NaN, +Inf or negative p
  tot = df_scale(df_from(acc), f);
  wt = warp_sum_df(tot);
  const int wf = __reduce_or_sync(0xffffffffu, bad ? SPEC_ST_NONFINITE : 0) | lflags | late();
  const Entry r =
      exchange<CL, kXSum>(sm, xk, Entry{0.f, 0, wt.hi, wt.lo, wf, {0, 0, 0}}, 0.f, rank, xs);
  flags |= r.flags;
  return DF{r.s_hi, r.s_lo};
}

// The current weights became those of this round: record its CTA totals for a draw.
template <int CL>
__device__ __forceinline__ void commit_round_totals(VerifySmem& sm, int xs) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (wid == 0 && lane < CL) sm.ccur[lane] = DF{sm.cpart[xs][lane].s_hi, sm.cpart[xs][lane].s_lo};
}

// ------------------------------------------------------------------------------------------------
// inverse-CDF draw: y = min{y : C(y) > u * total}, else the last y with a positive weight
// ------------------------------------------------------------------------------------------------
// Over the lanes' values v (DF, in order; incl = their inclusive scan): the first lane whose
// inclusive prefix exceeds t, with the prefix before it; if none does (or t < 0: "last positive"
// mode), the last lane with a positive value (-1 if none), and t becomes -1.
__device__ __forceinline__ int lane_crossing(DF v, DF incl, DF& t, DF& before) {
  const int lane = threadIdx.x & 31;
  DF excl{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
  if (lane == 0) excl = DF{0.f, 0.f};
  const unsigned cross = __ballot_sync(0xffffffffu, t.hi >= 0.f && df_gt(incl, t));
  if (cross) {
    const int L = __ffs(cross) - 1;
    before = DF{__shfl_sync(0xffffffffu, excl.hi, L), __shfl_sync(0xffffffffu, excl.lo, L)};
    return L;
  }
  const unsigned pos = __ballot_sync(0xffffffffu, v.hi > 0.f);
  t = DF{-1.f, 0.f};
  before = DF{0.f, 0.f};
  return pos ? 31 - __clz(pos) : -1;
}

// Weight of buffer position i under the state (cw, f) (e(y) scale).
template <class PD>
__device__ __forceinline__ float weight_at(const float* ebuf, const PD& pd, int i, float cw,
                                          float f) {
  const float e = ebuf[i];
  const float w = (cw == 0.f) ? e : fmaxf(fmaf(-cw, pd.at(i), e), 0.f);
  return __fmul_rn(w, f);
}

// Result of a draw: every CTA of the cluster agrees on `writer`, the CTA that holds the crossing
// (rank 0 if every weight is zero); `tok` is valid there (-1: every weight is zero).
struct Draw {
  int writer, tok;
};

// Levels: CTA of the cluster (sm.ccur, same in every CTA), warp of that CTA (sums of rs.tot),
// thread of that warp (rs.tot), element of that thread's run.  No exchange: the writer CTA finds
// the token alone and records the node itself.
template <int CL, class PD>
__device__ Draw cluster_draw(const Slice& s, const float* ebuf, const PD& pd,
                             const RunState& rs, float u, int rank, VerifySmem& sm) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  __syncthreads();  // sm.ccur is visible
  // level 1: CTA (lanes 0..7; lanes past CL hold zeros)
  const DF cv = lane < CL ? sm.ccur[lane] : DF{0.f, 0.f};
  const DF cincl = warp_scan8_df(cv);
  const DF tot{__shfl_sync(0xffffffffu, cincl.hi, 7), __shfl_sync(0xffffffffu, cincl.lo, 7)};
  DF t = (tot.hi > 0.f) ? df_scale(tot, u) : DF{-1.f, 0.f};
  DF before;
  const int cstar = lane_crossing(cv, cincl, t, before);
  if (cstar < 0) return Draw{0, -1};  // nothing positive anywhere
  if (rank != cstar) return Draw{cstar, -1};
  // every warp scans its threads' totals before the warp is chosen (the scans run side by side
  // instead of one after the search of level 2); a warp's total is its last lane's prefix, so
  // levels 2 and 3 agree on it
  const DF lincl = warp_scan_df(rs.tot);
  if (lane == 31) sm.wcur[wid] = lincl;
  __syncthreads();
  // level 2: warp of this CTA (every warp computes it; one acts)
  if (t.hi >= 0.f) t = df_add(t, DF{-before.hi, -before.lo});
  const DF wv = lane < kVWarps ? sm.wcur[lane] : DF{0.f, 0.f};
  int wstar = lane_crossing(wv, warp_scan8_df(wv), t, before);
  if (wstar < 0) wstar = kVWarps - 1;  // rounding: the CTA total was positive but no warp's is
  if (wid == wstar) {
    // level 3: thread of the crossing warp
    if (t.hi >= 0.f) t = df_add(t, DF{-before.hi, -before.lo});
    int Lc = lane_crossing(rs.tot, lincl, t, before);
    if (Lc < 0) Lc = 31;
    // level 4: the elements of that thread's run, 32 at a time, by the whole warp
    const float fL = __shfl_sync(0xffffffffu, rs.f, Lc);
    const float cwL = __shfl_sync(0xffffffffu, rs.cw, Lc);
    const int i0 = (wid * 32 + Lc) * s.ch;
    const DF t3 = (t.hi >= 0.f) ? df_add(t, DF{-before.hi, -before.lo}) : t;
    int y = -1, last_pos = -1;
    DF carry{0.f, 0.f};
    for (int base = 0; base < s.ch; base += 32) {
      const int i = base + lane;
      const float w = (i < s.ch) ? weight_at(ebuf, pd, i0 + i, cwL, fL) : 0.f;
      const DF run = df_add(carry, warp_scan_df(DF{w, 0.f}));
      const unsigned pos = __ballot_sync(0xffffffffu, w > 0.f);
      if (pos) last_pos = base + 31 - __clz(pos);
      const unsigned hb = __ballot_sync(0xffffffffu, t3.hi >= 0.f && df_gt(run, t3));
      if (hb) {
        y = base + __ffs(hb) - 1;
        break;
      }
      carry = DF{__shfl_sync(0xffffffffu, run.hi, 31), __shfl_sync(0xffffffffu, run.lo, 31)};
    }
    if (y < 0) y = last_pos;
    if (lane == 0) sm.found = (y >= 0) ? i0 + y + s.sbase : -1;
  }
  __syncthreads();
  return Draw{cstar, sm.found};
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

// Numerator e(x) = exp((l_x - M) / T) of a child's q^(0), as a double-float: the argument is
// formed exactly as a double-float, exponentiated by expf on its high part and corrected by
// (1 + low part).  Below expf's normal range (weights under 2^-126 of the row max) it is 0.
__device__ __forceinline__ DF child_numerator(float lx, float M, DF invT) {
  const DF d = df_two_sum(lx, -M);
  const DF a = df_mul(d, invT);
  if (!(a.hi >= -87.f)) return DF{0.f, 0.f};
  const float e = expf(a.hi);
  return df_fast_two_sum(e, __fmul_rn(e, a.lo));
}

struct NodeBufs {
  float* lbuf;  // logits, then e_t(y) at T > 0
  float* pbuf;  // draft probabilities
  uint32_t bar_l, bar_p;
};

// Exchange flag (never a status bit): some CTA of the cluster saw that the walk cannot reach the
// node (it ended, or took another branch), so the node's outcome is no longer needed.
constexpr int kWalkDone = 1 << 20;

// The upper half of this call's hand-over and walk-done words: a hash of the generation, offset
// by the call's epoch (replays of one captured call share the generation, not the epoch), with
// the top bit set -- which no zero word, small integer, non-negative count or record field left by
// another call carries, and which other words match only by chance.
__device__ __forceinline__ unsigned long long handover_tag(unsigned long long gen, uint32_t epoch) {
  uint32_t h = (uint32_t)gen * 0x9E3779B1u;
  h ^= h >> 15;
  h += epoch * 0x2545F491u;  // odd: distinct epochs, distinct tags (below 2^31 apart)
  h |= 0x80000000u;
  return h == 0xFFFFFFFFu ? 0x80000001ull : (unsigned long long)h;
}

// The walk can no longer reach node j (its outcome is not needed) once the walk has ended, or once
// an ancestor P on j's chain handed over an outcome other than "accept the child on the way to j"
// (a terminal, or another child).  Thread 0 loads the walk-done word and the hand-over words of
// the nearest kProbeDepth ancestors; `stop` reads them (false in every other thread).
constexpr int kProbeDepth = 3;
constexpr uint32_t kHandoverPublished = 1u << 31, kHandoverTerminal = 1u << 29;
constexpr uint32_t kHandoverValueMask = (1u << 22) - 1u;
struct StopProbe {
  unsigned long long done = 0, anc[kProbeDepth];
  int child[kProbeDepth];  // the child of that ancestor on the way to j
  int n = 0;
  __device__ static StopProbe issue(const VerifyArgs& a, int b, int j, bool me,
                                    const VerifySmem& sm) {
    StopProbe p;
    if (!me) return p;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(p.done) : "l"(a.walk_done + b)
                 : "memory");
    const unsigned long long* w = a.handover + (size_t)b * a.N;
#pragma unroll
    for (int k = 0; k < kProbeDepth; ++k) {
      const int c = k == 0 ? j : p.child[k - 1] > 0 ? sm.parent[p.child[k - 1]] : 0;
      p.child[k] = c;
      p.anc[k] = 0;
      if (c > 0) {
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(p.anc[k]) : "l"(w + sm.parent[c])
                     : "memory");
        p.n = k + 1;
      }
    }
    return p;
  }
  __device__ bool stop(const VerifyArgs& a, int j, unsigned long long tag) const {
    if ((done >> 32) == tag && (done & 1ull)) return true;
    bool off = false;
#pragma unroll
    for (int k = 0; k < kProbeDepth; ++k) {
      const unsigned long long v = anc[k];
      const uint32_t lo = (uint32_t)v;
      if (k < n && (v >> 32) == tag && (lo & kHandoverPublished) &&
          ((lo & kHandoverTerminal) || (int)(lo & kHandoverValueMask) - 1 != child[k]))
        off = true;
    }
    (void)a;
    (void)j;
    return off;
  }
};

// ------------------------------------------------------------------------------------------------
// one node: statistics, sibling tests, residual rounds, bonus if the walk can stop here
// ------------------------------------------------------------------------------------------------
// logits_staged: the kernel already issued the copy of this node's logit slice into nb.lbuf.
// ph_l, ph_p: the phases of the staging barriers' next waits (flipped here after each wait), so
// that one CTA can process several nodes in turn.
// The returned record is complete in CTA `writer` (every CTA gets the same writer); first_acc,
// flags and (at T = 0) the bonus are the same in every CTA.
// ONLINE: the walk runs while nodes finish (every-node form without per-child q); a node stops at
// the residual round in which it learns that the walk cannot reach it (StopProbe; its record then
// flags kWalkDone).
// HEAD: the node's logit row is the head-driven verification's row slot (a.head_rows).
template <int CL, bool PGLOBAL, bool SAMPLING, bool ONLINE = false, bool HEAD = false>
__device__ NodeStat process_node(const VerifyArgs& a, int b, int j, int rank, const NodeBufs& nb,
                                 bool logits_staged, DF invT_df, float k2, int& xk, int& writer,
                                 uint32_t& ph_l, uint32_t& ph_p, VerifySmem& sm) {
  const int N = a.N, V = a.V;
  list_children(j, N, sm);
  const int nk = sm.nk;
  const size_t row_off = ((size_t)b * N + j) * (size_t)V;
  const float* lrow = HEAD ? a.head_rows + head_row_offset(b, j, N, V) : a.logits + row_off;
  const float* prow = a.probs ? a.probs + row_off : nullptr;
  const Slice s = make_slice(lrow, V, rank, CL);  // the draft row has the same alignment
  constexpr bool sampling = SAMPLING;  // T > 0 (T == 0: greedy)
  if (!logits_staged) stage_slice(lrow, s, nb.lbuf, nb.bar_l, -INFINITY);
  const bool probs_staged = sampling && nk > 0 && !PGLOBAL;
  if (probs_staged) stage_slice(prow, s, nb.pbuf, nb.bar_p, 0.f);
  DraftSlice<PGLOBAL> pd;
  if constexpr (PGLOBAL) {
    pd = DraftSlice<true>{prow, s.sbase, s.lo, s.hi};
  } else {
    pd = DraftSlice<false>{nb.pbuf};
  }
  if ((int)threadIdx.x < nk) {  // gathers for the tests, overlapping the bulk copies
    const int kid = sm.kids[threadIdx.x];
    const int x = sm.tokens[kid];
    sm.g_lx[threadIdx.x] = __ldg(lrow + x);
    sm.g_px[threadIdx.x] = sampling ? __ldg(prow + x) : 0.f;
    sm.g_r[threadIdx.x] = __ldg(a.uniforms + (size_t)b * N + kid);
  }
  const float u_bonus = __ldg(a.uniforms + (size_t)b * N);
  const int lflags0 = wait_slice(nb.bar_l, ph_l, sm.first_polls);
  ph_l ^= 1u;
  int flags = 0;  // cluster-uniform: only ever updated from published partials
  writer = 0;
  NodeStat st;
  st.bonus = -1;
  st.s_hi = st.s_lo = 0.f;

  if constexpr (!sampling) {
    float gv;
    int gi;
    cluster_argmax<CL>(s, nb.lbuf, lflags0, rank, xk, gv, gi, flags, sm);
    if (gi < 0 || gi >= V) gi = 0;  // every value NaN: flagged
    int first = -1, nrej = nk;
    for (int t = 0; t < nk; ++t)
      if (sm.tokens[sm.kids[t]] == gi) {
        first = sm.kids[t];
        nrej = t;
        break;
      }
    if (rank == 0 && a.child_q && (int)threadIdx.x < nk) {
      const int kid = sm.kids[threadIdx.x];
      a.child_q[(size_t)b * N + kid] =
          (int)threadIdx.x <= nrej ? (sm.tokens[kid] == gi ? 1.f : 0.f) : -1.f;
    }
    st.m = gv;
    st.argmax = gi;
    st.first_acc = first;
    st.nrej = nrej;
    st.flags = flags;
    st.bonus = gi;  // the bonus wherever the walk stops here
    return st;
  } else {

  // ---- T > 0: statistics of q_j = softmax(l_j / T); e_t(y) replaces the logits in lbuf
  float M;
  DF S;
  RunState rs;
  cluster_stats<CL>(s, nb.lbuf, k2, lflags0, rank, xk, M, S, rs, flags, sm);
  // the online walk's tag: rank 0's call ticket arrived with that exchange
  const unsigned long long hv_tag = ONLINE ? handover_tag(a.gen, sm.ticket_c / (uint32_t)N) : 0ull;
  // Scalars every thread holds stay double-float: fp64 here is only for the few threads that
  // take a decision or update a numerator.
  DF D = S;
  if ((int)threadIdx.x < nk)
    sm.g_n[threadIdx.x] = child_numerator(sm.g_lx[threadIdx.x], M, invT_df);
  if (__syncthreads_or((int)threadIdx.x < nk && !(sm.g_px[threadIdx.x] >= 0.f &&
                                                   sm.g_px[threadIdx.x] <= FLT_MAX)))
    flags |= SPEC_ST_NONFINITE;

  int first = -1, nrej = nk;
  bool all_rejected = nk > 0;
  DF c{0.f, 0.f};  // current weights: max(0, e - c p)
  bool frozen = false, p_waited = false;
  int pflags = 0;
  for (int t = 0; t < nk; ++t) {
    const int kid = sm.kids[t];
    if ((int)threadIdx.x == t) {
      const DF n = sm.g_n[t];
      const DF rpD = df_mul(df_two_prod(sm.g_r[t], sm.g_px[t]), D);
      sm.decision = df_gt(n, rpD) ? 1 : 0;  // r < min(1, q/p) with q = n / D
      if (rank == 0 && a.child_q)
        a.child_q[(size_t)b * N + kid] = D.hi > 0.f ? __fdiv_rn(__fadd_rn(n.hi, n.lo), D.hi) : 0.f;
    }
    __syncthreads();
    if (sm.decision) {
      first = kid;
      nrej = t;
      all_rejected = false;
      break;
    }
    if (frozen) continue;  // a zero residual keeps the distribution: nothing to compute
    // rejected: residual of the current distribution (needed by the next sibling or the draw)
    if (!p_waited) {
      // CTA-local: reaches the cluster through the partials
      if (probs_staged) {
        pflags = wait_slice(nb.bar_p, ph_p, sm.first_polls);
        ph_p ^= 1u;
      }
      p_waited = true;
    }
    const DF c_next = df_add(c, D);
    const float c_t = rs.f > 0.f ? __fdiv_rn(__fadd_rn(c_next.hi, c_next.lo), rs.f) : 0.f;
    DF tot, wt;
    int xs;
    DF G;
    if constexpr (ONLINE) {
      // is this node's outcome still needed?  Loads issued now, read after the slice pass
      const StopProbe probe = StopProbe::issue(a, b, j, threadIdx.x == 0, sm);
      G = cluster_residual<CL>(s, nb.lbuf, pd, c_t, rs.f, t == 0, pflags, rank, xk, tot, wt, xs,
                               flags, sm,
                               [&] { return probe.stop(a, j, hv_tag) ? kWalkDone : 0; });
    } else {
      G = cluster_residual<CL>(s, nb.lbuf, pd, c_t, rs.f, t == 0, pflags, rank, xk, tot, wt, xs,
                               flags, sm);
    }
    pflags = 0;
    if constexpr (ONLINE) {
      if (flags & kWalkDone) {  // cluster-uniform (exchanged); no copy is in flight
        st.flags = flags;
        return st;
      }
    }
    if (G.hi > 0.f) {
      if ((int)threadIdx.x > t && (int)threadIdx.x < nk) {  // n <- max(0, n - p(x) D)
        const DF pD = df_mul(DF{sm.g_px[threadIdx.x], 0.f}, D);
        const DF nn = df_add(sm.g_n[threadIdx.x], DF{-pD.hi, -pD.lo});
        sm.g_n[threadIdx.x] = nn.hi > 0.f ? nn : DF{0.f, 0.f};
      }
      D = G;
      c = c_next;
      rs.tot = tot;
      rs.cw = c_t;
      commit_round_totals<CL>(sm, xs);
    } else {
      frozen = true;
    }
    __syncthreads();
  }
  if (probs_staged && !p_waited) {  // no copy left in flight (not needed)
    wait_slice(nb.bar_p, ph_p, kSpinLimit);
    ph_p ^= 1u;
  }
  const bool bad = (flags & (SPEC_ST_NONFINITE | SPEC_ST_TIMEOUT)) != 0;
  if ((nk == 0 || all_rejected) && !bad) {  // the walk can stop here: draw its bonus
    const Draw d = cluster_draw<CL>(s, nb.lbuf, pd, rs, u_bonus, rank, sm);
    writer = d.writer;
    st.bonus = d.tok;
  }
  if (rank == 0 && a.child_q && (int)threadIdx.x > nrej && (int)threadIdx.x < nk)
    a.child_q[(size_t)b * N + sm.kids[threadIdx.x]] = -1.f;
  st.m = M;
  st.argmax = -1;
  st.s_hi = S.hi;
  st.s_lo = S.lo;
  st.first_acc = first;
  st.nrej = nrej;
  st.flags = flags;
  if (bad) st.bonus = -1;
  return st;
  }
}

// ------------------------------------------------------------------------------------------------
// the walk (by the last cluster of the sequence to finish)
// ------------------------------------------------------------------------------------------------
// Reads every node record written in this call (L2: bypass L1) and follows the accepted children;
// leaves sm.path, sm.path_len, sm.terminal and the OR of the internal nodes' flags in sm.flags.
__device__ void walk_path(const VerifyArgs& a, int b, bool leaves_done, VerifySmem& sm) {
  const int N = a.N;
  int f = 0;
  if ((int)threadIdx.x < N) {
    const int i = threadIdx.x;
    if (sm.internal[i] || leaves_done) {
      const NodeStat* src = a.stats + (size_t)b * N + i;
      NodeStat st;
      st.first_acc = __ldcg(&src->first_acc);
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
}

// Writes the outputs of sequence b (one CTA).
__device__ void write_outputs(const VerifyArgs& a, int b, int bonus, int flags, VerifySmem& sm) {
  const int N = a.N;
  if (flags & (SPEC_ST_NONFINITE | SPEC_ST_TIMEOUT)) bonus = -1;
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

// Leaves not processed (large problems): the whole cluster walks and draws the bonus at a leaf
// terminal.  bar_l_used: whether this CTA already staged a row on nb.bar_l in this launch.
template <int CL, bool SAMPLING>
__device__ void walk_sequence_cluster(const VerifyArgs& a, int b, int rank, const NodeBufs& nb,
                                      bool bar_l_used, float k2, int& xk, VerifySmem& sm) {
  walk_path(a, b, false, sm);
  const int c = sm.terminal;
  int flags = sm.flags;
  int bonus = -1;
  int writer = 0;
  if (sm.internal[c]) {
    bonus = sm.st[c].bonus;
  } else {
    const size_t row_off = ((size_t)b * a.N + c) * (size_t)a.V;
    const float* lrow = a.logits + row_off;
    const Slice s = make_slice(lrow, a.V, rank, CL);
    stage_slice(lrow, s, nb.lbuf, nb.bar_l, -INFINITY);
    // CTA-local: published below
    const int lflags = wait_slice(nb.bar_l, bar_l_used ? 1 : 0, sm.first_polls);
    if constexpr (!SAMPLING) {
      float gv;
      int gi;
      cluster_argmax<CL>(s, nb.lbuf, lflags, rank, xk, gv, gi, flags, sm);
      bonus = (gi < 0 || gi >= a.V) ? 0 : gi;
    } else {
      float M;
      DF S;
      RunState rs;
      cluster_stats<CL>(s, nb.lbuf, k2, lflags, rank, xk, M, S, rs, flags, sm);
      const float u = __ldg(a.uniforms + (size_t)b * a.N);
      if (!(flags & (SPEC_ST_NONFINITE | SPEC_ST_TIMEOUT))) {
        // a leaf's q: the current weights are e (cw = 0), p is never read
        const Draw d = cluster_draw<CL>(s, nb.lbuf, DraftSlice<false>{nb.pbuf}, rs, u, rank, sm);
        writer = d.writer;
        bonus = d.tok;
      }
    }
  }
  if (rank == writer) write_outputs(a, b, bonus, flags, sm);
}

// ------------------------------------------------------------------------------------------------
// per-sequence arrival counter
// ------------------------------------------------------------------------------------------------
// The counter word holds (call generation << 32) | (kCounterTag << 16) | arrivals.  A word whose
// upper 48 bits are not this call's (generation, tag), or whose count is not below N, is claimed
// for this call -- set to (generation, tag, 0) -- by whichever cluster of the sequence starts
// first, so no zero-filled workspace is needed: whatever a caller's buffer held before (another
// call's node records, a count left by another call, garbage) is reset.  Only a word of this very
// generation and tag with a count in [0, N) is kept, i.e. one that a cluster of this call already
// claimed or arrived at.  Every cluster claims before it can arrive, and the last arrival only
// comes after all of them started.  Arrivals are plain atomic adds; the last one resets the count,
// which keeps CUDA-graph replays (same generation) correct.
constexpr unsigned long long kCounterTag = 0x5EC7ull;

__device__ __forceinline__ unsigned long long counter_id(unsigned long long gen) {
  return ((gen & 0xFFFFFFFFull) << 16) | kCounterTag;  // bits 16..63 of the word
}

__device__ __forceinline__ bool counter_valid(unsigned long long w, unsigned long long id, int N) {
  return (w >> 16) == id && (w & 0xFFFFull) < (unsigned long long)N;
}

__device__ __forceinline__ void claim_counter(unsigned long long* ctr, unsigned long long gen,
                                              int N) {
  const unsigned long long id = counter_id(gen);
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(ctr);
  for (int it = 0; it < 8 && !counter_valid(old, id, N); ++it) {
    const unsigned long long prev = atomicCAS(ctr, old, id << 16);
    if (prev == old) break;  // claimed
    old = prev;              // changed meanwhile: claimed or arrived at by another cluster?
  }
}

// The online walk's counter word: (generation << 32) | tickets taken.  A word of another
// generation is reset to (generation, 0) by whichever cluster of the sequence starts first.
__device__ __forceinline__ void claim_tickets(unsigned long long* ctr, unsigned long long gen) {
  const unsigned long long g = gen & 0xFFFFFFFFull;
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(ctr);
  for (int it = 0; it < 8 && (old >> 32) != g; ++it) {
    const unsigned long long prev = atomicCAS(ctr, old, g << 32);
    if (prev == old) break;
    old = prev;
  }
}

// Returns true for the last of the N arrivals.  Release: this thread's earlier global writes (the
// node record) are visible to whoever sees the count; acquire: the last arriver sees every other
// cluster's record.
__device__ __forceinline__ bool arrive(unsigned long long* ctr, unsigned long long gen, int N) {
  const unsigned long long id = counter_id(gen);
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], 1;" : "=l"(old) : "l"(ctr) : "memory");
  if ((old >> 16) == id && (old & 0xFFFFull) + 1 == (unsigned long long)N) {
    atomicExch(ctr, id << 16);
    return true;
  }
  return false;
}

// ------------------------------------------------------------------------------------------------
// walk hand-over (every-node form without per-child q)
// ------------------------------------------------------------------------------------------------
// A node's outcome goes into its hand-over word as soon as the node is done, and the walk starts
// at the root and follows the accepted children as their outcomes appear, instead of waiting for
// the sequence's last node.  Word: (tag << 32) | kPublished | kWalker | kTerminal |
// flags << kFlagShift | value, with tag = handover_tag(generation) and value = accepted child + 1,
// or for a terminal (the walk stops there: no child accepted, or the node hit NaN / a timeout)
// bonus + 1 (0: no bonus).  A word with another tag is empty.  At most two parties write a word
// in a call -- the node, and the walk when it reaches the node first (kWalker) -- and whichever
// comes second continues the walk.  Everything a party needs is in the word itself, so the
// accesses are relaxed (one word's accesses are ordered by coherence alone).  The walking CTA
// reads every node's word at once and follows them in shared memory; the root's word has one
// writer (the walk starts there), so the root publishes it with a plain store.
// Epochs: each node's cluster takes one ticket from the sequence's counter word ((generation <<
// 32) | tickets, claimed like the arrival counter) at its start, so the N tickets of a call are
// [kN, kN + N) and k = ticket / N is the call's epoch, the same in every cluster however late it
// starts; a replay of a captured call (same generation) takes the next N.  Words of earlier
// calls or replays carry other tags, so nothing has to be cleared and no node arrives at the end.
constexpr uint32_t kPublished = kHandoverPublished, kWalker = 1u << 30,
                   kTerminal = kHandoverTerminal;
constexpr int kFlagShift = 22;
constexpr uint32_t kValueMask = kHandoverValueMask;  // bonus + 1 < 2^22: V < 2^22 - 1
static_assert(kValueMask == (1u << kFlagShift) - 1u, "hand-over word layout");

__device__ __forceinline__ uint32_t handover_payload(const NodeStat& st, int j, int N) {
  const int fa = st.first_acc;
  const bool terminal =
      (st.flags & (SPEC_ST_NONFINITE | SPEC_ST_TIMEOUT)) != 0 || fa <= j || fa >= N;
  const uint32_t value =
      terminal ? (uint32_t)min(max(st.bonus + 1, 0), (int)kValueMask) : (uint32_t)(fa + 1);
  return (terminal ? kTerminal : 0u) | ((uint32_t)(st.flags & 0x7F) << kFlagShift) | value;
}

// Sets `bits` in the word (an empty word becomes this generation's); returns the word before.
// `guess`: its probable current value (a cleared word is 0).  Two writers at most: a few tries.
__device__ unsigned long long handover_set(unsigned long long* w, unsigned long long gen,
                                           uint32_t bits, unsigned long long guess) {
  unsigned long long cur = guess;
  for (int it = 0; it < 16; ++it) {
    const unsigned long long base = (cur >> 32) == gen ? cur : (gen << 32);
    const unsigned long long want = base | bits;
    unsigned long long prev;
    asm volatile("atom.relaxed.gpu.global.cas.b64 %0, [%1], %2, %3;"
                 : "=l"(prev)
                 : "l"(w), "l"(cur), "l"(want)
                 : "memory");
    if (prev == cur) return cur;
    cur = prev;
  }
  return cur;
}

__device__ __forceinline__ bool handed_over(unsigned long long v, unsigned long long gen) {
  return (v >> 32) == gen && (v & (unsigned long long)kPublished);
}

// ------------------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------------------
// PGLOBAL: draft rows read from global memory instead of staged (large problems with V ~ 128K).
// Four CTAs per SM (at most 64 registers a thread): at three, the 60 clusters of 8 CTAs of one
// 60-node tree do not all fit on the GPU at once, and the last clusters start only when the
// first ones leave.
// ONLINE (every node, no per-child q): the walk follows the hand-over words as nodes finish.
template <int CL, bool PGLOBAL, bool SAMPLING, bool LEAVES, bool ONLINE = false>
__global__ void __launch_bounds__(kVThreads, 4)
    verify_kernel(const VerifyArgs a, int cap, float invT_hi, float invT_lo,
                  float k2) {
  extern __shared__ __align__(16) float dyn[];
  __shared__ VerifySmem sm;
  __shared__ __align__(8) uint64_t bars[2];
  const NodeBufs nb{dyn, dyn + cap, smem_u32(&bars[0]), smem_u32(&bars[1])};
  const int rank = (CL > 1) ? int(cg::this_cluster().block_rank()) : 0;
  const int j = blockIdx.y, b = blockIdx.z;
  const int N = a.N;
  if (threadIdx.x == 0) {
    mbar_init(nb.bar_l, 1);
    mbar_init(nb.bar_p, 1);
    mbar_init(smem_u32(&sm.xbar[0]), 1);
    mbar_init(smem_u32(&sm.xbar[1]), 1);
    mbar_fence_init();
    sm.first_polls = a.first_polls;
    sm.ticket = 0;
  }
  __syncthreads();
  cluster_arrive_release();  // exchange barriers initialised (waited for before the first exchange)
  griddep_wait();  // the inputs may be produced by the preceding kernel in the stream
  // small problems process every node: its logit row is needed whatever the tree looks like, so
  // the copy goes out before anything else
  constexpr bool do_leaves = LEAVES;  // small problems: every node, leaves included
  constexpr bool early = LEAVES;
  if (early) {
    const float* lrow = a.logits + ((size_t)b * N + j) * (size_t)a.V;
    stage_slice(lrow, make_slice(lrow, a.V, rank, CL), nb.lbuf, nb.bar_l, -INFINITY);
  }
  // the claim's round trip overlaps the tree loads (issued by the first threads) instead of
  // delaying thread 0, which issues the copies
  if (rank == 0 && threadIdx.x == kVThreads - 1) {
    if constexpr (ONLINE) {
      claim_tickets(a.counters + b, a.gen);
    } else {
      claim_counter(a.counters + b, a.gen, N);
    }
  }
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
    if (early) wait_slice(nb.bar_l, 0, kSpinLimit);  // no copy left in flight
    cluster_wait_acquire();
    return;
  }
  cluster_wait_acquire();  // every CTA of the cluster can now receive exchanges
  if constexpr (ONLINE) {
    // this node's ticket; its round trip overlaps the wait for the logit slice (rank 0's ticket
    // reaches the cluster with the first exchange)
    if (threadIdx.x == kVThreads - 1) {
      if (rank == 0) sm.ticket = (uint32_t)atomicAdd(a.counters + b, 1ull);
      // the node's hand-over word as it is now: the likely value its publish replaces
      unsigned long long w;
      asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];"
                   : "=l"(w)
                   : "l"(a.handover + (size_t)b * N + j)
                   : "memory");
      sm.hv_guess = w;
    }
  }
  int xk = 0, writer = 0;
  uint32_t ph_l = 0, ph_p = 0;
  const bool work = sm.internal[j] || do_leaves;
  NodeStat st;
  if (work)
    st = process_node<CL, PGLOBAL, SAMPLING, ONLINE>(a, b, j, rank, nb, early, DF{invT_hi, invT_lo},
                                                     k2, xk,
                                             writer,
                                   ph_l, ph_p, sm);

  // the next kernel may start launching once every CTA is past its node (see the attention kernel)
  griddep_launch_dependents();
  if constexpr (ONLINE) {
    // hand the outcome over (the root starts the walk), follow the walk while the nodes it
    // reaches are done, and write the outputs where it ends
    if (rank != writer) return;
    const unsigned long long tag = handover_tag(a.gen, sm.ticket_c / (uint32_t)N);
    unsigned long long* hw = a.handover + (size_t)b * N;
    if (threadIdx.x == 0) {
      bool walk = false;
      uint32_t lo = 0;
      if (!(st.flags & kWalkDone)) {  // a node that stopped early hands nothing over
        lo = kPublished | handover_payload(st, j, N);
        if (j == 0) {  // the walk starts here and never comes back: no one else writes this word
          const unsigned long long v = (tag << 32) | lo;
          asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(hw), "l"(v) : "memory");
          walk = true;
        } else {
          const unsigned long long prev = handover_set(hw + j, tag, lo, sm.hv_guess);
          walk = (prev >> 32) == tag && (prev & (unsigned long long)kWalker);
        }
      }
      sm.terminal = walk ? j : -1;  // where the walk continues from
      sm.hv_lo = lo;
    }
    __syncthreads();
    if (sm.terminal < 0) return;
    // every node's word in one round trip, then the walk follows them in shared memory
    for (int i = threadIdx.x; i < N; i += kVThreads) {
      unsigned long long v;
      asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(hw + i) : "memory");
      sm.hv_snap[i] = v;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int c = sm.terminal, term = -1;
      uint32_t lo = sm.hv_lo;
      for (int steps = 0; steps < N; ++steps) {
        if (lo & kTerminal) {
          term = c;
          break;
        }
        const int n = (int)(lo & kValueMask) - 1;  // an accepted child of c: c < n < N
        unsigned long long v = sm.hv_snap[n];
        if (!handed_over(v, tag)) {  // not done when read: leave the walk to it, unless it is now
          v = handover_set(hw + n, tag, kWalker, v);
          if (!handed_over(v, tag)) break;
        }
        c = n;
        lo = (uint32_t)v;
      }
      sm.terminal = term;
      if (term >= 0) {
        int len = 0;
        for (int x = term; x > 0 && len < N; x = sm.parent[x]) ++len;
        int x = term;
        for (int i = len - 1; i >= 0; --i, x = sm.parent[x]) sm.path[i] = x;
        sm.path_len = len;
        sm.found = (int)(lo & kValueMask) - 1;  // the bonus
        sm.flags = (int)((lo >> kFlagShift) & 0x7Fu);
        // the other nodes may stop at their next residual round
        const unsigned long long v = (tag << 32) | 1ull;
        asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(a.walk_done + b), "l"(v)
                     : "memory");
      }
    }
    __syncthreads();
    if (sm.terminal >= 0) write_outputs(a, b, sm.found, sm.flags, sm);
    return;
  }
  // arrival: the last cluster of the sequence to finish walks the tree
  if constexpr (do_leaves) {
    // every possible stop already has its bonus, so the writer CTA finishes alone (this
    // cluster's exchanges are complete: the other CTAs may leave)
    if (rank != writer) return;
    if (threadIdx.x == 0) {
      a.stats[(size_t)b * N + j] = st;
      sm.is_last = arrive(a.counters + b, a.gen, N) ? 1 : 0;
    }
    __syncthreads();
    if (!sm.is_last) return;
    walk_path(a, b, true, sm);
    const int c = sm.terminal;
    write_outputs(a, b, sm.st[c].bonus, sm.flags | (sm.internal[c] ? 0 : sm.st[c].flags), sm);
    return;
  }
  if (rank == writer && threadIdx.x == 0) {
    if (work) a.stats[(size_t)b * N + j] = st;
    const int last = arrive(a.counters + b, a.gen, N) ? 1 : 0;
    if constexpr (CL > 1) {
      for (int r = 0; r < CL; ++r) dsmem_store_u32(dsmem_addr(&sm.is_last, r), (uint32_t)last);
    } else {
      sm.is_last = last;
    }
  }
  cluster_barrier<CL>();
  if (!sm.is_last) return;
  walk_sequence_cluster<CL, SAMPLING>(a, b, rank, nb, work, k2, xk, sm);
  cluster_barrier<CL>();  // keep shared memory alive for remote stores
}

// Path-only form (large problems, no per-child q requested): one cluster per sequence walks the
// tree, processing only the nodes the walk reaches -- the root, then each accepted child -- with
// the same per-node step as above.  A sequence reads (accepted + 1) target rows instead of every
// internal node's, at the price of one dependent step per accepted level.  No workspace.
template <int CL, bool PGLOBAL, bool SAMPLING>
__global__ void __launch_bounds__(kVThreads, 4)
    verify_path_kernel(const VerifyArgs a, int cap, float invT_hi, float invT_lo, float k2) {
  extern __shared__ __align__(16) float dyn[];
  __shared__ VerifySmem sm;
  __shared__ __align__(8) uint64_t bars[2];
  const NodeBufs nb{dyn, dyn + cap, smem_u32(&bars[0]), smem_u32(&bars[1])};
  const int rank = (CL > 1) ? int(cg::this_cluster().block_rank()) : 0;
  const int b = blockIdx.z;
  const int N = a.N;
  if (threadIdx.x == 0) {
    mbar_init(nb.bar_l, 1);
    mbar_init(nb.bar_p, 1);
    mbar_init(smem_u32(&sm.xbar[0]), 1);
    mbar_init(smem_u32(&sm.xbar[1]), 1);
    mbar_fence_init();
    sm.first_polls = a.first_polls;
    sm.ticket = 0;
  }
  __syncthreads();
  cluster_arrive_release();  // exchange barriers initialised (waited for before the first exchange)
  griddep_wait();  // the inputs may be produced by the preceding kernel in the stream
  const int bad = load_tree(a, b, sm);  // uniform across the cluster: same tree everywhere
  if (bad) {
    if (rank == 0) {
      if (threadIdx.x == 0) {
        a.accept_len[b] = -1;
        a.bonus[b] = -1;
        if (a.status) atomicOr(a.status + b, bad);
      }
      for (int i = threadIdx.x; i < N; i += kVThreads) {
        a.acc_tokens[(size_t)b * N + i] = -1;
        if (a.acc_nodes) a.acc_nodes[(size_t)b * N + i] = -1;
      }
    }
    cluster_wait_acquire();
    return;
  }
  cluster_wait_acquire();  // every CTA of the cluster can now receive exchanges
  int xk = 0, writer = 0, c = 0, len = 0, bonus = -1, flags = 0;
  uint32_t ph_l = 0, ph_p = 0;
  for (;;) {  // at most N steps: every accepted child has a larger index than its parent
    const NodeStat st = process_node<CL, PGLOBAL, SAMPLING>(a, b, c, rank, nb, false,
                                                            DF{invT_hi, invT_lo},
                                                  k2, xk, writer, ph_l, ph_p, sm);
    flags |= st.flags;  // cluster-uniform, so the loop's control flow is too
    if (flags & (SPEC_ST_NONFINITE | SPEC_ST_TIMEOUT)) break;
    const int fa = st.first_acc;
    if (fa <= c || fa >= N) {  // every child rejected (or none): c is the terminal node
      bonus = st.bonus;  // valid in CTA `writer`
      break;
    }
    if (threadIdx.x == 0) sm.path[len] = fa;
    ++len;
    c = fa;
    // this node's shared state (children, gathers, the slices rewritten in place) is free again;
    // its generic writes are ordered before the next node's bulk copies into the same buffers
    fence_async_smem();
    __syncthreads();
  }
  griddep_launch_dependents();  // once every sequence's walk is done (see the attention kernel)
  if (threadIdx.x == 0) sm.path_len = len;
  __syncthreads();
  if (rank == writer) write_outputs(a, b, bonus, flags, sm);
  cluster_barrier<CL>();  // keep shared memory alive for remote stores
}

// Node step of the verification driven by the LM head's statistics (verify_head.cu): one cluster
// per sequence processes the node head_state[b].pending, whose full logit row a row pass of the LM
// head has just written, with the per-node step above (sibling tests in order, residual rounds,
// the bonus draw).  An accepted child becomes the walk's position (the next statistics walk
// continues from it); otherwise the sequence's outputs are written.  Sequences without a pending
// node return at once.
template <int CL>
__global__ void __launch_bounds__(kVThreads, 4)
    verify_head_step_kernel(const VerifyArgs a, int cap, float invT_hi, float invT_lo, float k2) {
  extern __shared__ __align__(16) float dyn[];
  __shared__ VerifySmem sm;
  __shared__ __align__(8) uint64_t bars[2];
  const NodeBufs nb{dyn, dyn + cap, smem_u32(&bars[0]), smem_u32(&bars[1])};
  const int rank = (CL > 1) ? int(cg::this_cluster().block_rank()) : 0;
  const int b = blockIdx.z;
  const int N = a.N;
  if (threadIdx.x == 0) {
    mbar_init(nb.bar_l, 1);
    mbar_init(nb.bar_p, 1);
    mbar_init(smem_u32(&sm.xbar[0]), 1);
    mbar_init(smem_u32(&sm.xbar[1]), 1);
    mbar_fence_init();
    sm.first_polls = a.first_polls;
    sm.ticket = 0;
  }
  __syncthreads();
  cluster_arrive_release();  // exchange barriers initialised (waited for before the first exchange)
  griddep_wait();  // the walk state and the row come from the preceding kernels
  HeadWalk* hw = a.head_state + b;
  // the same value in every CTA of the cluster (written by an earlier kernel)
  const int c = *reinterpret_cast<const volatile int*>(&hw->pending);
  const int head_flags = (a.head_flag && *reinterpret_cast<const volatile int*>(a.head_flag))
                             ? SPEC_ST_TIMEOUT
                             : 0;
  const int bad = (c >= 0 && c < N) ? load_tree(a, b, sm) : SPEC_ST_BAD_TREE;
  if (bad || head_flags) {
    // no pending node (or a row pass gave up: the sequence ends flagged, without outputs)
    if (head_flags && c >= 0 && rank == 0 && threadIdx.x == 0) {
      a.accept_len[b] = -1;
      a.bonus[b] = -1;
      if (a.status) atomicOr(a.status + b, head_flags);
      hw->pending = -1;
      hw->done = 1;
      a.head_walk.row_dst[b] = -1;
    }
    if (head_flags && c >= 0 && rank == 0)
      for (int i = threadIdx.x; i < N; i += kVThreads) {
        a.acc_tokens[(size_t)b * N + i] = -1;
        if (a.acc_nodes) a.acc_nodes[(size_t)b * N + i] = -1;
      }
    griddep_launch_dependents();
    cluster_wait_acquire();
    return;
  }
  cluster_wait_acquire();  // every CTA of the cluster can now receive exchanges
  int xk = 0, writer = 0;
  uint32_t ph_l = 0, ph_p = 0;
  const NodeStat st = process_node<CL, false, true, false, true>(
      a, b, c, rank, nb, false, DF{invT_hi, invT_lo}, k2, xk, writer, ph_l, ph_p, sm);
  griddep_launch_dependents();
  const int flags = st.flags;  // cluster-uniform, as first_acc
  const int fa = st.first_acc;
  const bool next = !(flags & (SPEC_ST_NONFINITE | SPEC_ST_TIMEOUT)) && fa > c && fa < N;
  if (next) {
    // the walk moves to fa and goes on from there on the statistics, marking the next pass's row
    // (the last pass has none: the depth bound leaves no sequence open after it)
    if (rank == 0) {
      if (threadIdx.x < 32) {  // warp 0
        if (threadIdx.x == 0) {
          const int len = hw->len;
          if (len < kMaxNodes) hw->path[len] = fa;
          hw->len = len + 1;
          hw->cur = fa;
          hw->pending = -1;
        }
        __syncwarp();
        int wflags = 0, pend = -1;
        if (a.head_walk.active)
          pend = head_stats_walk(a.head_walk, a.probs, a.tokens, a.uniforms, b, N, a.V, fa, hw,
                                 wflags);
        if (threadIdx.x == 0) {
          if (wflags) {
            a.accept_len[b] = -1;
            a.bonus[b] = -1;
            if (a.status) atomicOr(a.status + b, wflags);
            hw->done = 1;
          }
          if (pend < 0) a.head_walk.row_dst[b] = -1;
          sm.found = wflags ? -2 : pend;
        }
      }
      __syncthreads();
      const int pend = sm.found;
      if (pend == -2) {
        for (int i = threadIdx.x; i < N; i += kVThreads) {
          a.acc_tokens[(size_t)b * N + i] = -1;
          if (a.acc_nodes) a.acc_nodes[(size_t)b * N + i] = -1;
        }
      } else if (pend >= 0) {
        head_copy_hidden(a.head_walk, b, N, pend, threadIdx.x, kVThreads);
      }
    }
  } else if (rank == writer) {  // c is the terminal node: the bonus is valid in this CTA
    const int len = min(hw->len, kMaxNodes);
    for (int i = threadIdx.x; i < len; i += kVThreads) sm.path[i] = hw->path[i];
    if (threadIdx.x == 0) sm.path_len = len;
    __syncthreads();
    write_outputs(a, b, st.bonus, flags, sm);
    if (threadIdx.x == 0) {
      hw->pending = -1;
      hw->done = 1;
      a.head_walk.row_dst[b] = -1;
    }
  }
  cluster_barrier<CL>();  // keep shared memory alive for remote stores
}

// ------------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------------
size_t verify_workspace_bytes(int B, int N, int V) {
  (void)V;
  // node records [B, N], arrival counters [B], hand-over words [B, N], walk-done words [B]
  return (size_t)B * N * (sizeof(NodeStat) + sizeof(unsigned long long)) +
         (size_t)B * 2 * sizeof(unsigned long long);
}

template <class... Params, class... Args>
static cudaError_t launch_ex(void (*kern)(Params...), dim3 grid, int cl, size_t smem,
                             cudaStream_t s, Args... args) {
  // the exchange arrays (VerifySmem::cpart, ccur) and the 8-lane combines hold kMaxCluster ranks
  if (cl < 1 || cl > kMaxCluster) return cudaErrorInvalidConfiguration;
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

// Per-buffer slice limit (floats): two buffers plus the static state fit in a CTA's 227 KB.
constexpr int kMaxSliceFloats = 26 * 1024;

// Cluster size: large enough that the slice buffers fit; for latency-bound (small) problems as
// large as slices of >= 1024 elements allow; otherwise aim for about one wave of CTAs, then grow
// (up to 8) until a CTA's buffers take at most ~72 KB, so that three CTAs share an SM: each node
// is a chain of dependent steps, and one CTA per SM leaves the SM idle between them.
constexpr size_t kLargeCtaBytes = 72 * 1024;

static int pick_cluster(long long units, int V, int num_sms, bool small, int nbuf) {
  int cl = 1;
  while (cl < 8 && slice_capacity(V, cl) > kMaxSliceFloats) cl *= 2;
  if (small) {
    // T = 0 (one buffer: an argmax pass and one exchange per node) measured faster with clusters
    // of 4 (6.3 against 6.7 us for the 60-node tree at V = 32000); T > 0, with its residual rounds,
    // with clusters of 8 (12.0 against 12.3 us)
    const int cap = nbuf > 1 ? 8 : 4;
    while (cl < cap && V / (cl * 2) >= 1024) cl *= 2;
    return cl;
  }
  while (cl < 8 && units * (cl * 2) <= (long long)num_sms * 3 / 2 && V / (cl * 2) >= 2048) cl *= 2;
  while (cl < kMaxCluster && (size_t)nbuf * slice_capacity(V, cl) * sizeof(float) > kLargeCtaBytes)
    cl *= 2;
  return cl;
}

// One instantiation per form (all nodes with or without the leaves, the path only), temperature
// kind (sampling or greedy) and draft-row staging, so that each kernel holds one code path.
template <int CL>
static cudaError_t launch_cl(const VerifyArgs& a, dim3 g, size_t smem, cudaStream_t s, int cap,
                             int leaves, float invT_hi, float invT_lo, float k2, bool path) {
  const bool sampling = a.T > 0.f;  // p_global is only ever set when sampling
  if (path) {
    if (!sampling)
      return launch_ex(verify_path_kernel<CL, false, false>, g, CL, smem, s, a, cap, invT_hi,
                       invT_lo, k2);
    if (a.p_global)
      return launch_ex(verify_path_kernel<CL, true, true>, g, CL, smem, s, a, cap, invT_hi,
                       invT_lo, k2);
    return launch_ex(verify_path_kernel<CL, false, true>, g, CL, smem, s, a, cap, invT_hi,
                     invT_lo, k2);
  }
  if (leaves) {
    // without per-child q the walk follows the nodes as they finish (bonus + 1 fits the word)
    if (a.child_q == nullptr && (unsigned)a.V < kValueMask) {
      if (!sampling)
        return launch_ex(verify_kernel<CL, false, false, true, true>, g, CL, smem, s, a, cap,
                         invT_hi, invT_lo, k2);
      return launch_ex(verify_kernel<CL, false, true, true, true>, g, CL, smem, s, a, cap,
                       invT_hi, invT_lo, k2);
    }
    if (!sampling)
      return launch_ex(verify_kernel<CL, false, false, true>, g, CL, smem, s, a, cap, invT_hi,
                       invT_lo, k2);
    return launch_ex(verify_kernel<CL, false, true, true>, g, CL, smem, s, a, cap, invT_hi,
                     invT_lo, k2);
  }
  if (!sampling)
    return launch_ex(verify_kernel<CL, false, false, false>, g, CL, smem, s, a, cap, invT_hi,
                     invT_lo, k2);
  if (a.p_global)
    return launch_ex(verify_kernel<CL, true, true, false>, g, CL, smem, s, a, cap, invT_hi,
                     invT_lo, k2);
  return launch_ex(verify_kernel<CL, false, true, false>, g, CL, smem, s, a, cap, invT_hi,
                   invT_lo, k2);
}

// Path-only form: one cluster per sequence, each step a chain of dependent passes over the
// slices, so clusters grow (up to 8) while about four CTAs per SM cover the batch.
static int pick_cluster_path(int B, int V, int num_sms) {
  int cl = 1;
  while (cl < 8 && slice_capacity(V, cl) > kMaxSliceFloats) cl *= 2;
  while (cl < 8 && (long long)B * cl * 2 <= (long long)num_sms * 4 && V / (cl * 2) >= 1024)
    cl *= 2;
  return cl;
}

bool verify_supported(int V) { return slice_capacity(V, 8) <= kMaxSliceFloats; }

cudaError_t launch_verify_head_step(const VerifyArgs& a, int num_sms, cudaStream_t s) {
  if (!(a.T > 0.f) || !a.head_rows || !a.head_state) return cudaErrorInvalidValue;
  const int cl = pick_cluster_path(a.B, a.V, num_sms);
  const int cap = slice_capacity(a.V, cl);
  // both rows staged: two slices of at most kMaxSliceFloats fit in shared memory
  const size_t smem = 2 * (size_t)cap * sizeof(float);
  const double invTd = 1.0 / (double)a.T;
  const float invT_hi = (float)invTd, invT_lo = (float)(invTd - (double)invT_hi);
  const float k2 = (float)(invTd * 1.4426950408889634);  // log2(e) / T
  const dim3 g(cl, 1, a.B);
  switch (cl) {
    case 1: return launch_ex(verify_head_step_kernel<1>, g, 1, smem, s, a, cap, invT_hi, invT_lo, k2);
    case 2: return launch_ex(verify_head_step_kernel<2>, g, 2, smem, s, a, cap, invT_hi, invT_lo, k2);
    case 4: return launch_ex(verify_head_step_kernel<4>, g, 4, smem, s, a, cap, invT_hi, invT_lo, k2);
    default:
      return launch_ex(verify_head_step_kernel<8>, g, 8, smem, s, a, cap, invT_hi, invT_lo, k2);
  }
}

cudaError_t launch_verify(const VerifyArgs& a, int num_sms, cudaStream_t s) {
  const bool small = (long long)a.B * a.N * a.V * 4 <= (64ll << 20);
  // small problems are latency-bound: process leaves speculatively too
  const int leaves = small ? 1 : 0;
  // large problems walk the accepted path only, unless every child's q is wanted
  const bool path = !small && a.child_q == nullptr;
  const long long units = (long long)a.B * (leaves ? a.N : (a.N + 1) / 2);
  const int cl = path ? pick_cluster_path(a.B, a.V, num_sms)
                      : pick_cluster(units, a.V, num_sms, small, a.T > 0.f ? 2 : 1);
  const int cap = slice_capacity(a.V, cl);
  // large problems whose two slices would still leave one CTA per SM read the draft row from
  // global memory (L2) instead of staging it (the path form stages it when its clusters leave
  // SMs to spare)
  VerifyArgs ak = a;
  const bool crowded = !path || (long long)a.B * cl > num_sms;
  ak.p_global = (!small && a.T > 0.f && crowded &&
                 2 * (size_t)cap * sizeof(float) > kLargeCtaBytes) ? 1 : 0;
  const size_t smem = (size_t)(a.T > 0.f && !ak.p_global ? 2 : 1) * cap * sizeof(float);
  const double invTd = a.T > 0.f ? 1.0 / (double)a.T : 0.0;
  const float invT_hi = (float)invTd, invT_lo = (float)(invTd - (double)invT_hi);
  const float k2 = (float)(invTd * 1.4426950408889634);  // log2(e) / T
  const dim3 g(cl, path ? 1 : a.N, a.B);
  switch (cl) {
    case 1: return launch_cl<1>(ak, g, smem, s, cap, leaves, invT_hi, invT_lo, k2, path);
    case 2: return launch_cl<2>(ak, g, smem, s, cap, leaves, invT_hi, invT_lo, k2, path);
    case 4: return launch_cl<4>(ak, g, smem, s, cap, leaves, invT_hi, invT_lo, k2, path);
    default: return launch_cl<8>(ak, g, smem, s, cap, leaves, invT_hi, invT_lo, k2, path);
  }
}

}  // namespace spectree
