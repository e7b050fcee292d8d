// Dynamic (EAGLE-2-style) draft-tree construction on the device (sm_103a).
//
// Method: EAGLE-3 explainer, 背景と動機 and EAGLE-2との統合 -- EAGLE-2 builds the draft tree at
// inference time from the draft head's outputs instead of using a fixed shape.  The pages give no
// procedure; this follows EAGLE-2's expand-then-rerank construction:
//   * a drafted node's value is the sum of the draft log-probabilities log softmax(l)[token] along
//     its path from the root (root value 0);
//   * level d expands the frontier (the root at d = 1): frontier slot i's K highest draft logits
//     (ties: lower token id) become candidates with candidate order i K + r, all joining the pool;
//     the K candidates of the level with the highest values (ties: lower order) form the next
//     frontier, best first;
//   * the tree is the root plus the N - 1 best candidates of the pool (ties: shallower, then lower
//     order), numbered by (depth, order), so parents precede children.
//
// State (the caller's workspace, per sequence): a 128-byte header (levels done, pool size, arrival
// counter, status bits, frontier) and the pool, one 16-byte entry per drafted node.
//
// expand_kernel: one CTA per draft row of the level.  A pass over the row (32 elements per thread
// in flight) finds each warp's best entry; L, the K-th best of those, bounds the row's K best from
// below.  A second pass (L2) sums exp(x - m) with a compensated sum for the log-sum-exp and
// collects the few entries >= L, which are ranked exactly.  The CTA appends its K candidates to
// the pool; the last CTA of the sequence to arrive (counter + fences, no waiting) ranks the
// level's candidates and writes the frontier.  finalize_kernel: one CTA per sequence sorts the
// pool (bitonic, by value then pool index) and writes the tree.
#include "common.cuh"
#include "internal.h"

namespace spectree {

namespace {

constexpr int kBThreads = 512;
constexpr int kFinThreads = 512;
constexpr int kChunk = 32;  // row elements per thread in flight

typedef unsigned long long u64;

struct BuildHeader {
  int32_t level;    // levels expanded so far
  int32_t count;    // pool entries
  int32_t arrived;  // CTAs of the level being expanded that are done
  int32_t flags;    // status bits seen so far
  int32_t frontier[kMaxTreeK];
  int32_t pad[32 - 4 - kMaxTreeK];
};
static_assert(sizeof(BuildHeader) == 128, "header layout");

struct PoolEntry {
  int32_t token, parent;
  float value;
  uint32_t meta;  // depth << 24 | (row + 1) << 12 | order; row + 1 = 0: not expanded
};
static_assert(sizeof(PoolEntry) == 16, "pool entry layout");

__device__ __forceinline__ uint32_t meta_of(int depth, int row1, int order) {
  return (uint32_t(depth) << 24) | (uint32_t(row1) << 12) | uint32_t(order);
}

__device__ __forceinline__ uint32_t order_key(float x) {  // larger float <-> larger key
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;  // -0 and +0 are equal logits: one key
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k) {  // inverse of order_key (-0 -> +0)
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// An element's key: a larger key is a larger value, then a lower token id; every key is > 0.
__device__ __forceinline__ unsigned long long elem_key(float x, int y) {
  return ((unsigned long long)order_key(x) << 32) | (0xffffffffu - (uint32_t)y);
}

// (x, y) ranks before (v, z): larger value, then lower index
__device__ __forceinline__ bool before(float x, int y, float v, int z) {
  return x > v || (x == v && y < z);
}

constexpr int kCandCap = 2048;  // keys at or above the threshold a CTA collects

struct ExpandSmem {
  unsigned long long wkey[kBThreads / 32];  // each warp's best key
  unsigned long long ckey[kCandCap];        // the keys >= L
  unsigned long long mkey, lkey;
  int nc;
  float wv[kBThreads / 32];
  int wi[kBThreads / 32], wt[kBThreads / 32];
  float best_v[kMaxTreeK];
  int best_i[kMaxTreeK];
  int win_t;
  float wsum_hi[kBThreads / 32], wsum_lo[kBThreads / 32];
  int last;
  // the last CTA: the level's candidates
  float cv[kMaxTreeK * kMaxTreeK];
  int rank[kMaxTreeK * kMaxTreeK];
};

__device__ __forceinline__ uint32_t cluster_atom_add_u32(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.relaxed.cluster.shared::cluster.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(addr), "r"(v)
               : "memory");
  return old;
}

// Exact top K of a whole row by per-thread insertion lists (lv / li, K x 512) and K rounds of a
// CTA-wide argmax; for rows whose threshold admits more than kCandCap keys.  Every thread calls it.
__device__ void slow_topk(ExpandSmem& sm, float* lv, int* li, const float* row, int V, int K) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  for (int k = 0; k < K; ++k) {
    lv[k * kBThreads + tid] = -INFINITY;
    li[k * kBThreads + tid] = 0x7fffffff;
  }
  for (int y = tid; y < V; y += kBThreads) {
    const float x = __ldg(row + y);
    if (!before(x, y, lv[(K - 1) * kBThreads + tid], li[(K - 1) * kBThreads + tid])) continue;
    int p = K - 1;  // shift the worse entries down, insert
    while (p > 0 && before(x, y, lv[(p - 1) * kBThreads + tid], li[(p - 1) * kBThreads + tid])) {
      lv[p * kBThreads + tid] = lv[(p - 1) * kBThreads + tid];
      li[p * kBThreads + tid] = li[(p - 1) * kBThreads + tid];
      --p;
    }
    lv[p * kBThreads + tid] = x;
    li[p * kBThreads + tid] = y;
  }
  int head = 0;
  for (int k = 0; k < K; ++k) {
    float v = head < K ? lv[head * kBThreads + tid] : -INFINITY;
    int y = head < K ? li[head * kBThreads + tid] : 0x7fffffff;
    int t = tid;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
      const int y2 = __shfl_xor_sync(0xffffffffu, y, o);
      const int t2 = __shfl_xor_sync(0xffffffffu, t, o);
      if (before(v2, y2, v, y)) {
        v = v2;
        y = y2;
        t = t2;
      }
    }
    if (lane == 0) {
      sm.wv[w] = v;
      sm.wi[w] = y;
      sm.wt[w] = t;
    }
    __syncthreads();
    if (tid == 0) {
      float bv = sm.wv[0];
      int bi = sm.wi[0], bt = sm.wt[0];
      for (int q = 1; q < kBThreads / 32; ++q)
        if (before(sm.wv[q], sm.wi[q], bv, bi)) {
          bv = sm.wv[q];
          bi = sm.wi[q];
          bt = sm.wt[q];
        }
      sm.best_v[k] = bv;
      sm.best_i[k] = bi;
      sm.win_t = bt;
    }
    __syncthreads();
    if (tid == sm.win_t) ++head;
  }
}

// Ranks the collected keys (sm.ckey[0 .. nc)) into sm.best_v / sm.best_i (every thread calls it).
__device__ void rank_candidates(ExpandSmem& sm, int nc, int K) {
  for (int c = threadIdx.x; c < nc; c += kBThreads) {
    const u64 kc = sm.ckey[c];
    int r = 0;
    for (int o = 0; o < nc; ++o) r += sm.ckey[o] > kc ? 1 : 0;
    if (r < K) {
      sm.best_v[r] = key_float((uint32_t)(kc >> 32));
      sm.best_i[r] = (int)(0xffffffffu - (uint32_t)kc);
    }
  }
}

// The end of a row's expansion (every thread of the CTA): the row's K candidates into the pool,
// the arrival, and for the last row of the sequence to arrive, the level's ranking and frontier.
__device__ void finish_row(ExpandSmem& sm, BuildHeader* hdr, PoolEntry* pool, int b, int i, int R,
                           int K, int level, int count, int f, float vf, float lse, bool bad,
                           int32_t* ftok, int32_t* fslot, int32_t* status) {
  const int tid = threadIdx.x;
  // ---- this row's candidates into the pool
  if (!bad && tid < K) {
    const float lp = fminf(__fsub_rn(sm.best_v[tid], lse), 0.f);  // a log-probability is <= 0
    PoolEntry e;
    e.token = sm.best_i[tid];
    e.parent = f;
    e.value = __fadd_rn(vf, lp);
    e.meta = meta_of(level, 0, i * K + tid);
    pool[count + i * K + tid] = e;
  }
  if (tid == 0) {
    const int row_idx = level == 1 ? 0 : 1 + (level - 2) * K + i;
    if (level == 1) {
      PoolEntry r;
      r.token = -1;
      r.parent = -1;
      r.value = 0.f;
      r.meta = meta_of(0, 1, 0);
      pool[0] = r;
    } else {
      pool[f].meta = __ldcg(&pool[f].meta) | (uint32_t(row_idx + 1) << 12);
    }
  }
  __threadfence();  // this CTA's pool writes before its arrival
  __syncthreads();
  if (tid == 0) sm.last = (atomicAdd(&hdr->arrived, 1) == R - 1);
  __syncthreads();
  if (!sm.last) return;
  // ---- the last CTA of the sequence: rank the level's candidates, write the frontier
  __threadfence();
  const int nc = R * K;
  const bool failed = (__ldcg(&hdr->flags) & SPEC_ST_NONFINITE) != 0;
  if (!failed) {
    for (int c = tid; c < nc; c += kBThreads) sm.cv[c] = __ldcg(&pool[count + c].value);
    __syncthreads();
    for (int c = tid; c < nc; c += kBThreads) {
      const float v = sm.cv[c];
      int r = 0;
      for (int o = 0; o < nc; ++o) r += before(sm.cv[o], o, v, c) ? 1 : 0;
      sm.rank[c] = r;
    }
    __syncthreads();
    for (int c = tid; c < nc; c += kBThreads) {
      const int r = sm.rank[c];
      if (r < K) {
        hdr->frontier[r] = count + c;
        if (ftok) ftok[(size_t)b * K + r] = __ldcg(&pool[count + c].token);
        if (fslot) fslot[(size_t)b * K + r] = c / K;
      }
    }
  } else if (status && tid == 0) {
    atomicOr(status + b, SPEC_ST_NONFINITE);
  }
  __syncthreads();
  if (tid == 0) {
    hdr->count = count + (failed ? 0 : nc);
    hdr->level = level;
    hdr->arrived = 0;
  }
}

__global__ void __launch_bounds__(kBThreads) expand_rows_kernel(const float* __restrict__ logits, int R,
                                                           int V, int K, int level,
                                                           uint8_t* __restrict__ state,
                                                           size_t stride, int32_t* ftok,
                                                           int32_t* fslot, int32_t* status) {
  __shared__ ExpandSmem sm;
  // each thread's best K entries, best first: value lv[k * 512 + t], token id li[k * 512 + t]
  extern __shared__ float4 lists_raw[];
  float* lv = reinterpret_cast<float*>(lists_raw);
  int* li = reinterpret_cast<int*>(lv + K * kBThreads);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int b = blockIdx.x / R, i = blockIdx.x % R;
  BuildHeader* hdr = reinterpret_cast<BuildHeader*>(state + (size_t)b * stride);
  PoolEntry* pool = reinterpret_cast<PoolEntry*>(state + (size_t)b * stride + sizeof(BuildHeader));
  griddep_wait();  // the rows and the state come from preceding work in the stream
  griddep_launch_dependents();

  // the sequence before this level
  int count = 1, f = 0;
  float vf = 0.f;
  if (level > 1) {
    const int lv = __ldcg(&hdr->level), fl = __ldcg(&hdr->flags);
    if (fl & SPEC_ST_NONFINITE) return;  // the construction stopped at an earlier level
    if (lv != level - 1) {               // out of order: the state stays as it is
      if (tid == 0 && i == 0 && status) atomicOr(status + b, SPEC_ST_BAD_TREE);
      return;  // every CTA of the sequence reads the same header and leaves
    }
    count = __ldcg(&hdr->count);
    f = __ldcg(&hdr->frontier[i]);
    vf = __ldcg(&pool[f].value);
  }
  const float* row = logits + ((size_t)b * R + i) * (size_t)V;

  if (tid == 0) {
    if (level == 1) {  // a new construction (one CTA per sequence at level 1)
      hdr->flags = 0;
      hdr->arrived = 0;
    }
    sm.lkey = 0ull;  // below every element's key: all elements, if fewer than K threads hold one
    sm.nc = 0;
  }
  // rows 16-byte aligned (V % 4 == 0): float4 loads; thread t's chunk elements are
  // base + 4 (t + 512 j) + e (vector) or base + t + 512 j (scalar)
  const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  auto elem = [&](int base, int j) -> int {  // the row index of element j of a chunk
    return vec ? base + 4 * (tid + kBThreads * (j >> 2)) + (j & 3) : base + tid + kBThreads * j;
  };
  auto load_chunk = [&](int base, float (&v)[kChunk]) {
    if (vec) {
#pragma unroll
      for (int j = 0; j < kChunk / 4; ++j) {
        const int y = base + 4 * (tid + kBThreads * j);
        float4 q = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (y < V) q = __ldg(reinterpret_cast<const float4*>(row + y));
        v[4 * j] = q.x;
        v[4 * j + 1] = q.y;
        v[4 * j + 2] = q.z;
        v[4 * j + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < kChunk; ++j) {
        const int y = base + tid + kBThreads * j;
        v[j] = y < V ? __ldg(row + y) : -INFINITY;
      }
    }
  };
  // ---- pass 1: each warp's best key (larger value, then lower token id); NaN / +Inf check
  bool bad = false;
  u64 best = 0ull;
  for (int base = 0; base < V; base += kBThreads * kChunk) {
    float v[kChunk];
    load_chunk(base, v);
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      const int y = elem(base, j);
      if (y >= V) continue;
      if (isnan(v[j]) || v[j] == INFINITY) bad = true;
      else best = max(best, elem_key(v[j], y));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
  if (lane == 0) sm.wkey[w] = best;  // the warp's best key
  if (__syncthreads_or(bad)) {
    if (tid == 0) atomicOr(&hdr->flags, SPEC_ST_NONFINITE);
    bad = true;
  }
  // ---- the row max and L, the K-th best of the warps' bests (K <= 16 warps): at least K
  // elements are >= L, so the K best elements all are
  if (!bad && tid < kBThreads / 32 && sm.wkey[tid] != 0ull) {
    const u64 mine = sm.wkey[tid];
    int r = 0;
    for (int t = 0; t < kBThreads / 32; ++t) r += sm.wkey[t] > mine ? 1 : 0;
    if (r == 0) sm.mkey = mine;
    if (r == K - 1) sm.lkey = mine;
  }
  __syncthreads();
  // ---- pass 2 (L2): log-sum-exp (compensated sum of exp(x - m)), and the keys >= L
  float lse = 0.f;
  if (!bad) {
    const float m = key_float((uint32_t)(sm.mkey >> 32));
    const u64 L = sm.lkey;
    CompSum acc;
    for (int base = 0; base < V; base += kBThreads * kChunk) {
      float v[kChunk];
      load_chunk(base, v);
#pragma unroll
      for (int j = 0; j < kChunk; ++j) {
        const int y = elem(base, j);
        if (y >= V) continue;
        acc.add(__expf(__fsub_rn(v[j], m)));
        const u64 k = elem_key(v[j], y);
        if (k >= L) {
          const int slot = atomicAdd(&sm.nc, 1);
          if (slot < kCandCap) sm.ckey[slot] = k;
        }
      }
    }
    float hi = acc.hi, lo = acc.lo;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {  // warp sum of the (hi, lo) pairs in two-float arithmetic
      const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
      const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
      const DF s = df_two_sum(hi, h2);
      hi = s.hi;
      lo = __fadd_rn(__fadd_rn(lo, l2), s.lo);
    }
    if (lane == 0) {
      sm.wsum_hi[w] = hi;
      sm.wsum_lo[w] = lo;
    }
    __syncthreads();
    float sh = sm.wsum_hi[0], sl = sm.wsum_lo[0];
    for (int q = 1; q < kBThreads / 32; ++q) {
      const DF s = df_two_sum(sh, sm.wsum_hi[q]);
      sh = s.hi;
      sl = __fadd_rn(__fadd_rn(sl, sm.wsum_lo[q]), s.lo);
    }
    // log(S) for S = sh + sl (sh >= 1: the max contributes exp(0))
    lse = __fadd_rn(m, __fadd_rn(logf(sh), __fdiv_rn(sl, sh)));
    // ---- the K best: rank the candidates (or, if too many reach L, the slow exact way)
    const int nc = sm.nc;
    if (nc <= kCandCap) rank_candidates(sm, nc, K);
    else slow_topk(sm, lv, li, row, V, K);
  }
  __syncthreads();
  finish_row(sm, hdr, pool, b, i, R, K, level, count, f, vf, lse, bad, ftok, fslot, status);
}

// Cluster form: the CL CTAs of a row each hold E elements per thread in registers (thread t of rank
// r: elements r * 512 E + t + 512 j), so the row is read once and the log-sum-exp pass reads
// registers.  Two DSMEM exchanges: every CTA's warp-best keys and non-finite flag to every CTA
// (each derives the max and L), then every CTA's exp-sum and keys >= L to rank 0, which finishes
// the row.
template <int CL, int E>
__global__ void __launch_bounds__(kBThreads) expand_cluster_kernel(
    const float* __restrict__ logits, int R, int V, int K, int level, uint8_t* __restrict__ state,
    size_t stride, int32_t* ftok, int32_t* fslot, int32_t* status) {
  __shared__ ExpandSmem sm;
  __shared__ unsigned long long xkey[CL][kBThreads / 32];  // every CTA's warp-best keys
  __shared__ int xbad[CL];
  __shared__ float xs_hi[CL], xs_lo[CL];  // every CTA's exp-sum (rank 0)
  extern __shared__ float4 lists_raw[];   // slow_topk's lists (rank 0)
  float* lv = reinterpret_cast<float*>(lists_raw);
  int* li = reinterpret_cast<int*>(lv + K * kBThreads);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int rank = CL > 1 ? int(blockIdx.x % CL) : 0;
  const int rowid = blockIdx.x / CL, b = rowid / R, i = rowid % R;
  BuildHeader* hdr = reinterpret_cast<BuildHeader*>(state + (size_t)b * stride);
  PoolEntry* pool = reinterpret_cast<PoolEntry*>(state + (size_t)b * stride + sizeof(BuildHeader));
  griddep_wait();  // the rows and the state come from preceding work in the stream
  griddep_launch_dependents();
  int count = 1, f = 0;
  float vf = 0.f;
  if (level > 1) {  // the same header for every CTA of the cluster: they leave together
    const int lv0 = __ldcg(&hdr->level), fl = __ldcg(&hdr->flags);
    if (fl & SPEC_ST_NONFINITE) return;
    if (lv0 != level - 1) {
      if (tid == 0 && i == 0 && rank == 0 && status) atomicOr(status + b, SPEC_ST_BAD_TREE);
      return;
    }
    count = __ldcg(&hdr->count);
    f = __ldcg(&hdr->frontier[i]);
    vf = __ldcg(&pool[f].value);
  }
  if (tid == 0) {
    if (level == 1 && rank == 0) {
      hdr->flags = 0;
      hdr->arrived = 0;
    }
    sm.nc = 0;
    sm.lkey = 0ull;
  }
  if constexpr (CL > 1) cluster_arrive_release();  // this CTA has started and zeroed its counter
  const float* row = logits + ((size_t)b * R + i) * (size_t)V;
  const int y0 = rank * kBThreads * E + tid;
  float x[E];
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const int y = y0 + j * kBThreads;
    x[j] = y < V ? __ldg(row + y) : -INFINITY;
  }
  bool bad = false;
  u64 best = 0ull;
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const int y = y0 + j * kBThreads;
    if (y >= V) continue;
    if (isnan(x[j]) || x[j] == INFINITY) bad = true;
    else best = max(best, elem_key(x[j], y));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
  bad = __syncthreads_or(bad);
  // ---- exchange 1: warp-best keys and the non-finite flag to every CTA
  if constexpr (CL > 1) {
    cluster_wait_acquire();  // every CTA has started: its shared memory may be written
    if (lane == 0)
      for (int r = 0; r < CL; ++r)
        dsmem_store_v2(dsmem_addr(&xkey[rank][w], r), (uint32_t)best, (uint32_t)(best >> 32));
    if (tid == 0)
      for (int r = 0; r < CL; ++r) dsmem_store_u32(dsmem_addr(&xbad[rank], r), bad ? 1u : 0u);
    cluster_arrive_release();
    cluster_wait_acquire();
  } else {
    if (lane == 0) xkey[0][w] = best;
    if (tid == 0) xbad[0] = bad;
    __syncthreads();
  }
  bool anybad = false;
  for (int r = 0; r < CL; ++r) anybad |= xbad[r] != 0;
  if (anybad) {
    if (rank != 0) return;
    if (tid == 0) atomicOr(&hdr->flags, SPEC_ST_NONFINITE);
    finish_row(sm, hdr, pool, b, i, R, K, level, count, f, vf, 0.f, true, ftok, fslot, status);
    return;
  }
  // ---- the row max and L, the K-th best of the CL x 16 warp-best keys (>= K elements reach it)
  constexpr int NX = CL * (kBThreads / 32);
  if (tid < NX) {
    const u64 mine = xkey[tid / (kBThreads / 32)][tid % (kBThreads / 32)];
    if (mine != 0ull) {
      int r = 0;
      for (int t = 0; t < NX; ++t) r += xkey[t / (kBThreads / 32)][t % (kBThreads / 32)] > mine;
      if (r == 0) sm.mkey = mine;
      if (r == K - 1) sm.lkey = mine;
    }
  }
  __syncthreads();
  const float m = key_float((uint32_t)(sm.mkey >> 32));
  const u64 L = sm.lkey;
  // ---- this CTA's exp-sum and keys >= L, to rank 0
  CompSum acc;
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const int y = y0 + j * kBThreads;
    if (y >= V) continue;
    acc.add(__expf(__fsub_rn(x[j], m)));
    const u64 k = elem_key(x[j], y);
    if (k >= L) {
      if constexpr (CL > 1) {
        const uint32_t slot = cluster_atom_add_u32(dsmem_addr(&sm.nc, 0), 1u);
        if (slot < (uint32_t)kCandCap)
          dsmem_store_v2(dsmem_addr(&sm.ckey[slot], 0), (uint32_t)k, (uint32_t)(k >> 32));
      } else {
        const int slot = atomicAdd(&sm.nc, 1);
        if (slot < kCandCap) sm.ckey[slot] = k;
      }
    }
  }
  float hi = acc.hi, lo = acc.lo;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {  // warp sum of the (hi, lo) pairs in two-float arithmetic
    const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
    const DF d = df_two_sum(hi, h2);
    hi = d.hi;
    lo = __fadd_rn(__fadd_rn(lo, l2), d.lo);
  }
  if (lane == 0) {
    sm.wsum_hi[w] = hi;
    sm.wsum_lo[w] = lo;
  }
  __syncthreads();
  if (tid == 0) {
    float sh = sm.wsum_hi[0], sl = sm.wsum_lo[0];
    for (int q = 1; q < kBThreads / 32; ++q) {
      const DF d = df_two_sum(sh, sm.wsum_hi[q]);
      sh = d.hi;
      sl = __fadd_rn(__fadd_rn(sl, sm.wsum_lo[q]), d.lo);
    }
    if constexpr (CL > 1) {
      dsmem_store_u32(dsmem_addr(&xs_hi[rank], 0), __float_as_uint(sh));
      dsmem_store_u32(dsmem_addr(&xs_lo[rank], 0), __float_as_uint(sl));
    } else {
      xs_hi[0] = sh;
      xs_lo[0] = sl;
    }
  }
  if constexpr (CL > 1) {
    cluster_arrive_release();
    cluster_wait_acquire();
    if (rank != 0) return;  // nothing reads another CTA's shared memory after this point
  } else {
    __syncthreads();
  }
  // ---- rank 0: the log-sum-exp, the K best, the row's end
  float sh = xs_hi[0], sl = xs_lo[0];
  for (int r = 1; r < CL; ++r) {
    const DF d = df_two_sum(sh, xs_hi[r]);
    sh = d.hi;
    sl = __fadd_rn(__fadd_rn(sl, xs_lo[r]), d.lo);
  }
  const float lse = __fadd_rn(m, __fadd_rn(logf(sh), __fdiv_rn(sl, sh)));
  const int nc = sm.nc;
  if (nc <= kCandCap) rank_candidates(sm, nc, K);
  else slow_topk(sm, lv, li, row, V, K);
  __syncthreads();
  finish_row(sm, hdr, pool, b, i, R, K, level, count, f, vf, lse, false, ftok, fslot, status);
}

template <int CL, int E>
cudaError_t launch_expand_cluster(const float* logits, int B, int R, int V, int K, int D, int level,
                                  void* state, int32_t* ftok, int32_t* fslot, int32_t* status,
                                  cudaStream_t s) {
  static_assert(CL >= 1 && CL <= 8, "clusters stay within the portable size");
  const size_t lists = (size_t)K * kBThreads * (sizeof(float) + sizeof(int));
  if (lists > 48 * 1024 - 24 * 1024) {  // with the static part above the default: opt in
    const cudaError_t e = cudaFuncSetAttribute(
        expand_cluster_kernel<CL, E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lists);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * R * CL));
  cfg.blockDim = dim3(kBThreads);
  cfg.dynamicSmemBytes = lists;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CL;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, expand_cluster_kernel<CL, E>, logits, R, V, K, level,
                            static_cast<uint8_t*>(state), tree_build_stride(K, D), ftok, fslot,
                            status);
}

__device__ __forceinline__ uint32_t value_key(float v) {  // larger value <-> smaller key
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // order-preserving
  return ~u;
}

__global__ void __launch_bounds__(kFinThreads) finalize_kernel(const uint8_t* __restrict__ state,
                                                               size_t stride,
                                                               const int32_t* root_tokens, int N,
                                                               int32_t* tree_tokens,
                                                               int32_t* tree_parent,
                                                               int32_t* node_row,
                                                               float* node_value,
                                                               int32_t* status) {
  // (value, pool index) keys, sorted ascending = best first; a node's pool index orders it by
  // (depth, candidate order), the tie rule
  __shared__ unsigned long long key[kMaxTreePool];
  __shared__ short spos[kMaxTreePool];  // chosen: tree position; else -1
  __shared__ int wscan[kFinThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, b = blockIdx.x;
  const BuildHeader* hdr = reinterpret_cast<const BuildHeader*>(state + (size_t)b * stride);
  const PoolEntry* pool =
      reinterpret_cast<const PoolEntry*>(state + (size_t)b * stride + sizeof(BuildHeader));
  griddep_wait();
  griddep_launch_dependents();
  const int level = __ldcg(&hdr->level), flags = __ldcg(&hdr->flags);
  const int n = (level >= 1 && !(flags & SPEC_ST_NONFINITE)) ? __ldcg(&hdr->count) : 1;
  if (tid == 0 && status && (flags & SPEC_ST_NONFINITE)) atomicOr(status + b, SPEC_ST_NONFINITE);
  int np2 = 1;
  while (np2 < n) np2 <<= 1;
  for (int c = tid; c < np2; c += kFinThreads) {
    // the root sorts first (it is always in the tree); padding last
    key[c] = c == 0 ? 0ull
             : c < n ? ((unsigned long long)value_key(__ldcg(&pool[c].value)) << 32) | (unsigned)c
                     : ~0ull;
    if (c < n) spos[c] = -1;
  }
  __syncthreads();
  for (int k = 2; k <= np2; k <<= 1) {  // bitonic sort, ascending
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int a = tid; a < np2; a += kFinThreads) {
        const int p = a ^ j;
        if (p > a) {
          const unsigned long long x = key[a], y = key[p];
          const bool up = (a & k) == 0;
          if ((x > y) == up) {
            key[a] = y;
            key[p] = x;
          }
        }
      }
      __syncthreads();
    }
  }
  const int nsel = min(N - 1, n - 1);  // the chosen candidates: key[1 .. nsel]
  for (int r = 1 + tid; r <= nsel; r += kFinThreads) spos[(int)(key[r] & 0xffffffffu)] = 0;
  __syncthreads();
  // tree position of a chosen node: 1 + chosen nodes with a lower pool index (block scan)
  int run = 0;  // chosen nodes below this thread's range
  const int per = (n + kFinThreads - 1) / kFinThreads;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int mine = 0;
  for (int c = max(lo, 1); c < hi; ++c) mine += spos[c] >= 0 ? 1 : 0;
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wscan[w] = incl;
  __syncthreads();
  for (int q = 0; q < w; ++q) run += wscan[q];
  run += incl - mine;
  for (int c = max(lo, 1); c < hi; ++c)
    if (spos[c] >= 0) spos[c] = (short)(1 + run++);
  __syncthreads();
  int32_t* tt = tree_tokens + (size_t)b * N;
  int32_t* tp = tree_parent + (size_t)b * N;
  int32_t* tr = node_row ? node_row + (size_t)b * N : nullptr;
  float* tv = node_value ? node_value + (size_t)b * N : nullptr;
  for (int j = tid; j < N; j += kFinThreads) {  // padding past the chosen nodes
    if (j > nsel) {
      tt[j] = -1;
      tp[j] = -1;
      if (tr) tr[j] = -1;
      if (tv) tv[j] = __int_as_float(0x7fc00000);
    }
  }
  if (tid == 0) {
    tt[0] = root_tokens[b];
    tp[0] = -1;
    if (tr) tr[0] = level >= 1 ? 0 : -1;
    if (tv) tv[0] = 0.f;
  }
  for (int r = 1 + tid; r <= nsel; r += kFinThreads) {
    const int c = (int)(key[r] & 0xffffffffu);
    const int j = spos[c];
    const PoolEntry e = pool[c];
    tt[j] = e.token;
    tp[j] = e.parent == 0 ? 0 : spos[e.parent];
    if (tr) tr[j] = int((e.meta >> 12) & 0xfffu) - 1;
    if (tv) tv[j] = e.value;
  }
}

}  // namespace

size_t tree_build_stride(int K, int D) {
  const long long pool = 1 + K + (long long)(D - 1) * K * K;
  return (sizeof(BuildHeader) + (size_t)pool * sizeof(PoolEntry) + 127) & ~size_t(127);
}

cudaError_t launch_tree_expand(const float* logits, int B, int R, int V, int K, int D, int level,
                               void* state, int32_t* ftok, int32_t* fslot, int32_t* status,
                               cudaStream_t s) {
  // a cluster per row with the row in registers (up to 8 CTAs x 512 threads x 32 elements) while
  // the launch stays within 2048 CTAs: it shortens a row's latency, and with more rows than that
  // one CTA per row already fills the GPU
  const int per16 = kBThreads * 16;
  const long long need = V <= per16 ? 1 : V <= 2 * per16 ? 2 : V <= 4 * per16 ? 4 : 8;
  if ((long long)B * R * need <= 2048 || (need == 1 && (long long)B * R <= 0x7fffffffLL)) {
    if (V <= per16) return launch_expand_cluster<1, 16>(logits, B, R, V, K, D, level, state, ftok,
                                                        fslot, status, s);
    if (V <= 2 * per16) return launch_expand_cluster<2, 16>(logits, B, R, V, K, D, level, state,
                                                            ftok, fslot, status, s);
    if (V <= 4 * per16) return launch_expand_cluster<4, 16>(logits, B, R, V, K, D, level, state,
                                                            ftok, fslot, status, s);
    if (V <= 8 * per16) return launch_expand_cluster<8, 16>(logits, B, R, V, K, D, level, state,
                                                            ftok, fslot, status, s);
    if (V <= 16 * per16) return launch_expand_cluster<8, 32>(logits, B, R, V, K, D, level, state,
                                                             ftok, fslot, status, s);
  }
  // larger rows: one CTA per row, two passes over it
  const size_t lists = (size_t)K * kBThreads * (sizeof(float) + sizeof(int));
  if (lists + sizeof(ExpandSmem) > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(expand_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lists);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * R));
  cfg.blockDim = dim3(kBThreads);
  cfg.dynamicSmemBytes = lists;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, expand_rows_kernel, logits, R, V, K, level,
                            static_cast<uint8_t*>(state), tree_build_stride(K, D), ftok, fslot,
                            status);
}

cudaError_t launch_tree_finalize(const void* state, int B, int K, int D, const int32_t* root_tokens,
                                 int N, int32_t* tree_tokens, int32_t* tree_parent,
                                 int32_t* node_row, float* node_value, int32_t* status,
                                 cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B);
  cfg.blockDim = dim3(kFinThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, finalize_kernel, static_cast<const uint8_t*>(state),
                            tree_build_stride(K, D), root_tokens, N, tree_tokens, tree_parent,
                            node_row, node_value, status);
}

}  // namespace spectree
