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
// expand_kernel: one CTA per draft row of the level.  A pass over the row keeps each thread's best K
// entries; K rounds of a CTA-wide argmax merge them; a second pass (L2) sums exp(x - m) with a
// compensated sum for the log-sum-exp.  The CTA appends its K candidates to the pool; the last CTA
// of the sequence to arrive (counter + fences, no waiting) ranks the level's candidates and writes
// the frontier.  finalize_kernel: one CTA per sequence ranks the pool by counting and writes the tree.
#include "common.cuh"
#include "internal.h"

namespace spectree {

namespace {

constexpr int kBThreads = 256;
constexpr int kFinThreads = 512;

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

// (x, y) ranks before (v, z): larger value, then lower index
__device__ __forceinline__ bool before(float x, int y, float v, int z) {
  return x > v || (x == v && y < z);
}

struct ExpandSmem {
  float lv[kMaxTreeK][kBThreads];  // each thread's best entries (value), best first
  int li[kMaxTreeK][kBThreads];    // and their token ids
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

__global__ void __launch_bounds__(kBThreads) expand_kernel(const float* __restrict__ logits, int R,
                                                           int V, int K, int level,
                                                           uint8_t* __restrict__ state,
                                                           size_t stride, int32_t* ftok,
                                                           int32_t* fslot, int32_t* status) {
  __shared__ ExpandSmem sm;
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

  // ---- pass 1: each thread's best K entries (insertion into its column of the lists)
  for (int k = 0; k < K; ++k) {
    sm.lv[k][tid] = -INFINITY;
    sm.li[k][tid] = 0x7fffffff;
  }
  if (tid == 0 && level == 1) {  // a new construction (one CTA per sequence at level 1)
    hdr->flags = 0;
    hdr->arrived = 0;
  }
  __syncthreads();
  bool bad = false;
  float worst_v = -INFINITY;
  int worst_i = 0x7fffffff;
  for (int y = tid; y < V; y += kBThreads) {
    const float x = __ldg(row + y);
    if (isnan(x) || x == INFINITY) {
      bad = true;
      continue;
    }
    if (!before(x, y, worst_v, worst_i)) continue;
    int p = K - 1;  // shift the worse entries down, insert
    while (p > 0 && before(x, y, sm.lv[p - 1][tid], sm.li[p - 1][tid])) {
      sm.lv[p][tid] = sm.lv[p - 1][tid];
      sm.li[p][tid] = sm.li[p - 1][tid];
      --p;
    }
    sm.lv[p][tid] = x;
    sm.li[p][tid] = y;
    worst_v = sm.lv[K - 1][tid];
    worst_i = sm.li[K - 1][tid];
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) atomicOr(&hdr->flags, SPEC_ST_NONFINITE);
    bad = true;
  }
  // ---- merge: K rounds of a CTA-wide argmax over the threads' heads
  int head = 0;
  if (!bad) {
    for (int k = 0; k < K; ++k) {
      float v = head < K ? sm.lv[head][tid] : -INFINITY;
      int y = head < K ? sm.li[head][tid] : 0x7fffffff;
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
  // ---- pass 2: log-sum-exp (compensated sum of exp(x - m), m = the row max)
  float lse = 0.f;
  if (!bad) {
    const float m = sm.best_v[0];
    CompSum acc;
    for (int y = tid; y < V; y += kBThreads) acc.add(__expf(__fsub_rn(__ldg(row + y), m)));
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
  }
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

__global__ void __launch_bounds__(kFinThreads) finalize_kernel(const uint8_t* __restrict__ state,
                                                               size_t stride,
                                                               const int32_t* root_tokens, int N,
                                                               int32_t* tree_tokens,
                                                               int32_t* tree_parent,
                                                               int32_t* node_row,
                                                               float* node_value,
                                                               int32_t* status) {
  __shared__ float sv[kMaxTreePool];
  __shared__ uint32_t smeta[kMaxTreePool];
  __shared__ short spos[kMaxTreePool];
  const int tid = threadIdx.x, b = blockIdx.x;
  const BuildHeader* hdr = reinterpret_cast<const BuildHeader*>(state + (size_t)b * stride);
  const PoolEntry* pool =
      reinterpret_cast<const PoolEntry*>(state + (size_t)b * stride + sizeof(BuildHeader));
  griddep_wait();
  griddep_launch_dependents();
  const int level = __ldcg(&hdr->level), flags = __ldcg(&hdr->flags);
  const int n = (level >= 1 && !(flags & SPEC_ST_NONFINITE)) ? __ldcg(&hdr->count) : 1;
  if (tid == 0 && status && (flags & SPEC_ST_NONFINITE)) atomicOr(status + b, SPEC_ST_NONFINITE);
  for (int c = tid; c < n; c += kFinThreads) {
    sv[c] = c ? __ldcg(&pool[c].value) : 0.f;
    smeta[c] = c ? __ldcg(&pool[c].meta) : 0u;
    spos[c] = -1;
  }
  __syncthreads();
  const int nsel = min(N - 1, n - 1);
  // rank among the candidates: larger value, then shallower, then lower order
  for (int c = 1 + tid; c < n; c += kFinThreads) {
    const float v = sv[c];
    const uint32_t k = smeta[c] & 0xff000fffu;  // depth and order
    int r = 0;
    for (int o = 1; o < n; ++o) {
      const float v2 = sv[o];
      r += (v2 > v || (v2 == v && (smeta[o] & 0xff000fffu) < k)) ? 1 : 0;
    }
    spos[c] = r < nsel ? 0 : -1;  // chosen (position below)
  }
  __syncthreads();
  // position: 1 + the chosen nodes before it in (depth, order)
  for (int c = 1 + tid; c < n; c += kFinThreads) {
    if (spos[c] < 0) continue;
    const uint32_t k = smeta[c] & 0xff000fffu;
    int p = 1;
    for (int o = 1; o < n; ++o) p += (spos[o] >= 0 && (smeta[o] & 0xff000fffu) < k) ? 1 : 0;
    spos[c] = (short)p;  // (other threads only test spos >= 0, which this keeps)
  }
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
  for (int c = 1 + tid; c < n; c += kFinThreads) {
    const int j = spos[c];
    if (j < 0) continue;
    const int par = __ldcg(&pool[c].parent);
    tt[j] = __ldcg(&pool[c].token);
    tp[j] = par == 0 ? 0 : spos[par];
    if (tr) tr[j] = int((smeta[c] >> 12) & 0xfffu) - 1;
    if (tv) tv[j] = sv[c];
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * R));
  cfg.blockDim = dim3(kBThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, expand_kernel, logits, R, V, K, level,
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
