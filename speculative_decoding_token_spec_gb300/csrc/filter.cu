// Top-k / top-p filtering of target-logit rows for filtered verification (sm_103a).
//
// Method: survey explainer, verification taxonomy -- speculative sampling carries over to top-k
// and top-p sampling, with the filtered target distribution in the accept/reject test and the
// residual.  Reading: temperature first, then top-k on the logits (every logit >= the k-th largest
// is kept), then top-p on the renormalised top-k distribution (a token is kept when the mass of
// the strictly more probable tokens is < top_p).  Both kept sets are "every logit >= a
// threshold" (probabilities are monotone in the logit), so each row reduces to two thresholds.
// The row is rewritten with -inf outside the kept set; softmax(l' / T) is then exactly the
// filtered, renormalised distribution, and the verification kernel runs on l' unchanged.
//
// Layout: a cluster of CL CTAs (1..8) per row, each holding a slice of E elements per thread in
// shared memory (thread t of rank r: elements r * 512 E + t + 512 i, loaded once).  Both
// thresholds are exact selections over the order-preserving integer keys of the fp32 logits:
//   1. the row max m (cluster-wide);
//   2. level 1: a histogram over 256 bins of the log2-distance to the max, d = (m - x) log2(e) / T,
//      1/8 unit per bin (bin 0: d >= 31.75 and -inf).  The bin is a monotone function of the
//      logit, so it orders the row like the keys do, and it spreads a logit row over many bins
//      (8-bit digits of the raw keys would pile it onto a few sign / exponent bins).  Counts serve
//      top-k, unnormalised probabilities e = 2^-d in 2^-40 fixed point serve top-p: integer sums,
//      exact and order-independent, each e truncated by at most 2^-40 of the max's.  Masses are
//      added as three 14-bit parts so that every shared-memory atomic is a native 32-bit one;
//   3. the bins that can hold a threshold follow from level 1 (the k-th largest key's bin; for
//      top-p, the bins between the positions the mass threshold takes for the smallest and the
//      largest top-k mass that bin allows).  When they hold at most kCap elements, their keys are
//      gathered into every CTA of the cluster and each CTA resolves both thresholds on its own
//      (radix levels over the bits where the candidates differ, CTA barriers only).  Otherwise
//      the cluster resolves them together, four 8-bit radix levels over the slices.
// Level totals reach every CTA through shared::cluster reductions and a cluster barrier, so every
// CTA takes the same decision from the same integers.  A row holding NaN or +Inf is copied
// unchanged (verification flags it).
#include "common.cuh"
#include "internal.h"

namespace spectree {

namespace {

constexpr int kFThreads = 512;
constexpr int kFWarps = kFThreads / 32;
constexpr float kTailD = 31.75f;  // log2-distance where level 1's tail bin starts
constexpr int kCap = 2048;        // keys gathered per row on the fast path
constexpr int kRank = 256;        // candidates a selection ranks directly (else radix levels)

typedef unsigned long long u64;

__device__ __forceinline__ uint32_t order_key(float x) {  // larger float <-> larger key
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;  // -0 and +0 are equal logits: one key
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k) {  // inverse of order_key (-0 -> +0)
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// e = 2^f (f <= 0) as an integer multiple of 2^-40, truncated (integer arithmetic on the fields
// of the float: the value is mantissa * 2^(exponent - 127 - 23 + 40)).
__device__ __forceinline__ u64 fixed_e(float f) {
  const uint32_t b = __float_as_uint(ex2_fast(f));
  const int ex = int(b >> 23);
  if (ex == 0) return 0ull;
  const u64 mant = (b & 0x7fffffu) | 0x800000u;
  const int sh = ex - 110;
  if (sh >= 0) return mant << sh;
  return sh > -24 ? (mant >> -sh) : 0ull;
}

// ceil(p * total) for 0 < p < 1, exactly: p = mant * 2^-s, and the 128-bit product is shifted
// right by s with the remainder rounding up (integer arithmetic; no FP64).
__device__ __forceinline__ u64 ceil_mul(float p, u64 total) {
  const uint32_t b = __float_as_uint(p);
  const int ex = int(b >> 23);
  const u64 mant = ex ? ((b & 0x7fffffu) | 0x800000u) : (b & 0x7fffffu);
  const int s = ex ? 150 - ex : 149;  // >= 24 for p < 1
  const u64 lo = total * mant, hi = __umul64hi(total, mant);
  u64 q;
  bool rem;
  if (s >= 128) {
    q = 0;
    rem = (hi | lo) != 0;
  } else if (s >= 64) {
    const int r = s - 64;
    q = r ? hi >> r : hi;
    rem = lo != 0 || (r && (hi & ((1ull << r) - 1)) != 0);
  } else {
    q = (lo >> s) | (hi << (64 - s));
    rem = (lo & ((1ull << s) - 1)) != 0;
  }
  return q + (rem ? 1ull : 0ull);
}

__device__ __forceinline__ void red_add_cluster(uint32_t addr, u64 v) {
  asm volatile("red.relaxed.cluster.shared::cluster.add.u64 [%0], %1;" ::"r"(addr), "l"(v)
               : "memory");
}
__device__ __forceinline__ void red_add_cluster32(uint32_t addr, uint32_t v) {
  asm volatile("red.relaxed.cluster.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v)
               : "memory");
}
__device__ __forceinline__ void red_max_cluster(uint32_t addr, uint32_t v) {
  asm volatile("red.relaxed.cluster.shared::cluster.max.u32 [%0], %1;" ::"r"(addr), "r"(v)
               : "memory");
}
__device__ __forceinline__ uint32_t atom_add_cluster32(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.relaxed.cluster.shared::cluster.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(addr), "r"(v)
               : "memory");
  return old;
}

// Histogram entry add: a count and, with masses, the mass e in three 14-bit parts (every part sum
// stays below 2^32 for any row of at most 2^18 elements).
__device__ __forceinline__ void hist_add(uint32_t (*h)[256], int b, bool masses, u64 e,
                                         uint32_t c = 1u) {
  atomicAdd(&h[0][b], c);
  if (masses) {
    const uint32_t m0 = uint32_t(e) & 0x3fffu, m1 = uint32_t(e >> 14) & 0x3fffu;
    const uint32_t m2 = uint32_t(e >> 28);
    if (m0) atomicAdd(&h[1][b], m0);
    if (m1) atomicAdd(&h[2][b], m1);
    if (m2) atomicAdd(&h[3][b], m2);
  }
}
__device__ __forceinline__ u64 parts_sum(const uint32_t (*h)[256], int b) {
  return (u64)h[1][b] + ((u64)h[2][b] << 14) + ((u64)h[3][b] << 28);
}

struct PickResult {
  int digit;
  u64 above_p, above_s;  // primary / secondary totals of the bins above the digit
  u64 sel_p, sel_s;      // the digit's own bin
};

struct Plan {
  int hk;             // level-1 bin of the k-th largest key (-1: no top-k)
  int glo, ghi;       // level-1 bins that can hold the top-p threshold (glo > ghi: none)
  int fast;           // gather the candidates (n <= kCap)
  uint32_t n;         // elements in the gathered bins
  u64 above_c;        // count of the bins above hk
  u64 above_m1;       // mass of the bins above hk
  u64 total;          // the row's mass (no top-k)
};

struct Selected {
  uint32_t key;  // the selected key
  u64 ge2;       // secondary total (masses when selecting by count) of the candidates >= key
};

struct FilterSmem {
  uint32_t lh[4][256];     // this CTA's histogram of the current level: count, mass parts
  uint32_t th[4][256];     // level 1: cluster totals of lh (remote reductions land here)
  u64 g1c[256], g1m[256];  // level 1 cluster totals, 64-bit
  union {
    struct {
      u64 rc[2][256], rm[2][256];  // cluster radix levels: totals, alternating
      u64 lc[256], lm[256];        // this CTA's histogram of a cluster radix level
    } rad;
    struct {
      uint32_t key[kCap];  // the gathered keys (written by every CTA of the cluster)
      u64 mass[kCap];      // their masses; before that, this CTA's keys to send (as uint32)
    } cand;
  } u;
  uint32_t skey[kRank];  // a selection's candidates, when they are few enough to rank
  u64 swt[kRank][2];      // and their weights: count (1) and mass
  u64 wsum[kFWarps], wv[8], ws[8];
  uint32_t lmax, cmax, ncand, kmin, kmax, lcount, gbase, nsel, sel;
  int glo_s, ghi_s;
  u64 sel_ge2;
  int lbad, cbad;
  PickResult pick, pick2;
};

// Cluster barrier (release / acquire) for CL > 1, a CTA barrier otherwise.
template <int CL>
__device__ __forceinline__ void cl_sync() {
  if constexpr (CL > 1) {
    cluster_arrive_release();
    cluster_wait_acquire();
  } else {
    __syncthreads();
  }
}

// Called by every thread of the CTA (two CTA barriers inside); thread t < 256 owns bin 255 - t and
// obtains its primary / secondary values with get(bin, v, s).  For each need, the highest bin d
// whose primary value makes the running total from the top reach it (base + bins above d + bin d
// >= need), with the primary / secondary totals above d and of bin d; bin 0 if never met.  The
// result for need2 (if given) is left in sm.pick2; own_above_s (if given) receives, in threads
// 0..255, the secondary total of the bins above the thread's own.
template <class Get>
__device__ PickResult pick_block(FilterSmem& sm, Get get, u64 base, u64 need,
                                 const u64* need2 = nullptr, u64* own_above_s = nullptr) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  u64 v = 0, sv = 0, iv = 0, is = 0;
  if (t < 256) {
    get(255 - t, v, sv);
    iv = v;
    is = sv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {  // inclusive scans over the warp's 32 bins
      const u64 a = __shfl_up_sync(0xffffffffu, iv, o);
      const u64 b = __shfl_up_sync(0xffffffffu, is, o);
      if (lane >= o) {
        iv += a;
        is += b;
      }
    }
    if (lane == 31) {
      sm.wv[w] = iv;
      sm.ws[w] = is;
    }
  }
  __syncthreads();
  if (t < 256) {
    u64 ov = 0, os = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < w) {
        ov += sm.wv[i];
        os += sm.ws[i];
      }
    }
    const u64 ev = ov + iv - v, es = os + is - sv;  // totals of the bins above
    if (own_above_s) *own_above_s = es;
    auto take = [&](u64 nd, PickResult& out) {
      const bool reach = base + ev + v >= nd;
      if ((reach && (t == 0 || base + ev < nd)) || (t == 255 && !reach)) {
        out.digit = 255 - t;
        out.above_p = ev;
        out.above_s = es;
        out.sel_p = v;
        out.sel_s = sv;
      }
    };
    take(need, sm.pick);
    if (need2) take(*need2, sm.pick2);
  }
  __syncthreads();
  return sm.pick;
}

// Sum over the CTA (every thread gets it).
__device__ u64 block_sum(FilterSmem& sm, u64 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) sm.wsum[threadIdx.x >> 5] = v;
  __syncthreads();
  u64 s = 0;
#pragma unroll
  for (int w = 0; w < kFWarps; ++w) s += sm.wsum[w];
  __syncthreads();
  return s;
}

// Fast path: among the gathered keys for which pred(key) holds, the key where the running total
// from the top (counts, or masses if by_mass) reaches need, given `base` above them, and the
// secondary total of the candidates >= that key.  Up to kRank candidates are ranked directly
// (each key's totals above it, summed by 2..8 threads); more go through radix levels of up to 8
// bits over the bits below their common prefix.  CTA barriers only.
template <class Pred>
__device__ Selected local_select(FilterSmem& sm, int n, Pred pred, u64 base, u64 need,
                                 bool by_mass) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid == 0) {
    sm.kmin = 0xffffffffu;
    sm.kmax = 0u;
    sm.nsel = 0u;
  }
  __syncthreads();
  uint32_t mn = 0xffffffffu, mx = 0u;
  for (int j0 = 0; j0 < n; j0 += kFThreads) {
    const int j = j0 + tid;
    const uint32_t key = j < n ? sm.u.cand.key[j] : 0u;
    const bool in = j < n && pred(key);
    const unsigned bal = __ballot_sync(0xffffffffu, in);
    uint32_t slot = 0;
    if (lane == 0 && bal) slot = atomicAdd(&sm.nsel, (uint32_t)__popc(bal));
    slot = __shfl_sync(0xffffffffu, slot, 0) + __popc(bal & ((1u << lane) - 1u));
    if (in) {
      mn = min(mn, key);
      mx = max(mx, key);
      if (slot < (uint32_t)kRank) {
        sm.skey[slot] = key;
        sm.swt[slot][0] = 1ull;
        sm.swt[slot][1] = sm.u.cand.mass[j];
      }
    }
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) {
    atomicMin(&sm.kmin, mn);
    atomicMax(&sm.kmax, mx);
  }
  __syncthreads();
  const int ns = (int)sm.nsel;
  Selected res;
  if (ns <= kRank) {
    // ---- rank: thread group i sums the weights of the keys above / at key i
    const int tpc = ns <= 64 ? 8 : (ns <= 128 ? 4 : 2);
    const int i = tid / tpc, part = tid % tpc;
    const int pw = by_mass ? 1 : 0;  // primary weight: mass or count
    u64 gt = 0, ge = 0, ge2 = 0;
    uint32_t ki = 0;
    if (i < ns) {
      ki = sm.skey[i];
      for (int j = part; j < ns; j += tpc) {
        const uint32_t kj = sm.skey[j];
        const u64 w1 = sm.swt[j][pw], w2 = sm.swt[j][pw ^ 1];
        if (kj > ki) gt += w1;
        if (kj >= ki) {
          ge += w1;
          ge2 += w2;
        }
      }
    }
    for (int o = 1; o < tpc; o <<= 1) {
      gt += __shfl_xor_sync(0xffffffffu, gt, o);
      ge += __shfl_xor_sync(0xffffffffu, ge, o);
      ge2 += __shfl_xor_sync(0xffffffffu, ge2, o);
    }
    if (tid == 0) {  // need never met: the smallest key, all candidates
      sm.sel = sm.kmin;
      sm.sel_ge2 = ~0ull;
    }
    __syncthreads();
    if (part == 0 && i < ns && base + gt < need && base + ge >= need) {
      sm.sel = ki;  // every candidate with the selected key writes the same values
      sm.sel_ge2 = ge2;
    }
    __syncthreads();
    res.key = sm.sel;
    res.ge2 = sm.sel_ge2;
    if (res.ge2 == ~0ull) {  // (not reached for a consistent need) total of all candidates
      u64 all2 = 0;
      for (int j = tid; j < ns; j += kFThreads) all2 += sm.swt[j][pw ^ 1];
      res.ge2 = block_sum(sm, all2);
    }
    __syncthreads();  // every thread is done with kmin / kmax / nsel / sel
    return res;
  }
  // ---- radix levels over the bits where the candidates differ
  const uint32_t diff = sm.kmin ^ sm.kmax;
  int nb = diff ? 32 - __clz(diff) : 0;
  uint32_t prefix = nb >= 32 ? 0u : (sm.kmin >> nb) << nb;
  u64 ab = base;
  while (nb > 0) {
    const int shift = max(nb - 8, 0);
    const uint32_t dmask = (1u << (nb - shift)) - 1u;
    for (int j = tid; j < n; j += kFThreads) {
      const uint32_t key = sm.u.cand.key[j];
      if (pred(key) && (nb >= 32 || (key >> nb) == (prefix >> nb)))
        hist_add(sm.lh, int((key >> shift) & dmask), by_mass, sm.u.cand.mass[j]);
    }
    __syncthreads();
    // each bin's owner reads it and clears it for the next level
    const PickResult r = pick_block(
        sm,
        [&](int d, u64& v, u64& w) {
          const u64 c = sm.lh[0][d], ms = by_mass ? parts_sum(sm.lh, d) : 0ull;
          sm.lh[0][d] = sm.lh[1][d] = sm.lh[2][d] = sm.lh[3][d] = 0u;
          v = by_mass ? ms : c;
          w = by_mass ? c : ms;
        },
        ab, need);
    ab += r.above_p;
    prefix |= (uint32_t)r.digit << shift;
    nb = shift;
  }
  res.key = prefix;
  u64 part2 = 0;  // secondary total of the candidates >= the selected key
  for (int j = tid; j < n; j += kFThreads) {
    const uint32_t key = sm.u.cand.key[j];
    if (key >= prefix && pred(key)) part2 += by_mass ? 1ull : sm.u.cand.mass[j];
  }
  res.ge2 = block_sum(sm, part2);
  __syncthreads();  // every thread is done with kmin / kmax
  return res;
}

template <int CL, int E>
__global__ void __launch_bounds__(kFThreads, 2) filter_kernel(const float* __restrict__ in,
                                                              float* __restrict__ out, int V,
                                                              float k2, int top_k, float top_p) {
  __shared__ FilterSmem sm;
  extern __shared__ float4 xs_raw[];  // the slice: element i of thread t at xs[i * 512 + t],
  float* xs = reinterpret_cast<float*>(xs_raw);  // then (E == 16) its level-1 bins, as bytes
  uint8_t* hb = reinterpret_cast<uint8_t*>(xs + E * kFThreads);
  constexpr bool kBinCache = E == 16;
  const int tid = threadIdx.x, lane = tid & 31;
  const int rank = (CL > 1) ? int(blockIdx.x % CL) : 0;
  const size_t row_id = blockIdx.x / CL;
  const float* row = in + row_id * (size_t)V;
  float* dst = out + row_id * (size_t)V;
  const int y0 = rank * kFThreads * E + tid;
  const bool use_k = top_k > 0 && top_k < V;
  const bool use_p = top_p < 1.f;

  for (int i = tid; i < 256; i += kFThreads)
#pragma unroll
    for (int a = 0; a < 4; ++a) sm.lh[a][i] = sm.th[a][i] = 0u;
  if (tid == 0) {
    sm.lmax = sm.cmax = sm.ncand = sm.lcount = 0u;
    sm.glo_s = sm.ghi_s = -1;
    sm.lbad = sm.cbad = 0;
  }
  if constexpr (CL > 1) cluster_arrive_release();  // this CTA's totals are zeroed
  griddep_wait();  // the logits may come from the preceding kernel
  griddep_launch_dependents();

  // ---- load (16 elements in flight per thread) and max pass
  uint32_t mk = 0;
  bool bad = false;
#pragma unroll
  for (int i0 = 0; i0 < E; i0 += 16) {
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int y = y0 + (i0 + i) * kFThreads;
      v[i] = (y < V) ? __ldg(row + y) : -INFINITY;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      xs[(i0 + i) * kFThreads + tid] = v[i];
      bad |= isnan(v[i]) || v[i] == INFINITY;
      mk = max(mk, order_key(v[i]));
    }
  }
  auto x = [&](int i) { return xs[i * kFThreads + tid]; };
  mk = __reduce_max_sync(0xffffffffu, mk);
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    atomicMax(&sm.lmax, mk);
    if (bad) sm.lbad = 1;
  }
  __syncthreads();
  if constexpr (CL > 1) {
    cluster_wait_acquire();  // every CTA's totals are zeroed: reductions may land
    if (tid < CL) {
      red_max_cluster(dsmem_addr(&sm.cmax, tid), sm.lmax);
      red_max_cluster(dsmem_addr(&sm.cbad, tid), (uint32_t)sm.lbad);
    }
    cl_sync<CL>();
  } else {
    if (tid == 0) {
      sm.cmax = sm.lmax;
      sm.cbad = sm.lbad;
    }
    __syncthreads();
  }
  if (sm.cbad) {  // the whole cluster takes this branch
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const int y = y0 + i * kFThreads;
      if (y < V) dst[y] = x(i);
    }
    return;
  }
  const float m = key_float(sm.cmax);
  // f(x) = (x - m) log2(e) / T <= 0, monotone in x; the level-1 bin of f: 255 at the max .. 2,
  // 0 for the tail and -inf
  auto fdist = [&](float v) { return __fmul_rn(__fsub_rn(v, m), k2); };
  auto bin_f = [](float f) -> int { return (f > -kTailD) ? 255 - (int)(-f * 8.f) : 0; };
  auto bin_key = [&](uint32_t key) { return bin_f(fdist(key_float(key))); };
  auto bin_at = [&](int i) -> int {  // level-1 bin of element i (after level 1)
    if constexpr (kBinCache) return hb[i * kFThreads + tid];
    return bin_f(fdist(x(i)));
  };
  const bool row_live = m != -INFINITY;  // an all -inf row keeps everything (all -inf)
  uint32_t th = 0;                       // keep key >= th
  if (row_live && (use_k || use_p)) {
    // ---- level 1
    u64 tail_c = 0, tail_m = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const int y = y0 + i * kFThreads;
      if (y >= V) continue;
      const float f = fdist(x(i));
      const int h = bin_f(f);
      if constexpr (kBinCache) hb[i * kFThreads + tid] = (uint8_t)h;
      const u64 e = use_p ? fixed_e(f) : 0ull;
      if (h == 0) {
        tail_c += 1;
        tail_m += e;
      } else {
        hist_add(sm.lh, h, use_p, e);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tail_c += __shfl_xor_sync(0xffffffffu, tail_c, o);
      tail_m += __shfl_xor_sync(0xffffffffu, tail_m, o);
    }
    if (lane == 0 && tail_c) hist_add(sm.lh, 0, use_p, tail_m, (uint32_t)tail_c);
    __syncthreads();
    if (tid < 256) {
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const uint32_t v = sm.lh[a][tid];
        sm.lh[a][tid] = 0u;
        if (v == 0u) continue;
        if constexpr (CL > 1) {
#pragma unroll
          for (int r = 0; r < CL; ++r) red_add_cluster32(dsmem_addr(&sm.th[a][tid], r), v);
        } else {
          sm.th[a][tid] += v;
        }
      }
    }
    cl_sync<CL>();
    if (tid < 256) {
      sm.g1c[tid] = sm.th[0][tid];
      sm.g1m[tid] = parts_sum(sm.th, tid);
    }
    __syncthreads();

    // ---- plan: the level-1 bins that can hold the thresholds
    Plan P;
    P.hk = -1;
    P.above_c = P.above_m1 = P.total = 0;
    P.glo = 256;
    P.ghi = -1;
    if (use_k) {
      // the k-th largest key's bin; the same scan gives every bin's mass above it, from which the
      // bins that can hold the top-p threshold follow: the top-k set's mass lies in (mass above
      // hk, mass above hk + bin hk], so the threshold bin lies between the bins where the
      // running mass from the top reaches top_p of either end (hk if no bin above does)
      u64 ev_m = 0, v_m = 0;
      const PickResult r = pick_block(
          sm,
          [&](int d, u64& v, u64& w) {
            v = sm.g1c[d];
            w = sm.g1m[d];
            v_m = w;
          },
          0ull, (u64)top_k, nullptr, &ev_m);
      P.hk = r.digit;
      P.above_c = r.above_p;
      P.above_m1 = r.above_s;
      if (use_p) {
        const u64 need_hi = ceil_mul(top_p, P.above_m1 + r.sel_s);
        const u64 need_lo = ceil_mul(top_p, P.above_m1);
        const int b = 255 - tid;
        if (tid < 256 && b > P.hk) {
          const u64 cum = ev_m + v_m;  // mass of the bins >= b
          if (cum >= need_hi && (tid == 0 || ev_m < need_hi)) atomicMax(&sm.glo_s, b);
          if (cum >= need_lo && (tid == 0 || ev_m < need_lo)) atomicMax(&sm.ghi_s, b);
        }
        __syncthreads();
        P.glo = max(sm.glo_s, P.hk);
        P.ghi = max(sm.ghi_s, P.hk);
      }
    } else if (use_p) {
      P.total = block_sum(sm, tid < 256 ? sm.g1m[tid] : 0ull);
      const PickResult r = pick_block(
          sm, [&](int d, u64& v, u64& w) { v = sm.g1m[d]; w = 0; }, 0ull,
          ceil_mul(top_p, P.total));
      P.glo = P.ghi = r.digit;
    }
    const u64 n64 = block_sum(
        sm, (tid < 256 && (tid == P.hk || (tid >= P.glo && tid <= P.ghi))) ? sm.g1c[tid] : 0ull);
    P.n = (uint32_t)min(n64, (u64)0xffffffffu);
    P.fast = n64 <= (u64)kCap;

    uint32_t tk = 0, tp = 0;
    u64 mass_k = 0;  // mass of the keys >= tk
    if (P.fast) {
      // ---- gather the keys of the planned bins into every CTA of the cluster: this CTA's
      // keys first to a local list, then one range of the cluster's list reserved at rank 0
      uint32_t* stage = reinterpret_cast<uint32_t*>(sm.u.cand.mass);
      uint32_t* lst = (CL > 1) ? stage : sm.u.cand.key;
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const int y = y0 + i * kFThreads;
        bool want = false;
        if (y < V) {
          const int h = bin_at(i);
          want = h == P.hk || (h >= P.glo && h <= P.ghi);
        }
        const unsigned bal = __ballot_sync(0xffffffffu, want);
        if (bal == 0u) continue;
        uint32_t base = 0;
        if (lane == 0) base = atomicAdd(&sm.lcount, (uint32_t)__popc(bal));
        base = __shfl_sync(0xffffffffu, base, 0);
        const uint32_t slot = base + __popc(bal & ((1u << lane) - 1u));
        if (want && slot < (uint32_t)kCap) lst[slot] = order_key(x(i));  // the plan counted them
      }
      if constexpr (CL > 1) {
        __syncthreads();
        if (tid == 0) sm.gbase = atom_add_cluster32(dsmem_addr(&sm.ncand, 0), sm.lcount);
        __syncthreads();
        const uint32_t cnt = sm.lcount, gb = sm.gbase;
        for (uint32_t j = tid; j < cnt; j += kFThreads) {
          const uint32_t slot = gb + j, key = stage[j];
          if (slot < (uint32_t)kCap) {
#pragma unroll
            for (int r = 0; r < CL; ++r) dsmem_store_u32(dsmem_addr(&sm.u.cand.key[slot], r), key);
          }
        }
      }
      cl_sync<CL>();
      const int n = (int)P.n;
      for (int j = tid; j < n; j += kFThreads)
        sm.u.cand.mass[j] = use_p ? fixed_e(fdist(key_float(sm.u.cand.key[j]))) : 0ull;
      __syncthreads();
      if (use_k) {
        const int hk = P.hk;
        const Selected sk = local_select(
            sm, n, [&](uint32_t key) { return bin_key(key) == hk; }, P.above_c, (u64)top_k,
            false);
        tk = sk.key;
        mass_k = P.above_m1 + sk.ge2;
      }
      if (use_p) {
        // ---- top-p over the top-k set, on the gathered keys
        const u64 total = use_k ? mass_k : P.total;
        const u64 need = ceil_mul(top_p, total);
        const u64 part_k = mass_k - P.above_m1;  // bin hk's keys >= tk
        const int hk = P.hk;
        const PickResult r = pick_block(
            sm,
            [&](int d, u64& v, u64& w) {
              v = (hk < 0 || d > hk) ? sm.g1m[d] : (d == hk ? part_k : 0ull);
              w = 0;
            },
            0ull, need);
        const int hp = r.digit;
        tp = local_select(
                 sm, n, [&](uint32_t key) { return key >= tk && bin_key(key) == hp; }, r.above_p,
                 need, true)
                 .key;
      }
    } else {
      // ---- cluster radix over the slices (large candidate sets)
      for (int i = tid; i < 256; i += kFThreads) {
        sm.u.rad.lc[i] = sm.u.rad.lm[i] = 0ull;
        sm.u.rad.rc[0][i] = sm.u.rad.rm[0][i] = 0ull;
        sm.u.rad.rc[1][i] = sm.u.rad.rm[1][i] = 0ull;
      }
      cl_sync<CL>();  // every CTA's radix totals are zeroed before reductions land
      int lvl = 0;
      // Four radix levels over the candidates `cand` (bit i: element i), primary = counts or
      // masses; returns the selected key, adding the primary / secondary totals above it to
      // ap / as and setting sp / ss to the selected key's own.
      auto radix = [&](uint64_t cand, bool by_mass, u64 need, u64& ap, u64& as, u64& sp,
                       u64& ss) -> uint32_t {
        uint32_t prefix = 0;
        for (int shift = 24; shift >= 0; shift -= 8, ++lvl) {
          const int b = lvl & 1;
#pragma unroll
          for (int i = 0; i < E; ++i) {
            if (!((cand >> i) & 1ull)) continue;
            const float xi = x(i);
            const uint32_t dg = (order_key(xi) >> shift) & 255u;
            atomicAdd(&sm.u.rad.lc[dg], 1ull);
            if (use_p) atomicAdd(&sm.u.rad.lm[dg], fixed_e(fdist(xi)));
          }
          if (tid < 256) {  // the other totals were read at the previous level: clear them
            sm.u.rad.rc[b ^ 1][tid] = 0ull;
            sm.u.rad.rm[b ^ 1][tid] = 0ull;
          }
          __syncthreads();
          if (tid < 256) {
            const u64 c = sm.u.rad.lc[tid], ms = use_p ? sm.u.rad.lm[tid] : 0ull;
            sm.u.rad.lc[tid] = sm.u.rad.lm[tid] = 0ull;
            if (c) {
              if constexpr (CL > 1) {
#pragma unroll
                for (int r = 0; r < CL; ++r) {
                  red_add_cluster(dsmem_addr(&sm.u.rad.rc[b][tid], r), c);
                  if (ms) red_add_cluster(dsmem_addr(&sm.u.rad.rm[b][tid], r), ms);
                }
              } else {
                sm.u.rad.rc[b][tid] += c;
                sm.u.rad.rm[b][tid] += ms;
              }
            }
          }
          cl_sync<CL>();
          const u64* C = sm.u.rad.rc[b];
          const u64* M = sm.u.rad.rm[b];
          const PickResult pr = pick_block(
              sm,
              [&](int d, u64& v, u64& w) {
                v = by_mass ? M[d] : C[d];
                w = by_mass ? C[d] : M[d];
              },
              ap, need);
          ap += pr.above_p;
          as += pr.above_s;
          sp = pr.sel_p;
          ss = pr.sel_s;
          prefix |= (uint32_t)pr.digit << shift;
#pragma unroll
          for (int i = 0; i < E; ++i)
            if (((cand >> i) & 1ull) && ((order_key(x(i)) >> shift) & 255u) != (uint32_t)pr.digit)
              cand &= ~(1ull << i);
        }
        return prefix;
      };
      if (use_k) {
        uint64_t cand = 0;
#pragma unroll
        for (int i = 0; i < E; ++i) {
          const int y = y0 + i * kFThreads;
          if (y < V && bin_at(i) == P.hk) cand |= 1ull << i;
        }
        u64 ac = P.above_c, am = P.above_m1, sc = 0, smass = 0;
        tk = radix(cand, false, (u64)top_k, ac, am, sc, smass);
        mass_k = am + smass;
      }
      if (use_p) {
        const u64 total = use_k ? mass_k : P.total;
        const u64 need = ceil_mul(top_p, total);
        const u64 part_k = mass_k - P.above_m1;
        const int hk = P.hk;
        const PickResult p1 = pick_block(
            sm,
            [&](int d, u64& v, u64& w) {
              v = (hk < 0 || d > hk) ? sm.g1m[d] : (d == hk ? part_k : 0ull);
              w = 0;
            },
            0ull, need);
        uint64_t cand = 0;
#pragma unroll
        for (int i = 0; i < E; ++i) {
          const int y = y0 + i * kFThreads;
          if (y < V) {
            const float xi = x(i);
            if (bin_at(i) == p1.digit && order_key(xi) >= tk) cand |= 1ull << i;
          }
        }
        u64 am = p1.above_p, ac = 0, sm_ = 0, sc = 0;
        tp = radix(cand, true, need, am, ac, sm_, sc);
      }
    }
    th = max(tk, tp);
  }
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int y = y0 + i * kFThreads;
    if (y < V) {
      const float xi = x(i);
      dst[y] = order_key(xi) >= th ? xi : -INFINITY;
    }
  }
}

template <int CL, int E>
cudaError_t launch_fk(const float* in, float* out, int rows, int V, float k2, int top_k,
                      float top_p, cudaStream_t s) {
  static_assert(CL >= 1 && CL <= 8, "clusters stay within the portable size");
  const size_t smem = (size_t)E * kFThreads * (sizeof(float) + (E == 16 ? 1 : 0));
  if (smem + sizeof(FilterSmem) > 48 * 1024) {  // above the default limit: opt in
    const cudaError_t e = cudaFuncSetAttribute(
        filter_kernel<CL, E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)rows * CL);
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = smem;
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
  return cudaLaunchKernelEx(&cfg, filter_kernel<CL, E>, in, out, V, k2, top_k, top_p);
}

}  // namespace

bool filter_supported(int V) { return V >= 1 && V <= 8 * kFThreads * 64; }

cudaError_t launch_filter(const float* in, float* out, int rows, int V, float T, int top_k,
                          float top_p, int num_sms, cudaStream_t s) {
  const float k2 = (float)(1.4426950408889634 / (double)T);  // log2(e) / T
  // the fewest elements per thread (16, 32, 64) that a cluster of at most 8 CTAs covers
  const long long per16 = (long long)kFThreads * 16;
  if (V <= 8 * per16) {
    const long long cl = (V + per16 - 1) / per16;
    // more rows than one wave of two CTAs per SM: half the CTAs per row with twice the elements
    // per thread (each row's chain is longer, but there are half as many waves: 3 840 rows of
    // 32 000 took 754 us this way against 958 us)
    if (cl >= 2 && (long long)rows * cl > 2ll * num_sms) {
      if (cl <= 2) return launch_fk<1, 32>(in, out, rows, V, k2, top_k, top_p, s);
      if (cl <= 4) return launch_fk<2, 32>(in, out, rows, V, k2, top_k, top_p, s);
      return launch_fk<4, 32>(in, out, rows, V, k2, top_k, top_p, s);
    }
    if (cl <= 1) return launch_fk<1, 16>(in, out, rows, V, k2, top_k, top_p, s);
    if (cl <= 2) return launch_fk<2, 16>(in, out, rows, V, k2, top_k, top_p, s);
    if (cl <= 4) return launch_fk<4, 16>(in, out, rows, V, k2, top_k, top_p, s);
    return launch_fk<8, 16>(in, out, rows, V, k2, top_k, top_p, s);
  }
  if (V <= 16 * per16) return launch_fk<8, 32>(in, out, rows, V, k2, top_k, top_p, s);
  if (filter_supported(V)) return launch_fk<8, 64>(in, out, rows, V, k2, top_k, top_p, s);
  return cudaErrorInvalidValue;
}

}  // namespace spectree
