// Tree-masked split-KV attention for draft-tree verification (sm_103a).
//
// Method: EAGLE paper explainer, "Static tree" section -- the target model verifies every path of
// the draft tree in one forward pass under a tree attention mask; speculative-decoding survey
// explainer, taxonomy "Token Tree verification".  Node i of sequence b attends to prefix slots
// 0..L_b-1 and to the slots L_b + j of its ancestors j (itself included).
//
// Decomposition.  The query rows of one (sequence, KV head) are the tree nodes x the g query heads
// sharing that KV head (row = i * g + h, R = N * g rows).  One CTA handles a block of 128 MMA rows
// over one split of the key range; the splits of a (sequence, KV head, row block) form one
// thread-block cluster and combine their partial results on chip at the end.
//
// Key groups.  A tcgen05 MMA always computes 128 rows.  When R <= 64 (multi-head attention over a
// tree of up to 64 nodes) MMA rows 64..127 repeat query rows 0..63: rows 0..63 take keys 0..63 of
// every 128-key chunk and rows 64..127 keys 64..127, so every TMEM lane quadrant (and so every SM
// sub-partition) does softmax work, and rows r and r + 64 end with partial results over disjoint
// key sets that the final combine merges like two more splits.
//
// Warp roles (320 threads, one CTA per SM):
//   warp 0       TMA producer: K/V chunks of 128 keys into a 3-slot ring (192 KB at D = 128: one
//                chunk's K and V per slot), 128-byte swizzled boxes; a split's first chunks are
//                requested right after the set-up barrier, before the prefix length is known;
//   warp 1       allocates 512 TMEM columns; one lane issues the MMAs as soon as their inputs are
//                ready (a non-blocking state machine over the mbarriers):
//                  S = Q K_c^T   (M = 128, N = 128 keys, K = D; Q and K from shared memory)
//                  O += P_c V_c  (M = 128, N = D, K = 128 keys; P from TMEM, V from shared memory)
//                with completions signalled by tcgen05.commit on mbarriers;
//   warps 2..9   softmax, one MMA row (= TMEM lane) per thread and two warps per lane quadrant:
//                key set 0 (warps 2..5) takes the first 32 keys of each 64-key half of a chunk,
//                key set 1 (warps 6..9) the second 32, each with its own running max, sum and O
//                accumulator in TMEM (O[0] at column 256, O[1] at 384), so the two warps of a row
//                never exchange anything in the main loop.  Mask from the node's visibility bits
//                (prefix, then the ancestors' tree slots), online softmax in the log2 domain, P as
//                bf16 pairs written over the scores it came from.  The reference max is only raised
//                when a chunk's max exceeds it by more than 8 (2^8 headroom in fp32); only then is
//                that key set's O in TMEM rescaled.
//   The ring's slots fill and drain by halves: a chunk's K half is refilled once its scores are
//   read, its V half once its PV completed.
// Combine.  A query's partials inside the CTA (2 key sets, and with key groups the rows r and
// r + 64) merge with one named barrier; each merged row's unnormalised O (as bf16), max m and sum
// l then go into the shared memory of the cluster CTA that owns the row (row % splits) through
// distributed-shared-memory stores; the owner weights the S partials by 2^(m - M) / sum(l 2^(m - M))
// in fp32 and writes the bf16 output and the log-sum-exp.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace spectree {

constexpr int kChunkKeys = 128;  // keys per K/V chunk: one ring slot, one pipeline step
constexpr int kMaxSplits = 8;  // portable cluster size

struct AttnKParams {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* lse;
  const int32_t* prefix_lens;
  const int32_t* parent;
  int32_t* status;
  int B, N, Hq, Hkv, g, R, Lmax;
  int kg;  // key groups per MMA row block: 2 when R <= 64, else 1
  int row_blocks, splits, tiles_per_split, tiles_total;
  float scale_log2;  // softmax_scale * log2(e)
  // paged cache (page_size > 0): slot s of sequence b in page block_table[b * max_pages + s / P],
  // row s % P, pages [num_pages][Hkv][P][D]; 0: contiguous [B][Hkv][Lmax][D]
  int page_size, max_pages, num_pages;
  const int32_t* block_table;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// byte offset of (row, 16-byte chunk) inside a 128-byte-swizzled box
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return uint32_t(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// V rows of a chunk are stored in the order the PV MMAs consume them: 32-key blocks 0, 2, 1, 3
// (so that P of keys 0..31, 64..95, 32..63, 96..127 sits in TMEM columns 0, 16, 32, 48).  The map
// is its own inverse: V row block j holds key block v_block_key(j), key block b sits in row block
// v_block_key(b).
__host__ __device__ constexpr int v_block_key(int j) { return ((j & 1) << 1) | (j >> 1); }

__device__ __forceinline__ float ex2_approx(float x) {  // hardware 2^x (P is rounded to bf16)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {  // one three-input max
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (a0, a1) * m + c on the packed fp32 pipe (two lanes of one instruction, each rounded as fmaf)
__device__ __forceinline__ void ffma2(float& a0, float& a1, float m, float c) {
  uint64_t a, mm, cc;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(mm) : "f"(m));
  asm("mov.b64 %0, {%1, %1};" : "=l"(cc) : "f"(c));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(a) : "l"(a), "l"(mm), "l"(cc));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a));
}

// (s0, s1) += (a0, a1) on the packed fp32 pipe
__device__ __forceinline__ void fadd2(float& s0, float& s1, float a0, float a1) {
  uint64_t s, a;
  asm("mov.b64 %0, {%1, %2};" : "=l"(s) : "f"(s0), "f"(s1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(s) : "l"(s), "l"(a));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(s));
}

__device__ __forceinline__ void tmem_ldq(uint32_t taddr, float (&v)[32]) { tmem_ld32(taddr, v); }
__device__ __forceinline__ void tmem_ldq(uint32_t taddr, float (&v)[16]) { tmem_ld16(taddr, v); }

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int D>
struct TcCfg {
  static constexpr int NB = D / 64;               // 64-dim swizzle boxes per row
  static constexpr int KEYS = kChunkKeys;         // keys per chunk
  static constexpr int BOX = KEYS * 128;          // [128 keys x 64 dims] bf16 box: 16 KB
  static constexpr int TILE = 2 * NB * BOX;       // K + V of one chunk
  static constexpr int RING = 192 * 1024;         // K/V ring
  static constexpr int SLOTS = RING / TILE;       // 3 (D = 128) or 6 (D = 64) chunks
  static constexpr int QBOX = 128 * 128;          // [128 rows x 64 dims] bf16: 16 KB
  static constexpr int OFF_Q = RING;
  static constexpr int OFF_BAR = OFF_Q + NB * QBOX;
  static constexpr int SMEM = 1024 /*alignment slack*/ + OFF_BAR + 512;
  // TMEM columns: S[0] 0..127, S[1] 128..255 (one chunk each: 128 keys in fp32); P of a chunk
  // overwrites columns 0..63 of its S buffer (128 bf16 keys packed in pairs, in the V row order:
  // keys 0..31, 64..95, 32..63, 96..127 in columns 0, 16, 32, 48); O[key set] at 256 + 128 ks
  // (the two softmax warp sets each accumulate their own keys).
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t S_COLS = 128;
  static constexpr uint32_t O_COL = 256;
  static constexpr int THREADS = 320;
  static constexpr int RSTRIDE = D + 4;           // floats per exchanged row (padding: no bank clash)
  static constexpr int STAGE_OFF = RING / 2;      // in-CTA key-group exchange, after the combine
                                                  // receive area
};
// One CTA per SM: a second CTA on the SM would block in its 512-column TMEM allocation while the
// first may be waiting for it at a cluster barrier.  More than half the SM's shared memory each
// rules that out.
static_assert(TcCfg<128>::SMEM > 116 * 1024 && TcCfg<64>::SMEM > 116 * 1024, "one CTA per SM");

// Rows of one key group that one CTA of the cluster owns in the final combine.
__host__ __device__ inline int owned_rows(int kg, int splits) {
  return (128 / kg + splits - 1) / splits;
}

// PAGED: the cache is paged (p.page_size > 0); a separate instantiation so that the contiguous
// kernel carries none of the page-table code.  KG: the key groups per 128-row block (2 when a
// head has at most 64 query rows, else 1), also a separate instantiation: each kernel then holds
// one code path for the softmax and the combine (measured 11.2 against 11.8 us a call for the
// 60-node tree on 32 heads of 128 with one kernel for both).
template <int D, bool PAGED, int KG>
__global__ void __launch_bounds__(320, 1) tree_attn_kernel(
    const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
    const AttnKParams p) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int par_s[kMaxNodes];
  __shared__ unsigned long long anc_s[kMaxNodes];
  __shared__ int abort_s;
  __shared__ int bad_s;  // SPEC_ST_BAD_TREE / SPEC_ST_BAD_LEN found in the set-up
  __shared__ uint32_t tmem_s;

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = base;
  uint8_t* q_s = base + C::OFF_Q;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::OFF_BAR);
  // A slot's K and V halves fill and drain separately.  B_FULL: its K landed; B_VFULL: its V
  // landed (a chunk's QK needs only K); B_KEMPTY: the QK that read its K completed (a softmax warp
  // arrives once it sees the scores); B_VEMPTY: the PV that read its V completed (also how the
  // softmax warps learn that a chunk's PV is done).  A chunk holds its K for the QK only, so the
  // next K request into the slot goes out while the softmax of the chunk still runs.
  const int B_FULL = 0, B_VEMPTY = C::SLOTS, B_SFULL = 2 * C::SLOTS,
            B_PFULL = 2 * C::SLOTS + 4, B_DONE = 2 * C::SLOTS + 7,
            B_SETUP = 2 * C::SLOTS + 8, B_VFULL = 2 * C::SLOTS + 9, B_KEMPTY = 3 * C::SLOTS + 9;
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x;  // == rank in the cluster (cluster dims = (splits, 1, 1))
  const int kvh = blockIdx.y / p.row_blocks, rb = blockIdx.y % p.row_blocks;
  const int b = blockIdx.z;
  constexpr int kg = KG;
  const int N = p.N, g = p.g, S = p.splits;

  // ---- set-up, with the first K/V tiles in flight as early as possible
  const int tps = p.tiles_per_split;
  const int t_begin = split * tps;
  const int row0 = PAGED ? 0 : (b * p.Hkv + kvh) * p.Lmax;  // contiguous cache
  const int spec = max(0, min(C::SLOTS, min(tps, p.tiles_total - t_begin)));  // before L is known
  if (tid == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  griddep_wait();  // every global access below may depend on the preceding kernel in the stream
  if (tid == 0) {
    for (int i = 0; i < C::SLOTS; ++i) {
      mbar_init(bar(B_FULL + i), 1);
      mbar_init(bar(B_VFULL + i), 1);
      mbar_init(bar(B_VEMPTY + i), 1);
      mbar_init(bar(B_KEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {  // [S / P buffer]
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_PFULL + i), 8);
    }
    mbar_init(bar(B_DONE), 1);
    mbar_init(bar(B_SETUP), 1);
    mbar_fence_init();
    abort_s = 0;
    bad_s = 0;
  }
  // The small inputs go out first: requests issued after a split's K/V stream wait behind it.
  // Q: the CTA's distinct query rows (64 with key groups, else 128), two rows per warp instruction
  // (coalesced); rows past R are zeros.
  constexpr int QCH = D / 8;  // 16-byte chunks per row
  constexpr int QIT = 128 * QCH / 256;  // per softmax thread
  const int qrows = 128 / kg;
  uint4 qv[QIT];
  if (warp >= 2) {
#pragma unroll
    for (int k = 0; k < QIT; ++k) {
      const int idx = (tid - 64) + k * 256, row = idx / QCH, ch = idx % QCH;
      const int qrow = rb * 128 + row;
      qv[k] = make_uint4(0, 0, 0, 0);
      if (row < qrows && qrow < p.R) {
        const int i = qrow / g, hl = qrow % g;
        qv[k] = __ldg(reinterpret_cast<const uint4*>(
                          p.q + (((size_t)b * N + i) * p.Hq + kvh * g + hl) * D) + ch);
      }
    }
  }
  int parent_i = 0;
  if (tid >= 64 && tid < 64 + N) parent_i = __ldg(p.parent + (size_t)b * N + (tid - 64));
  const int L = __ldg(p.prefix_lens + b);
  __syncthreads();  // the barriers are initialised; the small loads are on their way
  // One chunk (keys 128 ci .. 128 ci + 127 of this sequence and KV head) into ring slot sl; warp 0
  // calls it with every lane.  Contiguous cache: ten boxes (rows of the [B Hkv Lmax, D] view) from
  // lane 0.  Paged cache: up to 32 boxes, one per lane, so that one instruction sends the whole
  // chunk (a copy issued by one thread costs about 100 cycles); `yl` is page_rows(ci) of this
  // lane; an entry outside [0, num_pages) (or past the table) aims its boxes past the tensor,
  // which reads zeros (the set-up flags it when a slot the call needs is there).  K boxes of
  // min(P, 128) rows, V boxes of min(P, 32) rows in the PV block order (see v_block_key).
  const int P = PAGED ? p.page_size : 0;
  const int Pd = PAGED ? p.page_size : 1;   // P as a divisor (the paged code only runs with P > 0)
  const int past = p.num_pages * p.Hkv * P;  // paged: first row past the tensor
  auto page_rows = [&](int ci) -> int {     // lane l: first row of the chunk's l-th page
    int yl = past;
    const int lp0 = (ci * C::KEYS) / Pd;
    if (lane < (P >= C::KEYS ? 1 : C::KEYS / Pd) && lp0 + lane < p.max_pages) {
      const int pg = __ldg(p.block_table + (size_t)b * p.max_pages + lp0 + lane);
      if (pg >= 0 && pg < p.num_pages) yl = (pg * p.Hkv + kvh) * P;
    }
    return yl;
  };
  // One half of a chunk into ring slot sl: its K boxes (completing on B_FULL) or its V boxes
  // (on B_VFULL).  Warp 0 calls it with every lane.
  auto issue_half = [&](int sl, int ci, int yl, bool v) {
    uint8_t* st = ring + sl * C::TILE;
    const uint32_t fb = bar((v ? B_VFULL : B_FULL) + sl);
    if (lane == 0) mbar_arrive_expect_tx(fb, C::TILE / 2);
    if (P == 0) {  // contiguous: issued by one lane (measured faster than spread over lanes)
      if (lane == 0) {
        const int y = row0 + ci * C::KEYS;
        if (!v) {
#pragma unroll
          for (int bx = 0; bx < C::NB; ++bx)
            tma_load_2d(smem_u32(st + bx * C::BOX), &tmap_k, fb, bx * 64, y);
        } else {
#pragma unroll
          for (int bx = 0; bx < C::NB; ++bx)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_load_2d(smem_u32(st + (C::NB + bx) * C::BOX + j * 32 * 128), &tmap_v, fb,
                          bx * 64, y + 32 * v_block_key(j));
        }
      }
      return;
    }
    __syncwarp();
    const int rows = v ? ((P >= 32) ? 32 : P) : ((P >= C::KEYS) ? C::KEYS : P);  // box rows
    const int per = C::KEYS / rows;  // boxes per 64-dim block
    const int nbox = C::NB * per;    // <= 32: one box per lane
    const int ln = lane < nbox ? lane : 0;
    const int i = ln % per, bx = ln / per;
    int key = ci * C::KEYS, dst;
    if (!v) {
      key += i * rows;
      dst = bx * C::BOX + i * rows * 128;
    } else {
      const int j = (i * rows) >> 5, t = (i * rows) & 31;  // V row block j, row t in it
      key += 32 * v_block_key(j) + t;
      dst = (C::NB + bx) * C::BOX + (32 * j + t) * 128;
    }
    int y = __shfl_sync(0xffffffffu, yl, key / Pd - (ci * C::KEYS) / Pd);
    y = y >= past ? past : y + key % Pd;
    if (lane < nbox) tma_load_2d(smem_u32(st + dst), v ? &tmap_v : &tmap_k, fb, bx * 64, y);
  };
  auto issue_chunk = [&](int sl, int ci, int yl) {
    issue_half(sl, ci, yl, false);
    issue_half(sl, ci, yl, true);
  };
  if (warp == 0) {
    // the split's first chunks do not depend on the prefix length: issue them now (a chunk past
    // L_b + N is simply not consumed).  Nothing else waits for this issue.  Paged: every page
    // entry first (independent loads), then the copies.
    if constexpr (PAGED) {
      int yl[C::SLOTS];
#pragma unroll
      for (int it = 0; it < C::SLOTS; ++it) yl[it] = it < spec ? page_rows(t_begin + it) : 0;
#pragma unroll
      for (int it = 0; it < C::SLOTS; ++it)
        if (it < spec) issue_chunk(it, t_begin + it, yl[it]);
    } else {
      for (int it = 0; it < spec; ++it) issue_chunk(it, t_begin + it, 0);
    }
  }
  if (warp == 1) tmem_alloc(smem_u32(&tmem_s), C::TMEM_COLS);

  // softmax threads: MMA row r (TMEM lane r), key group gi, query row qrow of this KV head
  const int r = 32 * (warp & 3) + lane;
  const int ks = (warp - 2) >> 2;  // softmax warps: key set (the first or second 32 keys of a half)
  const int gi = (kg == 2) ? (r >> 6) : 0;
  const int qloc = (kg == 2) ? (r & 63) : r;  // row within this CTA's block of query rows
  const int qrow = rb * 128 + qloc;
  const bool live = qrow < p.R;
  if (warp >= 2) {
    if (tid < 64 + N) par_s[tid - 64] = parent_i;
    // Q rows -> swizzled shared memory (key groups: rows r and r + 64 alike)
#pragma unroll
    for (int k = 0; k < QIT; ++k) {
      const int idx = (tid - 64) + k * 256, row = idx / QCH, ch = idx % QCH;
      if (row < qrows) {
        *reinterpret_cast<uint4*>(q_s + (ch >> 3) * C::QBOX + swz(row, ch & 7)) = qv[k];
        if (kg == 2)
          *reinterpret_cast<uint4*>(q_s + (ch >> 3) * C::QBOX + swz(row + 64, ch & 7)) = qv[k];
      }
    }
    fence_async_smem();  // Q is read by the tensor cores (async proxy)
  }
  if (warp >= 1) {  // warp 0 may still be issuing copies: it learns the outcome from B_SETUP
    named_bar_sync(2, 288);
    // tree: every node validates its own parent and walks its ancestor chain (in parallel)
    if (tid >= 64 && tid < 64 + N) {
      const int i = tid - 64;
      const int pi = par_s[i];
      if (i == 0 ? pi != -1 : (pi < 0 || pi >= i)) atomicOr(&bad_s, SPEC_ST_BAD_TREE);
      unsigned long long m = 1ull << i;
      int k = pi;
      for (int steps = 0; k >= 0 && k < N && steps < N; ++steps) {
        m |= 1ull << k;
        k = par_s[k];
      }
      anc_s[i] = m;
    }
    if (tid == 64 && (L < 0 || L + N > p.Lmax)) atomicOr(&bad_s, SPEC_ST_BAD_LEN);
    if (PAGED && L >= 0 && L + N <= p.Lmax) {
      // paged: every page holding a slot this split reads must be a real page
      const int P = p.page_size;
      const int k_lo = t_begin * C::KEYS, k_hi = min((t_begin + tps) * C::KEYS, L + N);
      if (k_hi > k_lo)
        for (int lp = k_lo / P + (tid - 32); lp <= (k_hi - 1) / P; lp += 288) {
          const int pg = __ldg(p.block_table + (size_t)b * p.max_pages + lp);
          if (pg < 0 || pg >= p.num_pages) atomicOr(&bad_s, SPEC_ST_BAD_PAGE);
        }
    }
    tc_fence_before();
    named_bar_sync(2, 288);
    tc_fence_after();
    if (tid == 64) mbar_arrive(bar(B_SETUP));
  } else if (!mbar_wait(bar(B_SETUP), 0)) {
    abort_s = 1;
  }
  const int bad_bits = bad_s;
  const bool bad = bad_bits != 0;
  if (tid == 64 && bad && p.status &&
      ((bad_bits & SPEC_ST_BAD_PAGE) || (split == 0 && kvh == 0 && rb == 0)))
    atomicOr(p.status + b, bad_bits);
  const uint32_t tmem = tmem_s;

  const int total_keys = bad ? 0 : L + N;
  const int ntiles = (total_keys + C::KEYS - 1) / C::KEYS;
  const int t_end = min(ntiles, t_begin + tps);
  const int my_tiles = max(0, t_end - t_begin);
  const int U = my_tiles;  // pipeline steps: one chunk each

  auto wait = [&](int i, uint32_t parity) -> bool {
    if (abort_s) return false;
    if (mbar_wait(bar(i), parity)) return true;
    abort_s = 1;
    return false;
  };

  float m_used = -INFINITY, l = 0.f;  // softmax threads: running max (log2 units) and sum
  bool ok_rows = true;                // softmax warps: every step completed (no timeout)
  if (warp == 0) {
    // ---------------- TMA producer (the whole warp: it reads block-table entries in parallel).
    // K of chunk kq goes out once the QK of the chunk before it in the slot completed, V of chunk
    // vq once that chunk's PV completed; whichever is ready first.
    int kq = spec, vq = spec;
    int yk = (P > 0 && kq < my_tiles) ? page_rows(t_begin + kq) : 0;  // page rows of chunk kq
    int yv = yk;                                                     // ... and of chunk vq
    uint32_t idle = 0;
    while (vq < my_tiles) {
      bool progressed = false;
      if (kq < my_tiles) {
        const int s = kq % C::SLOTS;
        const uint32_t par = ((kq / C::SLOTS) - 1) & 1;
        if (kq < C::SLOTS || __any_sync(0xffffffffu, mbar_test(bar(B_KEMPTY + s), par))) {
          if (kq >= C::SLOTS) mbar_wait(bar(B_KEMPTY + s), par);  // complete: every lane acquires
          issue_half(s, t_begin + kq, yk, false);
          ++kq;
          if (P > 0 && kq < my_tiles) yk = page_rows(t_begin + kq);
          progressed = true;
        }
      }
      if (vq < kq) {
        const int s = vq % C::SLOTS;
        const uint32_t par = ((vq / C::SLOTS) - 1) & 1;
        if (vq < C::SLOTS || __any_sync(0xffffffffu, mbar_test(bar(B_VEMPTY + s), par))) {
          if (vq >= C::SLOTS) mbar_wait(bar(B_VEMPTY + s), par);
          issue_half(s, t_begin + vq, yv, true);
          ++vq;
          if (P > 0 && vq < my_tiles) yv = page_rows(t_begin + vq);
          progressed = true;
        }
      }
      if (progressed) {
        idle = 0;
      } else if (++idle > kSpinLimit || abort_s) {
        abort_s = 1;
        break;
      } else {
        __nanosleep(20);
      }
    }
    if (lane == 0) {
      // never leave with a copy in flight: speculative tiles nobody consumed, or an abort
      // (bounded waits)
      if (abort_s || my_tiles < spec) {
        for (int it = max(0, kq - C::SLOTS); it < kq; ++it)
          if (abort_s || it >= my_tiles) mbar_wait(bar(B_FULL + it % C::SLOTS), (it / C::SLOTS) & 1);
        for (int it = max(0, vq - C::SLOTS); it < vq; ++it)
          if (abort_s || it >= my_tiles)
            mbar_wait(bar(B_VFULL + it % C::SLOTS), (it / C::SLOTS) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: QK of step u once its K landed and the PV of step u - 2 was
    // issued (that PV reads the P that step u overwrites, and the tensor pipe runs a CTA's MMAs
    // in issue order; its issue also means the softmax is done with S[u % 2]); PV of step u once
    // its P is written (which the softmax signals only after the chunk's V landed).  Whichever is
    // ready goes first, and each probes one barrier: a probe costs the issuer a shared-memory
    // round trip, during which the tensor pipe drains.
    if (lane == 0 && my_tiles > 0) {
      constexpr uint32_t IQK = idesc_bf16_f32(128, C::KEYS, false);
      constexpr uint32_t IPV = idesc_bf16_f32(128, D, true);
      const uint32_t q_addr = smem_u32(q_s);
      int nq = 0, np = 0;
      uint32_t idle = 0;
      while (np < U) {
        bool progressed = false;
        if (nq < U && nq <= np + 1) {
          const int sl = nq % C::SLOTS;
          if (mbar_test(bar(B_FULL + sl), (nq / C::SLOTS) & 1)) {
            tc_fence_after();
            const uint32_t k_addr = smem_u32(ring + sl * C::TILE);
            const uint32_t d = tmem + (uint32_t)((nq & 1) * C::S_COLS);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint64_t ad =
                  smem_desc_sw128(q_addr + (ks >> 2) * C::QBOX + (ks & 3) * 32, 16, 1024);
              const uint64_t bd =
                  smem_desc_sw128(k_addr + (ks >> 2) * C::BOX + (ks & 3) * 32, 16, 1024);
              tc_mma_bf16(d, ad, bd, IQK, ks > 0 ? 1u : 0u);
            }
            tc_commit(bar(B_SFULL + (nq & 1)));
            ++nq;
            progressed = true;
          }
        }
        if (np < nq && mbar_test(bar(B_PFULL + (np & 1)), (np >> 1) & 1)) {
          tc_fence_after();
          const int sl = np % C::SLOTS;
          // V rows 0..63 (keys 0..31, 64..95) belong to key set 0, rows 64..127 to key set 1:
          // each set accumulates into its own O
          const uint32_t p_tm = tmem + (uint32_t)((np & 1) * C::S_COLS);
          const uint32_t v_addr = smem_u32(ring + sl * C::TILE + C::NB * C::BOX);
#pragma unroll
          for (int kk = 0; kk < C::KEYS / 16; ++kk) {
            const uint64_t bd = smem_desc_sw128(v_addr + kk * 2048, C::BOX, 1024);
            tc_mma_bf16_ts(tmem + C::O_COL + (uint32_t)((kk >> 2) * 128), p_tm + (uint32_t)(kk * 8),
                           bd, IPV, (np > 0 || (kk & 3) > 0) ? 1u : 0u);
          }
          tc_commit(bar(B_VEMPTY + sl));  // the slot's V half may be refilled
          ++np;
          progressed = true;
        }
        if (progressed) {
          idle = 0;
        } else if (++idle > kSpinLimit || abort_s) {
          abort_s = 1;
          break;
        } else {
          __nanosleep(20);  // leave the issue slots to the softmax warp of this sub-partition
        }
      }
      tc_commit(bar(B_DONE));  // every MMA issued above has completed once this phase completes
      mbar_wait(bar(B_DONE), 0);
    }
  } else {
    // ---------------- softmax: one MMA row per thread, two warps per row.  Key set ks (warps
    // 2..5: ks = 0, warps 6..9: ks = 1) takes keys 32 ks..32 ks + 31 of each 64-key half of a chunk
    // -- the half gi with key groups, both halves otherwise -- with its own running max, sum and O
    // accumulator, so the two warps of a row never exchange anything.
    const int node = min(qrow / g, N - 1);
    const unsigned long long anc = anc_s[node];
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t o_col = C::O_COL + (uint32_t)(ks * 128);
    const float sc = p.scale_log2;
    const int tg = tid - 64;  // 0..255
    float zero16[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) zero16[c] = 0.f;
    // visibility of the 32 keys key0..key0+31 (bit c: key key0 + c): the prefix part, then the
    // tree slots L + j of the node's ancestors j.  One code path for every chunk.
    auto visible32 = [&](int key0) -> uint32_t {
      const int pre = L - key0;
      unsigned long long vis = pre >= 64 ? ~0ull : (pre <= 0 ? 0ull : (1ull << pre) - 1ull);
      const int j0 = key0 - L;
      if (j0 > -64 && j0 < N) vis |= j0 >= 0 ? (anc >> j0) : (anc << -j0);
      return (uint32_t)vis;
    };
    for (int u = 0; u < U; ++u) {
      if (!__all_sync(0xffffffffu, wait(B_SFULL + (u & 1), (u >> 1) & 1))) {
        ok_rows = false;
        break;
      }
      tc_fence_after();
      // the QK of this chunk completed: its K half of the slot may be refilled (one commit less
      // for the MMA issuer, whose every instruction delays the next MMA)
      if (warp == 2 && lane == 0) mbar_arrive(bar(B_KEMPTY + u % C::SLOTS));
      const int ckey0 = (t_begin + u) * C::KEYS;
      const uint32_t scol0 = (uint32_t)((u & 1) * C::S_COLS);
      // this thread's 32-key blocks: half hf = gi (key groups) or 0 and 1; S columns
      // 64 hf + 32 ks, P columns 32 ks + 16 hf (inside the S columns this warp has read)
      constexpr int NH = (kg == 2) ? 1 : 2;
      float x[NH][32];
#pragma unroll
      for (int hh = 0; hh < NH; ++hh)
        tmem_ld32(lane_base + scol0 + (uint32_t)(64 * ((kg == 2) ? gi : hh) + 32 * ks), x[hh]);
      tmem_wait_ld();
      float mx = -INFINITY;
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) {
        const uint32_t vis = visible32(ckey0 + 64 * ((kg == 2) ? gi : hh) + 32 * ks);
        if (vis != 0xffffffffu) {  // only blocks at the end of the prefix or in the tree
#pragma unroll
          for (int c = 0; c < 32; ++c) x[hh][c] = ((vis >> c) & 1u) ? x[hh][c] : -INFINITY;
        }
        float m0 = max3f(x[hh][0], x[hh][1], x[hh][2]), m1 = max3f(x[hh][3], x[hh][4], x[hh][5]);
#pragma unroll
        for (int c = 6; c < 30; c += 4) {
          m0 = max3f(m0, x[hh][c], x[hh][c + 1]);
          m1 = max3f(m1, x[hh][c + 2], x[hh][c + 3]);
        }
        mx = max3f(mx, max3f(m0, x[hh][30], x[hh][31]), m1);
      }
      const float mt = mx * sc;  // scale > 0
      const bool raise = mt > m_used + 8.f;
      float factor = 1.f;
      if (raise) {
        factor = (m_used == -INFINITY) ? 0.f : ex2_approx(m_used - mt);
        m_used = mt;
      }
      const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
      float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) {
        const int hf = (kg == 2) ? gi : hh;
        float pk[16];  // P as bf16 pairs (bit patterns), key 2c in the low half of column c
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          float a0 = x[hh][2 * c], a1 = x[hh][2 * c + 1];
          ffma2(a0, a1, sc, neg_m);
          a0 = ex2_approx(a0);
          a1 = ex2_approx(a1);
          if (c & 1) fadd2(r2, r3, a0, a1); else fadd2(r0, r1, a0, a1);
          pk[c] = __uint_as_float(pack_bf16(a0, a1));
        }
        tmem_st16(lane_base + scol0 + (uint32_t)(32 * ks + 16 * hf), pk);
      }
      const float rs = (r0 + r1) + (r2 + r3);
      // key groups: the other group's P columns of this set are zero for this row
      if (kg == 2) tmem_st16(lane_base + scol0 + (uint32_t)(32 * ks + 16 * (1 - gi)), zero16);
      l = l * factor + rs;
      // The chunk holding the last key L + N - 1: V rows past it hold whatever the cache holds
      // there (possibly NaN); their P is 0, but 0 * NaN is not, so zero those rows.
      if (ckey0 + C::KEYS > total_keys) {
        const int sl = u % C::SLOTS;
        if (__all_sync(0xffffffffu, wait(B_VFULL + sl, (u / C::SLOTS) & 1))) {
          const int nv = total_keys - ckey0;  // 1..127 valid keys
          const int units = C::NB * (C::KEYS - nv) * 8;
          for (int w = tg; w < units; w += 256) {
            const int bx = w / ((C::KEYS - nv) * 8), rem = w % ((C::KEYS - nv) * 8);
            const int key = nv + rem / 8, vrow = 32 * v_block_key(key >> 5) + (key & 31);
            *reinterpret_cast<uint4*>(ring + sl * C::TILE + (C::NB + bx) * C::BOX + vrow * 128 +
                                      (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_async_smem();  // the zeros are read by the tensor cores (async proxy)
        }
      }
      // O rescale (only after the first step, only if some row of this warp raised its max)
      if (u > 0 && __any_sync(0xffffffffu, raise)) {
        const int up = u - 1;  // its PV completed: O holds every earlier chunk
        if (__all_sync(0xffffffffu, wait(B_VEMPTY + up % C::SLOTS, (up / C::SLOTS) & 1))) {
          tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            float o[32];
            tmem_ld32(lane_base + o_col + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] *= factor;
            tmem_st32(lane_base + o_col + c0, o);
          }
        }
      }
      tmem_wait_st();  // P (and a rescaled O) are in TMEM before the PV MMA reads them
      tc_fence_before();
      __syncwarp();
      // P is written and the scores read; the chunk's V has landed too, so that the MMA issuer
      // probes this one barrier before the PV (the QK of step u + 2, which overwrites S[u % 2],
      // follows that PV)
      if (!__all_sync(0xffffffffu, wait(B_VFULL + u % C::SLOTS, (u / C::SLOTS) & 1))) {
        ok_rows = false;
        break;
      }
      if (lane == 0) mbar_arrive(bar(B_PFULL + (u & 1)));
    }
    if (ok_rows && U > 0) {  // the last PV completed
      const int ul = U - 1;
      ok_rows = __all_sync(0xffffffffu, wait(B_VEMPTY + ul % C::SLOTS, (ul / C::SLOTS) & 1));
    }
    if (ok_rows && U > 0) tc_fence_after();
  }

  // The next kernel in the stream may start launching now: signalled at the start, its CTAs
  // would sit on SMs (holding their shared memory) while this kernel still runs, and the two
  // kernels of a verification step measured 1.8 us slower per step that way.
  griddep_launch_dependents();
  // ---------------- combine across the cluster (all threads of every CTA take part)
  // A query's partials inside the CTA -- the two accumulators (key sets 0 and 1) of its lane and,
  // with key groups, of lane r + 64 too (the same query over different keys) -- merge into one,
  // which goes to the cluster CTA that owns the row.  Partial: (m, l, O) with m = NaN after a
  // timeout and l = 0 when it saw no key (its O is then never read).
  const int QO = owned_rows(kg, S);
  // [S][QO][RSTRIDE floats] partial rows, then one trash row that rows without data are pushed into
  // (so the push has no branch), then the (m, l) pairs [S][QO].  The ring is idle now.  A partial
  // row travels as bf16 in the first half of its slot: unnormalised O keeps fp32's exponent range,
  // and half the bytes cross the cluster (measured rel-L2 against the oracle 2.8e-3 against 2.2e-3
  // with fp32 partials for the 60-node tree on 32 heads of 128; the output is bf16 anyway).
  float* recv_o = reinterpret_cast<float*>(ring);
  float2* recv_ml = reinterpret_cast<float2*>(recv_o + ((size_t)S * QO + 1) * C::RSTRIDE);
  // in-CTA exchange: the (m, l) of every (key set, lane) [2][128], then the raw accumulator
  // values a lane hands to the other key group, [2 accumulators][64 rows][RSTRIDE]
  float2* stage_ml = reinterpret_cast<float2*>(ring + C::STAGE_OFF);
  float* stage_o = reinterpret_cast<float*>(stage_ml + 256);
  const float m_own = ok_rows ? (l > 0.f ? m_used : -INFINITY) : NAN;
  const float l_own = (ok_rows && l > 0.f) ? l : 0.f;
  // Split barrier: this CTA's ring is free for the peers' pushes once every thread arrived (TMA
  // copies drained, MMAs complete); the in-CTA merge below only touches this CTA's own memory, so
  // it runs while the slower CTAs arrive, and each thread waits just before its first remote store.
  // One split (S == 1): no peer, no push, no owner pass -- each thread normalises its merged piece
  // of the row and writes it (the owner pass of a single partial gives the same bits).
  const bool single = S == 1;
  if (!single) cluster_arrive_release();
  __syncthreads();  // this CTA: the producer drained its copies and the MMAs completed
  if (!single && warp < 2) cluster_wait_acquire();
  // row q = rb * 128 + qloc of this block: node i = q / g, query head kvh * g + q % g
  auto out_row = [&](int qrow_) -> __nv_bfloat16* {
    return p.out + (((size_t)b * N + qrow_ / g) * p.Hq + kvh * g + qrow_ % g) * D;
  };
  auto put_lse = [&](int qrow_, bool tmo_, bool has_, float m_, float lsum_) {
    if (p.lse)
      p.lse[((size_t)b * p.Hq + kvh * g + qrow_ % g) * N + qrow_ / g] =
          has_ ? (m_ + __log2f(lsum_)) * 0.69314718055994531f : -INFINITY;
    if (tmo_ && p.status) atomicOr(p.status + b, SPEC_ST_TIMEOUT);
  };
  if (warp >= 2) {
    const uint32_t lane_tm = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const int owner = qloc % S, ql = qloc / S;
    stage_ml[ks * 128 + r] = make_float2(m_own, l_own);
    auto sel = [](float w, float v) { return w != 0.f ? w * v : 0.f; };  // v may be garbage
    auto push_ml = [&](bool tmo, bool has, float m, float lsum) {
      dsmem_store_v2(dsmem_addr(recv_ml + (size_t)split * QO + ql, owner),
                     __float_as_uint(tmo ? NAN : (has ? m : -INFINITY)),
                     __float_as_uint(has ? lsum : 0.f));
    };
    if (kg == 2) {
      // Query qloc has four partials: (key group g, key set k) = lane 64 g + qloc, accumulator k.
      // The thread of (g, k) combines columns quarter 2 g + k of all four and pushes them; it
      // hands its lane's raw values of quarter 2 (1 - g) + k to the other group first.  One
      // barrier covers the states and the hand-over.
      constexpr int Q4 = D / 4;
      const int my_c = (2 * gi + ks) * Q4, give_c = (2 * (1 - gi) + ks) * Q4;
      {
        float g0[Q4], g1[Q4];
        tmem_ldq(lane_tm + C::O_COL + (uint32_t)give_c, g0);
        tmem_ldq(lane_tm + C::O_COL + 128u + (uint32_t)give_c, g1);
        tmem_wait_ld();
        float* s0 = stage_o + qloc * C::RSTRIDE + give_c;
        float* s1 = stage_o + (64 + qloc) * C::RSTRIDE + give_c;
#pragma unroll
        for (int k = 0; k < Q4; k += 4) {
          *reinterpret_cast<float4*>(s0 + k) = make_float4(g0[k], g0[k + 1], g0[k + 2], g0[k + 3]);
          *reinterpret_cast<float4*>(s1 + k) = make_float4(g1[k], g1[k + 1], g1[k + 2], g1[k + 3]);
        }
      }
      float o0[Q4], o1[Q4];
      tmem_ldq(lane_tm + C::O_COL + (uint32_t)my_c, o0);  // in flight across the barrier
      tmem_ldq(lane_tm + C::O_COL + 128u + (uint32_t)my_c, o1);
      named_bar_sync(1, 256);  // the eight softmax warps
      float2 st[2][2];         // [group][key set]
#pragma unroll
      for (int g2 = 0; g2 < 2; ++g2)
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) st[g2][k2] = stage_ml[k2 * 128 + g2 * 64 + qloc];
      bool tmo = false;
      float M = -INFINITY;
#pragma unroll
      for (int g2 = 0; g2 < 2; ++g2)
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
          tmo |= isnan(st[g2][k2].x);
          M = st[g2][k2].y > 0.f ? fmaxf(M, st[g2][k2].x) : M;
        }
      float w[2][2], Lsum = 0.f;
#pragma unroll
      for (int g2 = 0; g2 < 2; ++g2)
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
          w[g2][k2] = st[g2][k2].y > 0.f ? ex2_approx(st[g2][k2].x - M) : 0.f;
          Lsum = fmaf(w[g2][k2], st[g2][k2].y, Lsum);
        }
      const bool has = !tmo && Lsum > 0.f;
      const float* r0 = stage_o + qloc * C::RSTRIDE + my_c;
      const float* r1 = stage_o + (64 + qloc) * C::RSTRIDE + my_c;
      const float wo0 = gi ? w[1][0] : w[0][0], wo1 = gi ? w[1][1] : w[0][1];  // own lane
      const float wx0 = gi ? w[0][0] : w[1][0], wx1 = gi ? w[0][1] : w[1][1];  // the other lane
      auto merged4 = [&](int k, float (&v)[4]) {  // columns my_c + k .. + 3 of the merged row
        const float4 x0 = *reinterpret_cast<const float4*>(r0 + k);
        const float4 x1 = *reinterpret_cast<const float4*>(r1 + k);
        const float xa[4] = {x0.x, x0.y, x0.z, x0.w}, xb[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          v[j] = sel(wo0, o0[k + j]) + sel(wo1, o1[k + j]) + sel(wx0, xa[j]) + sel(wx1, xb[j]);
      };
      if (single) {
        tmem_wait_ld();
        if (live) {
          const float inv = has ? __frcp_rn(Lsum) : 0.f;
          __nv_bfloat16* orow = out_row(qrow) + my_c;
#pragma unroll
          for (int k = 0; k < Q4; k += 8) {
            float a[4], c4[4];
            merged4(k, a);
            merged4(k + 4, c4);
            *reinterpret_cast<uint4*>(orow + k) =
                make_uint4(pack_bf16(a[0] * inv, a[1] * inv), pack_bf16(a[2] * inv, a[3] * inv),
                           pack_bf16(c4[0] * inv, c4[1] * inv), pack_bf16(c4[2] * inv, c4[3] * inv));
          }
          if (gi == 0 && ks == 0) put_lse(qrow, tmo, has, M, Lsum);
        }
      } else {
        cluster_wait_acquire();  // every CTA's ring is free: the pushes may start
        if (live && gi == 0 && ks == 0) push_ml(tmo, has, M, Lsum);
        const size_t row = (live && has) ? (size_t)split * QO + ql : (size_t)S * QO;
        const uint32_t dst =
            dsmem_addr(reinterpret_cast<__nv_bfloat16*>(recv_o + row * C::RSTRIDE) + my_c, owner);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < Q4; k += 8) {
          float v[4], u[4];
          merged4(k, v);
          merged4(k + 4, u);
          dsmem_store_v4(dst + k * 2, make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]),
                                                 pack_bf16(u[0], u[1]), pack_bf16(u[2], u[3])));
        }
      }
    } else {
      // no key groups: the two accumulators of this lane; the thread of key set k pushes half k
      // of the columns, 32 at a time
      named_bar_sync(1, 256);
      const float2 s0 = stage_ml[r], s1 = stage_ml[128 + r];
      const bool tmo = isnan(s0.x) || isnan(s1.x);
      const float M = fmaxf(s0.y > 0.f ? s0.x : -INFINITY, s1.y > 0.f ? s1.x : -INFINITY);
      const float w0 = s0.y > 0.f ? ex2_approx(s0.x - M) : 0.f;
      const float w1 = s1.y > 0.f ? ex2_approx(s1.x - M) : 0.f;
      const float Lsum = s0.y * w0 + s1.y * w1;
      const bool has = !tmo && Lsum > 0.f;
      constexpr int HC = D / 2 < 32 ? D / 2 : 32;
      if (single) {
        const float inv = has ? __frcp_rn(Lsum) : 0.f;
        __nv_bfloat16* orow = out_row(qrow);
#pragma unroll 1
        for (int c0 = ks * (D / 2); c0 < (ks + 1) * (D / 2); c0 += HC) {
          float a0[HC], a1[HC];
          tmem_ldq(lane_tm + C::O_COL + (uint32_t)c0, a0);
          tmem_ldq(lane_tm + C::O_COL + 128u + (uint32_t)c0, a1);
          tmem_wait_ld();
          if (live) {
#pragma unroll
            for (int k = 0; k < HC; k += 8) {
              float v[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) v[j] = (sel(w0, a0[k + j]) + sel(w1, a1[k + j])) * inv;
              *reinterpret_cast<uint4*>(orow + c0 + k) =
                  make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                             pack_bf16(v[6], v[7]));
            }
          }
        }
        if (live && ks == 0) put_lse(qrow, tmo, has, M, Lsum);
      } else {
        cluster_wait_acquire();  // every CTA's ring is free: the pushes may start
        if (live && ks == 0) push_ml(tmo, has, M, Lsum);
        const size_t row = (live && has) ? (size_t)split * QO + ql : (size_t)S * QO;
        const uint32_t dst = dsmem_addr(recv_o + row * C::RSTRIDE, owner);
#pragma unroll 1
        for (int c0 = ks * (D / 2); c0 < (ks + 1) * (D / 2); c0 += HC) {
          float a0[HC], a1[HC];
          tmem_ldq(lane_tm + C::O_COL + (uint32_t)c0, a0);
          tmem_ldq(lane_tm + C::O_COL + 128u + (uint32_t)c0, a1);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < HC; k += 8) {
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = sel(w0, a0[k + j]) + sel(w1, a1[k + j]);
            dsmem_store_v4(dst + (c0 + k) * 2,
                           make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]),
                                      pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7])));
          }
        }
      }
    }
  }
  if (!single) {
    tc_fence_before();  // this thread's TMEM reads are done
    cluster_arrive_release();
    cluster_wait_acquire();
    // nothing reads TMEM any more: free it now rather than at the end
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, C::TMEM_COLS);
    }
  }
  // owner: rows qloc = ql * S + split of this block, 16 output columns per item (one round of
  // items for the 60-node tree on three splits).  out = sum_e 2^(m_e - M) O_e / sum_e 2^(m_e - M)
  // l_e over the row's S partials e (one per split).
  const int E = S;
  constexpr int C16 = D / 16;
  for (int it = tid; !single && it < QO * C16; it += C::THREADS) {
    const int ql = it / C16, c = (it % C16) * 16, ql_loc = ql * S + split;
    const int q = rb * 128 + ql_loc;
    if (ql_loc >= 128 / kg || q >= p.R) continue;
    // one online pass over the partials (selects, no branches in the body)
    float M = -INFINITY, Ls = 0.f;
    float acc[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] = 0.f;
    bool timeout = false;
    for (int e = 0; e < E; ++e) {
      const float2 ml = recv_ml[(size_t)e * QO + ql];
      timeout |= isnan(ml.x);
      const bool has = ml.y > 0.f;  // partials without keys pushed no O row: never read it
      const float mn = has ? fmaxf(M, ml.x) : M;
      const float a = (M == mn) ? 1.f : ex2_approx(M - mn);
      const float w = has ? ex2_approx(ml.x - mn) : 0.f;
      const uint4* src = reinterpret_cast<const uint4*>(
          reinterpret_cast<const __nv_bfloat16*>(recv_o + ((size_t)e * QO + ql) * C::RSTRIDE) + c);
      const uint4 h0 = src[0], h1 = src[1];
      const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float v0 = __uint_as_float(hw[j] << 16), v1 = __uint_as_float(hw[j] & 0xffff0000u);
        acc[2 * j] = fmaf(acc[2 * j], a, has ? w * v0 : 0.f);
        acc[2 * j + 1] = fmaf(acc[2 * j + 1], a, has ? w * v1 : 0.f);
      }
      Ls = fmaf(Ls, a, w * (has ? ml.y : 0.f));
      M = mn;
    }
    const bool row_ok = !timeout && Ls > 0.f;
    const float inv = row_ok ? __frcp_rn(Ls) : 0.f;
    const float Lsum = Ls;
    const int i = q / g, hq = kvh * g + q % g;
    uint4* dst = reinterpret_cast<uint4*>(p.out + (((size_t)b * N + i) * p.Hq + hq) * D + c);
    auto out8 = [&](int k) {  // columns c + k .. c + k + 7, normalised, as bf16
      return make_uint4(pack_bf16(acc[k] * inv, acc[k + 1] * inv),
                        pack_bf16(acc[k + 2] * inv, acc[k + 3] * inv),
                        pack_bf16(acc[k + 4] * inv, acc[k + 5] * inv),
                        pack_bf16(acc[k + 6] * inv, acc[k + 7] * inv));
    };
    dst[0] = out8(0);
    dst[1] = out8(8);
    if (c == 0) {
      if (p.lse)
        p.lse[((size_t)b * p.Hq + hq) * N + i] =
            row_ok ? (M + __log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
      if (timeout && p.status) atomicOr(p.status + b, SPEC_ST_TIMEOUT);
    }
  }
  if (single) {
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, C::TMEM_COLS);
    }
  }
}

// ------------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------------
extern "C" typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                               void*, const cuuint64_t*, const cuuint64_t*,
                                               const cuuint32_t*, const cuuint32_t*,
                                               CUtensorMapInterleave, CUtensorMapSwizzle,
                                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled encode_fn() {
  static PFN_encodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled>(p);
  });
  return fn;
}

static bool make_kv_map(CUtensorMap* m, const void* ptr, int D, long long rows, int box_rows) {
  PFN_encodeTiled fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
static cudaLaunchConfig_t launch_config(int splits, dim3 grid, cudaStream_t s,
                                        cudaLaunchAttribute (&attr)[2]) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = splits;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(TcCfg<D>::THREADS);
  cfg.dynamicSmemBytes = TcCfg<D>::SMEM;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// Opt the kernel into its shared-memory size on the current device (once per device).
template <int D, bool PAGED, int KG>
static cudaError_t prepare_kernel() {
  constexpr int kDev = 64;
  static std::mutex mu;
  static bool done[kDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    e = cudaFuncSetAttribute(tree_attn_kernel<D, PAGED, KG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TcCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

// Clusters of `splits` CTAs that fit on the device at once (0 if the query fails).
template <int D>
static int clusters_per_wave(int splits) {
  constexpr int kDev = 64;
  static std::mutex mu;
  static int cache[kDev][kMaxSplits + 1] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDev) return 0;
  if (prepare_kernel<D, false, 1>() != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev][splits] == 0) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = launch_config<D>(splits, dim3(splits, 1, 1), nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tree_attn_kernel<D, false, 1>, &cfg) != cudaSuccess || n < 1)
      return 0;
    cache[dev][splits] = n;
  }
  return cache[dev][splits];
}

bool attn_plan(int B, int N, int Hq, int Hkv, int D, int Lmax, int num_sms, AttnPlan* plan) {
  if (B < 1 || N < 1 || N > kMaxNodes || Hkv < 1 || Hq < Hkv || Hq % Hkv || Lmax < N) return false;
  if (D != 64 && D != 128) return false;
  const int R = N * (Hq / Hkv);
  plan->kg = R <= 64 ? 2 : 1;
  plan->row_blocks = plan->kg == 2 ? 1 : (R + 127) / 128;
  plan->tiles = (Lmax + kChunkKeys - 1) / kChunkKeys;
  const long long units = (long long)B * Hkv * plan->row_blocks;
  const int sms = num_sms > 0 ? num_sms : 148;
  // cost = waves x (pipeline steps + fixed set-up / combine cost of about three steps)
  int best = 1;
  double best_cost = 1e300;
  for (int s = 1; s <= kMaxSplits && s <= plan->tiles; ++s) {
    const int tps = (plan->tiles + s - 1) / s;
    if ((plan->tiles + tps - 1) / tps != s) continue;  // same split as a smaller s
    const size_t rows = (size_t)s * owned_rows(plan->kg, s);
    const size_t recv = (rows + 1) * (size_t)(D + 4) * 4 + rows * 8;  // + the trash row
    if (recv > (size_t)(D == 128 ? TcCfg<128>::STAGE_OFF : TcCfg<64>::STAGE_OFF)) continue;
    int per_wave = s == 1 ? sms : (D == 128 ? clusters_per_wave<128>(s) : clusters_per_wave<64>(s));
    if (per_wave < 1) per_wave = s == 1 ? sms : sms / (2 * s);  // conservative guess
    if (per_wave < 1) continue;
    const long long waves = (units + per_wave - 1) / per_wave;
    const double cost = (double)waves * (tps + 3.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  plan->splits = best;
  plan->tiles_per_split = (plan->tiles + best - 1) / best;
  plan->ws_bytes = 0;  // the splits are combined on chip
  return true;
}

template <int D, bool PAGED, int KG>
static cudaError_t launch_dk(const CUtensorMap& mk, const CUtensorMap& mv, const AttnKParams& kp,
                            cudaStream_t s) {
  // the combine's receive area and owned-row split assume the portable cluster size at most
  if (kp.splits < 1 || kp.splits > kMaxSplits) return cudaErrorInvalidConfiguration;
  cudaError_t e = prepare_kernel<D, PAGED, KG>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg =
      launch_config<D>(kp.splits, dim3(kp.splits, kp.Hkv * kp.row_blocks, kp.B), s, attr);
  return cudaLaunchKernelEx(&cfg, tree_attn_kernel<D, PAGED, KG>, mk, mv, kp);
}

template <int D, bool PAGED>
static cudaError_t launch_d(const CUtensorMap& mk, const CUtensorMap& mv, const AttnKParams& kp,
                            cudaStream_t s) {
  return kp.kg == 2 ? launch_dk<D, PAGED, 2>(mk, mv, kp, s) : launch_dk<D, PAGED, 1>(mk, mv, kp, s);
}

cudaError_t launch_attention(const AttnArgs& a, const AttnPlan& plan, cudaStream_t s) {
  CUtensorMap mk, mv;
  const int P = a.page_size;
  const long long rows =
      P > 0 ? (long long)a.num_pages * a.Hkv * P : (long long)a.B * a.Hkv * a.Lmax;
  // K in boxes of a whole chunk (or page); V in 32-key boxes (or pages), stored in the PV order
  const int kb = P > 0 && P < kChunkKeys ? P : kChunkKeys, vb = P > 0 && P < 32 ? P : 32;
  if (!make_kv_map(&mk, a.k, a.D, rows, kb) || !make_kv_map(&mv, a.v, a.D, rows, vb))
    return cudaErrorInvalidValue;
  AttnKParams kp;
  kp.q = static_cast<const __nv_bfloat16*>(a.q);
  kp.out = static_cast<__nv_bfloat16*>(a.out);
  kp.lse = a.lse;
  kp.prefix_lens = a.prefix_lens;
  kp.parent = a.parent;
  kp.status = a.status;
  kp.B = a.B;
  kp.N = a.N;
  kp.Hq = a.Hq;
  kp.Hkv = a.Hkv;
  kp.g = a.Hq / a.Hkv;
  kp.R = a.N * kp.g;
  kp.Lmax = a.Lmax;
  kp.kg = plan.kg;
  kp.row_blocks = plan.row_blocks;
  kp.splits = plan.splits;
  kp.tiles_per_split = plan.tiles_per_split;
  kp.tiles_total = plan.tiles;
  kp.scale_log2 = a.scale * 1.4426950408889634f;
  kp.page_size = P;
  kp.max_pages = a.max_pages;
  kp.num_pages = a.num_pages;
  kp.block_table = a.block_table;
  if (P > 0)
    return a.D == 128 ? launch_d<128, true>(mk, mv, kp, s) : launch_d<64, true>(mk, mv, kp, s);
  return a.D == 128 ? launch_d<128, false>(mk, mv, kp, s) : launch_d<64, false>(mk, mv, kp, s);
}

}  // namespace spectree
