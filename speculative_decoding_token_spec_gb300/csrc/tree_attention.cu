// Tree-masked split-KV attention for draft-tree verification (sm_103a).
//
// Method: EAGLE paper explainer, "Static tree" section -- the target model verifies every path of
// the draft tree in one forward pass under a tree attention mask; speculative-decoding survey
// explainer, taxonomy "Token Tree verification".  Node i of sequence b attends to prefix slots
// 0..L_b-1 and to the slots L_b + j of its ancestors j (itself included).
//
// Decomposition (flash-decode style): one CTA per (sequence, KV head, row block, split).  The
// CTA's query rows are the tree nodes x the g query heads sharing the KV head (row = i * g + h).
// K/V tiles of 64 keys stream through a 4-stage TMA ring (128-byte swizzled boxes, one mbarrier per
// stage, bounded waits).  S = Q K^T and O += P V run on the tensor cores (mma.sync bf16 -> fp32);
// the online softmax runs in registers in the log2 domain.  Tiles that reach past the prefix are
// masked with the per-node ancestor bitmask built from the parent array in shared memory.  With
// more than one split the CTA writes unnormalised partials (O, m, l) and a merge kernel combines
// them by log-sum-exp weights.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace spectree {

constexpr int kTileKeys = 64;
constexpr int kStages = 4;
constexpr int kBoxBytes = kTileKeys * 128;  // one 64-key x 64-dim bf16 box

struct AttnKParams {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* lse;
  const int32_t* prefix_lens;
  const int32_t* parent;
  int32_t* status;
  float* part_o;   // [B, Hkv, splits, Rpad, D]
  float2* part_ml; // [B, Hkv, splits, Rpad]  (m in log2 units of scaled scores, l)
  int B, N, Hq, Hkv, g, R, Rpad, Lmax, D;
  int splits, tiles_per_split, row_blocks, tiles_total;
  float scale_log2;  // softmax_scale * log2(e)
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
      " {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// byte offset of (row, 16-byte chunk) inside a 128-byte-swizzled box
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return uint32_t(row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <int D>
__host__ __device__ constexpr int stage_bytes() {
  return 2 * (D / 64) * kBoxBytes;
}

template <int D, int WARPS>
__host__ __device__ constexpr int attn_smem_bytes() {
  return 1024 /*align slack*/ + kStages * stage_bytes<D>() + (D / 64) * (16 * WARPS) * 128 + 64;
}

template <int D, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) tree_attn_kernel(
    const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
    const AttnKParams p) {
  constexpr int ROWS = 16 * WARPS;
  constexpr int NBOX = D / 64;
  constexpr int KSTEPS = D / 16;
  constexpr int DT = D / 8;  // 8-wide output column tiles
  extern __shared__ uint8_t smem_raw[];
  __shared__ int par_s[kMaxNodes];
  __shared__ unsigned long long anc_s[kMaxNodes];
  __shared__ int bad_s;

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* kv_base = base;                                   // kStages x (K boxes, V boxes)
  uint8_t* q_base = base + kStages * stage_bytes<D>();       // NBOX x ROWS x 128 B
  uint64_t* bars = reinterpret_cast<uint64_t*>(q_base + NBOX * ROWS * 128);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y / p.row_blocks, rb = blockIdx.y % p.row_blocks;
  const int b = blockIdx.z;
  const int N = p.N, g = p.g;

  if (tid == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  griddep_wait();  // every global access below may depend on the preceding kernel in the stream
  griddep_launch_dependents();
  if (tid < N) par_s[tid] = __ldg(p.parent + (size_t)b * N + tid);
  const int L = __ldg(p.prefix_lens + b);
  __syncthreads();
  if (tid == 0) {
    int st = build_ancestors(par_s, N, anc_s);
    if (L < 0 || L + N > p.Lmax) st |= SPEC_ST_BAD_LEN;
    bad_s = st;
    if (st && split == 0 && kvh == 0 && rb == 0 && p.status) atomicOr(p.status + b, st);
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(bars + s), 1);
    mbar_fence_init();
  }
  __syncthreads();
  const bool bad = bad_s != 0;

  // this split's tiles
  const int total_keys = bad ? 0 : L + N;
  const int ntiles = (total_keys + kTileKeys - 1) / kTileKeys;
  const int t_begin = split * p.tiles_per_split;
  const int t_end = min(ntiles, t_begin + p.tiles_per_split);
  const int my_tiles = max(0, t_end - t_begin);
  const int row0 = (b * p.Hkv + kvh) * p.Lmax;  // first cache row of this (sequence, KV head)

  auto issue = [&](int it) {
    const int s = it % kStages;
    const uint32_t bar = smem_u32(bars + s);
    uint8_t* st = kv_base + s * stage_bytes<D>();
    mbar_arrive_expect_tx(bar, stage_bytes<D>());
    const int y = row0 + (t_begin + it) * kTileKeys;
#pragma unroll
    for (int bx = 0; bx < NBOX; ++bx) {
      tma_load_2d(smem_u32(st + bx * kBoxBytes), &tmap_k, bar, bx * 64, y);
      tma_load_2d(smem_u32(st + (NBOX + bx) * kBoxBytes), &tmap_v, bar, bx * 64, y);
    }
  };
  if (tid == 0)
    for (int it = 0; it < min(kStages, my_tiles); ++it) issue(it);

  // Q rows of this CTA -> swizzled shared memory (zeros beyond R)
  const int r_cta = rb * ROWS;
  for (int c = tid; c < ROWS * (D / 8); c += WARPS * 32) {
    const int row = c / (D / 8), ch = c % (D / 8);
    const int r = r_cta + row;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < p.R) {
      const int i = r / g, hl = r % g;
      const __nv_bfloat16* src = p.q + (((size_t)b * N + i) * p.Hq + kvh * g + hl) * D + ch * 8;
      v = __ldg(reinterpret_cast<const uint4*>(src));
    }
    *reinterpret_cast<uint4*>(q_base + (ch >> 3) * (ROWS * 128) + swz(row, ch & 7)) = v;
  }
  __syncthreads();

  // Q fragments of this warp's 16 rows
  uint32_t qa[KSTEPS][4];
  {
    const int m = lane >> 3;
    const int row = warp * 16 + (m & 1) * 8 + (lane & 7);
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      const int ch = ks * 2 + (m >> 1);
      ldsm_x4(smem_u32(q_base + (ch >> 3) * (ROWS * 128) + swz(row, ch & 7)), qa[ks][0],
              qa[ks][1], qa[ks][2], qa[ks][3]);
    }
  }

  // rows handled by this thread: ra (fragment rows g) and ra + 8
  const int ra = r_cta + warp * 16 + (lane >> 2);
  const int node_a = min(ra / g, N - 1), node_b = min((ra + 8) / g, N - 1);
  const unsigned long long anc_a = anc_s[node_a], anc_b = anc_s[node_b];

  float o[DT][4];
#pragma unroll
  for (int i = 0; i < DT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  bool timed_out = false;
  int it = 0;

  for (; it < my_tiles; ++it) {
    const int s = it % kStages;
    const bool ok = mbar_wait(smem_u32(bars + s), (it / kStages) & 1);
    const uint8_t* kst = kv_base + s * stage_bytes<D>();
    const uint8_t* vst = kst + NBOX * kBoxBytes;

    // ---- S = Q K^T  (16 rows x 64 keys per warp)
    float sc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
    {
      const int m = lane >> 3;
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        const uint8_t* kb = kst + (ks >> 2) * kBoxBytes;
        const int ch = (ks & 3) * 2 + (m & 1);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int key = np * 16 + (m >> 1) * 8 + (lane & 7);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_u32(kb + swz(key, ch)), b0, b1, b2, b3);
          mma_bf16(sc[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          mma_bf16(sc[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        }
      }
    }

    // ---- scale, mask, online softmax
    const int key0 = (t_begin + it) * kTileKeys;
    const bool need_mask = key0 + kTileKeys > L;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = sc[n][e] * p.scale_log2;
        if (need_mask) {
          const int col = key0 + n * 8 + 2 * (lane & 3) + (e & 1);
          const int j = col - L;
          const unsigned long long anc = (e < 2) ? anc_a : anc_b;
          const bool vis = j < 0 || (j < N && ((anc >> j) & 1ull));
          if (!vis) v = -INFINITY;
        }
        sc[n][e] = v;
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mx = -INFINITY;
#pragma unroll
      for (int n = 0; n < 8; ++n) mx = fmaxf(mx, fmaxf(sc[n][2 * h], sc[n][2 * h + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run[h], mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = exp2f(m_run[h] - m_use);
      float rs = 0.f;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const float p0 = exp2f(sc[n][2 * h] - m_use);
        const float p1 = exp2f(sc[n][2 * h + 1] - m_use);
        sc[n][2 * h] = p0;
        sc[n][2 * h + 1] = p1;
        rs += p0 + p1;
      }
      l_run[h] = l_run[h] * alpha + rs;
#pragma unroll
      for (int dn = 0; dn < DT; ++dn) {
        o[dn][2 * h] *= alpha;
        o[dn][2 * h + 1] *= alpha;
      }
      m_run[h] = m_new;
    }

    // ---- O += P V
    {
      const int m = lane >> 3;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t a0 = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
        const uint32_t a1 = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
        const uint32_t a2 = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        const uint32_t a3 = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
        const int key = kk * 16 + (m & 1) * 8 + (lane & 7);
#pragma unroll
        for (int dp = 0; dp < DT / 2; ++dp) {
          const uint8_t* vb = vst + (dp >> 2) * kBoxBytes;
          const int ch = (dp & 3) * 2 + (m >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_u32(vb + swz(key, ch)), b0, b1, b2, b3);
          mma_bf16(o[2 * dp], a0, a1, a2, a3, b0, b1);
          mma_bf16(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }

    // ---- release the stage (all warps done with it) and refill it
    if (__syncthreads_or(ok ? 0 : 1)) {
      timed_out = true;
      break;
    }
    if (tid == 0 && it + kStages < my_tiles) issue(it + kStages);
  }
  if (timed_out) {
    // let the loads already issued land before the CTA exits (bounded as well)
    if (tid == 0)
      for (int j = it + 1; j < min(my_tiles, it + kStages + 1); ++j)
        mbar_wait(smem_u32(bars + (j % kStages)), (j / kStages) & 1);
    __syncthreads();
  }

  // full row sums across the quad
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }

  const int cq = 2 * (lane & 3);
  if (p.splits == 1) {
    // final output directly
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = ra + 8 * h;
      if (r >= p.R) continue;
      const int i = r / g, hl = r % g, hq = kvh * g + hl;
      const bool live = !bad && !timed_out && l_run[h] > 0.f;
      const float inv = live ? 1.f / l_run[h] : 0.f;
      __nv_bfloat16* dst = p.out + (((size_t)b * N + i) * p.Hq + hq) * D + cq;
#pragma unroll
      for (int dn = 0; dn < DT; ++dn) {
        *reinterpret_cast<__nv_bfloat162*>(dst + dn * 8) =
            __floats2bfloat162_rn(o[dn][2 * h] * inv, o[dn][2 * h + 1] * inv);
      }
      if (p.lse && (lane & 3) == 0)
        p.lse[((size_t)b * p.Hq + hq) * N + i] =
            live ? (m_run[h] + log2f(l_run[h])) * 0.69314718055994531f : -INFINITY;
    }
    if (timed_out && tid == 0 && p.status) atomicOr(p.status + b, SPEC_ST_TIMEOUT);
  } else {
    const size_t slot = ((size_t)(b * p.Hkv + kvh) * p.splits + split) * p.Rpad;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = ra + 8 * h;  // < Rpad always
      if ((lane & 3) == 0)
        p.part_ml[slot + r] = make_float2(timed_out ? NAN : m_run[h], timed_out ? 0.f : l_run[h]);
      if (l_run[h] > 0.f && !timed_out) {
        float* dst = p.part_o + (slot + r) * D + cq;
#pragma unroll
        for (int dn = 0; dn < DT; ++dn)
          *reinterpret_cast<float2*>(dst + dn * 8) = make_float2(o[dn][2 * h], o[dn][2 * h + 1]);
      }
    }
  }
}

// ------------------------------------------------------------------------------------------------
// 5th-generation tensor-core variant (tcgen05 + TMEM), warp-specialised
// ------------------------------------------------------------------------------------------------
// One CTA per (sequence, KV head, block of 128 query rows, split); 10 warps:
//   warp 0       TMA producer: K/V tiles of 64 keys into a 4-stage ring (128-byte swizzle);
//   warp 1       allocates TMEM; one lane issues the MMAs:
//                  S_j = Q K_j^T   (M = 128 rows, N = 64 keys, K = D)  into TMEM S[j % 2]
//                  O  += P_j V_j   (M = 128, N = D, K = 64 keys)        into TMEM O
//                each completion is signalled through tcgen05.commit on an mbarrier;
//   warps 2..9   softmax: query row r (= TMEM lane r) is shared by warps w and w + 4 of the same
//                TMEM lane quadrant, each taking half of the row's 64 scores (and half of the O
//                columns).  They mask with the node's ancestor bitmask past the prefix, exchange
//                the row max through shared memory (named barrier per warp pair), and write P_j
//                (bf16, swizzled, K-major) for the PV MMA.  The reference max is only raised when
//                a tile's max exceeds it by more than 8 (2^8 headroom); only then is the O row in
//                TMEM rescaled.  Row sums stay per half until the epilogue.
// The QK MMA of tile j+1 is issued before the PV of tile j, so the softmax of one tile overlaps
// the tensor-core work of the next.
template <int D>
struct TcCfg {
  static constexpr int NB = D / 64;               // 64-dim swizzle boxes per row
  static constexpr int KEYS = 64;                 // keys per tile
  static constexpr int ST = 4;                    // K/V pipeline stages
  static constexpr int BOX = KEYS * 128;          // [64 keys x 64 dims] bf16 box: 8 KB
  static constexpr int STAGE = 2 * NB * BOX;      // K + V
  static constexpr int QBOX = 128 * 128;          // [128 rows x 64 dims] bf16: 16 KB
  static constexpr int PBUF = 128 * KEYS * 2;     // [128 rows x 64 keys] bf16: 16 KB
  static constexpr int OFF_Q = ST * STAGE;
  static constexpr int OFF_P = OFF_Q + NB * QBOX;
  static constexpr int OFF_BAR = OFF_P + 2 * PBUF;
  static constexpr int OFF_RED = OFF_BAR + 256;   // row-max exchange: [2 halves][128 rows] fp32
  static constexpr int SMEM = 1024 + OFF_RED + 2 * 128 * 4;
  static constexpr uint32_t TMEM_COLS = 256;      // S[0]: 0..63, S[1]: 64..127, O: 128..128+D
  static constexpr uint32_t O_COL = 128;
  static constexpr int THREADS = 320;
  static constexpr int SOFTMAX_THREADS = 256;
};

__device__ __forceinline__ float ex2_approx(float x) {  // hardware 2^x (P is rounded to bf16)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// AND of v over the 64 threads of a softmax warp pair (also a barrier for the pair), so both warps
// of a pair always take the same branch around their shared named barriers.
__device__ __forceinline__ bool pair_and(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.and.pred po, %2, 64, pi;\n"
      " selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0;
}

template <int D>
__global__ void __launch_bounds__(320, 1) tree_attn_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
    const AttnKParams p) {
  using C = TcCfg<D>;
  constexpr int HALF = C::KEYS / 2;  // scores per softmax thread per tile
  constexpr int DH = D / 2;          // O columns per softmax thread
  extern __shared__ uint8_t smem_raw[];
  __shared__ int par_s[kMaxNodes];
  __shared__ unsigned long long anc_s[kMaxNodes];
  __shared__ int abort_s;
  __shared__ uint32_t tmem_s;

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* kv = base;
  uint8_t* q_s = base + C::OFF_Q;
  uint8_t* p_s = base + C::OFF_P;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::OFF_BAR);
  float* red = reinterpret_cast<float*>(base + C::OFF_RED);  // [half][row]
  const int B_FULL = 0, B_EMPTY = C::ST, B_SFULL = 2 * C::ST, B_SFREE = 2 * C::ST + 2,
            B_PFULL = 2 * C::ST + 4, B_PV = 2 * C::ST + 6, B_DONE = 2 * C::ST + 7;
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y / p.row_blocks, rb = blockIdx.y % p.row_blocks;
  const int b = blockIdx.z;
  const int N = p.N, g = p.g;

  // ---- set-up, with the first K/V tiles in flight as early as possible
  const int tps = p.tiles_per_split;
  const int t_begin = split * tps;
  const int row0 = (b * p.Hkv + kvh) * p.Lmax;
  const int spec = max(0, min(C::ST, min(tps, p.tiles_total - t_begin)));  // issued before L is known
  if (tid == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  griddep_wait();  // every global access below may depend on the preceding kernel in the stream
  griddep_launch_dependents();
  if (tid == 0) {
    for (int i = 0; i < C::ST; ++i) {
      mbar_init(bar(B_FULL + i), 1);
      mbar_init(bar(B_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_SFREE + i), C::SOFTMAX_THREADS);
      mbar_init(bar(B_PFULL + i), C::SOFTMAX_THREADS);
    }
    mbar_init(bar(B_PV), 1);
    mbar_init(bar(B_DONE), 1);
    mbar_fence_init();
    abort_s = 0;
    // the split's first tiles do not depend on the prefix length: issue them now (a tile past
    // L_b + N is simply not consumed)
    for (int it = 0; it < spec; ++it) {
      mbar_arrive_expect_tx(bar(B_FULL + it), C::STAGE);
      uint8_t* st = kv + it * C::STAGE;
      const int y = row0 + (t_begin + it) * C::KEYS;
#pragma unroll
      for (int bx = 0; bx < C::NB; ++bx) {
        tma_load_2d(smem_u32(st + bx * C::BOX), &tmap_k, bar(B_FULL + it), bx * 64, y);
        tma_load_2d(smem_u32(st + (C::NB + bx) * C::BOX), &tmap_v, bar(B_FULL + it), bx * 64, y);
      }
    }
  }
  if (warp == 1) tmem_alloc(smem_u32(&tmem_s), C::TMEM_COLS);
  if (tid >= 64 && tid < 64 + N) par_s[tid - 64] = __ldg(p.parent + (size_t)b * N + (tid - 64));
  const int L = __ldg(p.prefix_lens + b);

  // softmax threads: row r_loc (TMEM lane), half 0 (warps 2..5) or 1 (warps 6..9)
  const int half = (warp >= 6) ? 1 : 0;
  const int r_loc = 32 * (warp & 3) + lane;
  const int r_glob = rb * 128 + r_loc;
  if (warp >= 2) {  // Q rows -> swizzled shared memory (zeros beyond R); each half loads half
    const bool live = r_glob < p.R;
    const int i = live ? r_glob / g : 0, hl = live ? r_glob % g : 0;
    const __nv_bfloat16* src = p.q + (((size_t)b * N + i) * p.Hq + kvh * g + hl) * D;
#pragma unroll
    for (int cc = 0; cc < D / 16; ++cc) {
      const int ch = half * (D / 16) + cc;
      const uint4 v = live ? __ldg(reinterpret_cast<const uint4*>(src) + ch) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(q_s + (ch >> 3) * C::QBOX + swz(r_loc, ch & 7)) = v;
    }
    fence_async_smem();  // Q is read by the tensor cores (async proxy)
  }
  __syncthreads();
  // tree: every node validates its own parent and walks its ancestor chain (in parallel)
  int st_bits = 0;
  if (tid < N) {
    const int pi = par_s[tid];
    if (tid == 0 ? pi != -1 : (pi < 0 || pi >= tid)) st_bits = SPEC_ST_BAD_TREE;
    unsigned long long m = 1ull << tid;
    int k = pi;
    for (int steps = 0; k >= 0 && k < N && steps < N; ++steps) {
      m |= 1ull << k;
      k = par_s[k];
    }
    anc_s[tid] = m;
  }
  if (tid == 0 && (L < 0 || L + N > p.Lmax)) st_bits |= SPEC_ST_BAD_LEN;
  const int bad_tree = __syncthreads_or(st_bits & SPEC_ST_BAD_TREE);
  const int bad_len = __syncthreads_or(st_bits & SPEC_ST_BAD_LEN);
  const bool bad = (bad_tree | bad_len) != 0;
  if (tid == 0 && bad && split == 0 && kvh == 0 && rb == 0 && p.status)
    atomicOr(p.status + b, (bad_tree ? SPEC_ST_BAD_TREE : 0) | (bad_len ? SPEC_ST_BAD_LEN : 0));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_s;

  const int total_keys = bad ? 0 : L + N;
  const int ntiles = (total_keys + C::KEYS - 1) / C::KEYS;
  const int t_end = min(ntiles, t_begin + tps);
  const int my_tiles = max(0, t_end - t_begin);

  auto wait = [&](int i, uint32_t parity) -> bool {
    if (abort_s) return false;
    if (mbar_wait(bar(i), parity)) return true;
    abort_s = 1;
    return false;
  };

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      int issued = spec;
      for (int it = spec; it < my_tiles; ++it) {
        const int s = it % C::ST;
        if (it >= C::ST && !wait(B_EMPTY + s, ((it / C::ST) - 1) & 1)) break;
        uint8_t* st = kv + s * C::STAGE;
        mbar_arrive_expect_tx(bar(B_FULL + s), C::STAGE);
        const int y = row0 + (t_begin + it) * C::KEYS;
#pragma unroll
        for (int bx = 0; bx < C::NB; ++bx) {
          tma_load_2d(smem_u32(st + bx * C::BOX), &tmap_k, bar(B_FULL + s), bx * 64, y);
          tma_load_2d(smem_u32(st + (C::NB + bx) * C::BOX), &tmap_v, bar(B_FULL + s), bx * 64, y);
        }
        issued = it + 1;
      }
      // never leave with a copy in flight: speculative tiles nobody consumed, or an abort
      // (bounded waits)
      if (abort_s || my_tiles < spec)
        for (int it = max(0, issued - C::ST); it < issued; ++it)
          if (abort_s || it >= my_tiles) mbar_wait(bar(B_FULL + it % C::ST), (it / C::ST) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0 && my_tiles > 0) {
      constexpr uint32_t IQK = idesc_bf16_f32(128, C::KEYS, false);
      constexpr uint32_t IPV = idesc_bf16_f32(128, D, true);
      const uint32_t q_addr = smem_u32(q_s);
      auto issue_qk = [&](int j) -> bool {
        const int s = j % C::ST;
        if (!wait(B_FULL + s, (j / C::ST) & 1)) return false;
        if (j >= 2 && !wait(B_SFREE + (j & 1), ((j >> 1) - 1) & 1)) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(kv + s * C::STAGE);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t ad = smem_desc_sw128(q_addr + (ks >> 2) * C::QBOX + (ks & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(k_addr + (ks >> 2) * C::BOX + (ks & 3) * 32, 16, 1024);
          tc_mma_bf16(tmem + (uint32_t)((j & 1) * C::KEYS), ad, bd, IQK, ks > 0 ? 1u : 0u);
        }
        tc_commit(bar(B_SFULL + (j & 1)));
        return true;
      };
      bool ok = issue_qk(0);
      for (int j = 0; ok && j < my_tiles; ++j) {
        if (j + 1 < my_tiles && !issue_qk(j + 1)) break;
        if (!wait(B_PFULL + (j & 1), (j >> 1) & 1)) break;
        tc_fence_after();
        const int s = j % C::ST;
        const uint32_t v_addr = smem_u32(kv + s * C::STAGE + C::NB * C::BOX);
        const uint32_t p_addr = smem_u32(p_s + (j & 1) * C::PBUF);
#pragma unroll
        for (int kk = 0; kk < C::KEYS / 16; ++kk) {
          const uint64_t ad = smem_desc_sw128(p_addr + kk * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(v_addr + kk * 2048, C::BOX, 1024);
          tc_mma_bf16(tmem + C::O_COL, ad, bd, IPV, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(B_PV));
        tc_commit(bar(B_EMPTY + s));
      }
      tc_commit(bar(B_DONE));  // every MMA issued above has completed once this phase completes
      mbar_wait(bar(B_DONE), 0);
    }
  } else {
    // ---------------- softmax: half a query row per thread
    const int node = min(r_glob / g, N - 1);
    const unsigned long long anc = anc_s[node];
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const int pair_bar = 1 + (warp & 3);  // named barrier shared by warps w and w + 4
    const float sc = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    for (int j = 0; j < my_tiles; ++j) {
      if (!pair_and(pair_bar, wait(B_SFULL + (j & 1), (j >> 1) & 1))) break;
      tc_fence_after();
      float x[HALF];
      tmem_ld32(lane_base + (uint32_t)((j & 1) * C::KEYS + half * HALF), x);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(B_SFREE + (j & 1)));  // S[j % 2] may be overwritten by QK of tile j + 2

      const int key0 = (t_begin + j) * C::KEYS + half * HALF;
      float mx = -INFINITY;
      if (key0 + HALF > L) {  // keys past the prefix: ancestor mask
#pragma unroll
        for (int c = 0; c < HALF; ++c) {
          const int jj = key0 + c - L;
          const bool vis = jj < 0 || (jj < N && ((anc >> jj) & 1ull));
          x[c] = vis ? x[c] : -INFINITY;
          mx = fmaxf(mx, x[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < HALF; ++c) mx = fmaxf(mx, x[c]);
      }
      // row max over both halves (scaled, log2 units)
      red[half * 128 + r_loc] = mx;
      named_bar_sync(pair_bar, 64);
      const float mt = fmaxf(mx, red[(half ^ 1) * 128 + r_loc]) * sc;
      named_bar_sync(pair_bar, 64);  // the exchange slot is reused next tile
      const bool raise = mt > m_used + 8.f;
      float factor = 1.f;
      if (raise) {
        factor = (m_used == -INFINITY) ? 0.f : ex2_approx(m_used - mt);
        m_used = mt;
      }
      const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
      float rs0 = 0.f, rs1 = 0.f;
      uint32_t pk[HALF / 2];
#pragma unroll
      for (int c = 0; c < HALF / 2; ++c) {
        const float p0 = ex2_approx(fmaf(x[2 * c], sc, neg_m));
        const float p1 = ex2_approx(fmaf(x[2 * c + 1], sc, neg_m));
        rs0 += p0;
        rs1 += p1;
        pk[c] = pack_bf16(p0, p1);
      }
      l = l * factor + (rs0 + rs1);
      uint8_t* prow = p_s + (j & 1) * C::PBUF;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
        *reinterpret_cast<uint4*>(prow + swz(r_loc, half * 4 + cc)) =
            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      fence_async_smem();
      // O rescale (only after the first tile, only if some row of this warp raised its max)
      if (j > 0 && __any_sync(0xffffffffu, raise)) {
        if (__all_sync(0xffffffffu, wait(B_PV, (j - 1) & 1))) {
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < DH; c0 += 32) {
            float o[32];
            tmem_ld32(lane_base + C::O_COL + half * DH + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] *= factor;
            tmem_st32(lane_base + C::O_COL + half * DH + c0, o);
          }
          tmem_wait_st();
        }
      }
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + (j & 1)));
    }

    // ---------------- epilogue: row sum over both halves, then this thread's half of the row
    red[half * 128 + r_loc] = l;
    named_bar_sync(pair_bar, 64);
    const float lrow = l + red[(half ^ 1) * 128 + r_loc];
    const bool ok = __all_sync(0xffffffffu, my_tiles > 0 && wait(B_PV, (my_tiles - 1) & 1));
    if (ok) tc_fence_after();
    const bool live_row = r_glob < p.R;
    const int i = r_glob / g, hq = kvh * g + r_glob % g;
    if (p.splits == 1) {
      const bool live = ok && !bad && lrow > 0.f;
      const float inv = live ? 1.f / lrow : 0.f;
      __nv_bfloat16* dst = p.out + (((size_t)b * N + i) * p.Hq + hq) * D + half * DH;
#pragma unroll
      for (int c0 = 0; c0 < DH; c0 += 32) {
        float o[32];
        if (ok) {
          tmem_ld32(lane_base + C::O_COL + half * DH + c0, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = 0.f;
        }
        if (live_row) {
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            const uint4 w = make_uint4(pack_bf16(o[c] * inv, o[c + 1] * inv),
                                       pack_bf16(o[c + 2] * inv, o[c + 3] * inv),
                                       pack_bf16(o[c + 4] * inv, o[c + 5] * inv),
                                       pack_bf16(o[c + 6] * inv, o[c + 7] * inv));
            *reinterpret_cast<uint4*>(dst + c0 + c) = w;
          }
        }
      }
      if (half == 0 && live_row && p.lse)
        p.lse[((size_t)b * p.Hq + hq) * N + i] =
            live ? (m_used + log2f(lrow)) * 0.69314718055994531f : -INFINITY;
      if (half == 0 && !ok && my_tiles > 0 && live_row && p.status)
        atomicOr(p.status + b, SPEC_ST_TIMEOUT);
    } else {
      const size_t slot = ((size_t)(b * p.Hkv + kvh) * p.splits + split) * p.Rpad + r_glob;
      const bool has = ok && lrow > 0.f;
      if (half == 0) p.part_ml[slot] = make_float2((my_tiles > 0 && !ok) ? NAN : m_used, has ? lrow : 0.f);
      if (ok) {  // warp-uniform: the TMEM loads are warp-collective
        float* dst = p.part_o + slot * D + half * DH;
#pragma unroll
        for (int c0 = 0; c0 < DH; c0 += 32) {
          float o[32];
          tmem_ld32(lane_base + C::O_COL + half * DH + c0, o);
          tmem_wait_ld();
          if (has) {
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              *reinterpret_cast<float4*>(dst + c0 + c) =
                  make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Combine the splits of one row: out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
// One warp per (sequence, KV head, row).
template <int D>
__global__ void __launch_bounds__(256) tree_attn_merge_kernel(const AttnKParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + warp;
  const int kvh = blockIdx.y, b = blockIdx.z;
  griddep_wait();
  griddep_launch_dependents();
  if (r >= p.R) return;
  const size_t slot0 = (size_t)(b * p.Hkv + kvh) * p.splits * p.Rpad;
  float M = -INFINITY;
  bool timeout = false;
  for (int s = 0; s < p.splits; ++s) {
    const float2 ml = p.part_ml[slot0 + (size_t)s * p.Rpad + r];
    if (isnan(ml.x)) timeout = true;
    else if (ml.y > 0.f) M = fmaxf(M, ml.x);
  }
  constexpr int PER = D / 32;
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;
  float Lsum = 0.f;
  if (M != -INFINITY && !timeout) {
    for (int s = 0; s < p.splits; ++s) {
      const size_t idx = slot0 + (size_t)s * p.Rpad + r;
      const float2 ml = p.part_ml[idx];
      if (!(ml.y > 0.f)) continue;
      const float w = exp2f(ml.x - M);
      Lsum += w * ml.y;
      const float* src = p.part_o + idx * D + lane * PER;
      if constexpr (PER == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
        acc[2] += w * v.z;
        acc[3] += w * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
      }
    }
  }
  const bool live = Lsum > 0.f;
  const float inv = live ? 1.f / Lsum : 0.f;
  const int i = r / p.g, hq = kvh * p.g + r % p.g;
  __nv_bfloat16* dst = p.out + (((size_t)b * p.N + i) * p.Hq + hq) * D + lane * PER;
#pragma unroll
  for (int k = 0; k < PER; k += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + k) =
        __floats2bfloat162_rn(acc[k] * inv, acc[k + 1] * inv);
  if (lane == 0) {
    if (p.lse)
      p.lse[((size_t)b * p.Hq + hq) * p.N + i] =
          live ? (M + log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
    if (timeout && p.status) atomicOr(p.status + b, SPEC_ST_TIMEOUT);
  }
}

// ------------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------------
template <int D, int WARPS>
static int occupancy() {
  int occ = 0;
  auto kern = tree_attn_kernel<D, WARPS>;
  constexpr int smem = attn_smem_bytes<D, WARPS>();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, WARPS * 32, smem) != cudaSuccess)
    return 1;
  return occ > 0 ? occ : 1;
}

bool attn_plan(int B, int N, int Hq, int Hkv, int D, int Lmax, int num_sms, AttnPlan* plan) {
  if (B < 1 || N < 1 || N > kMaxNodes || Hkv < 1 || Hq < Hkv || Hq % Hkv || Lmax < N) return false;
  if (D != 64 && D != 128) return false;
  const int g = Hq / Hkv;
  const int R = N * g;
  plan->tc = true;          // tcgen05 / TMEM kernel: blocks of 128 query rows, 1 CTA per SM
  plan->warps = 8;          // 128 rows per block (the row-block size of the tensor-core kernel)
  const int rows = 128;
  plan->row_blocks = (R + rows - 1) / rows;
  plan->tiles = (Lmax + kTileKeys - 1) / kTileKeys;
  int occ = 1;
  const long long slots = (long long)(num_sms > 0 ? num_sms : 148) * occ;
  const long long base = (long long)B * Hkv * plan->row_blocks;
  int best = 1;
  double best_cost = 1e300;
  for (int s = 1; s <= plan->tiles && s <= 64; ++s) {
    const int tps = (plan->tiles + s - 1) / s;
    const long long waves = (base * s + slots - 1) / slots;
    const double cost = (double)waves * (tps + 2.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  const int tps = (plan->tiles + best - 1) / best;
  plan->splits = (plan->tiles + tps - 1) / tps;
  const long long Rpad = (long long)plan->row_blocks * rows;
  plan->ws_bytes = plan->splits > 1
                       ? (size_t)B * Hkv * plan->splits * Rpad * ((size_t)D * 4 + 8) + 256
                       : 0;
  return true;
}

extern "C" typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                               void*, const cuuint64_t*, const cuuint64_t*,
                                               const cuuint32_t*, const cuuint32_t*,
                                               CUtensorMapInterleave, CUtensorMapSwizzle,
                                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled encode_fn() {
  static PFN_encodeTiled fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled>(p);
  }
  return fn;
}

static bool make_kv_map(CUtensorMap* m, const void* ptr, int D, long long rows) {
  PFN_encodeTiled fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, kTileKeys};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
static cudaError_t launch_tc(const CUtensorMap& mk, const CUtensorMap& mv, const AttnKParams& kp,
                             const AttnPlan& plan, cudaStream_t s) {
  auto kern = tree_attn_tc_kernel<D>;
  constexpr int smem = TcCfg<D>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.splits, kp.Hkv * plan.row_blocks, kp.B);
  cfg.blockDim = dim3(TcCfg<D>::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, mk, mv, kp);
  if (e != cudaSuccess || plan.splits == 1) return e;
  cfg.gridDim = dim3((kp.R + 7) / 8, kp.Hkv, kp.B);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, tree_attn_merge_kernel<D>, kp);
}

template <int D, int WARPS>
static cudaError_t launch_d(const CUtensorMap& mk, const CUtensorMap& mv, const AttnKParams& kp,
                            const AttnPlan& plan, cudaStream_t s) {
  auto kern = tree_attn_kernel<D, WARPS>;
  constexpr int smem = attn_smem_bytes<D, WARPS>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.splits, kp.Hkv * plan.row_blocks, kp.B);
  cfg.blockDim = dim3(WARPS * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, mk, mv, kp);
  if (e != cudaSuccess || plan.splits == 1) return e;
  cfg.gridDim = dim3((kp.R + 7) / 8, kp.Hkv, kp.B);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, tree_attn_merge_kernel<D>, kp);
}

cudaError_t launch_attention(const AttnArgs& a, const AttnPlan& plan, cudaStream_t s) {
  CUtensorMap mk, mv;
  const long long rows = (long long)a.B * a.Hkv * a.Lmax;
  if (!make_kv_map(&mk, a.k, a.D, rows) || !make_kv_map(&mv, a.v, a.D, rows))
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
  kp.Rpad = plan.row_blocks * (plan.tc ? 128 : 16 * plan.warps);
  kp.Lmax = a.Lmax;
  kp.D = a.D;
  kp.splits = plan.splits;
  kp.tiles_per_split = (plan.tiles + plan.splits - 1) / plan.splits;
  kp.tiles_total = plan.tiles;
  kp.row_blocks = plan.row_blocks;
  kp.scale_log2 = a.scale * 1.4426950408889634f;
  const size_t o_bytes = (size_t)a.B * a.Hkv * plan.splits * kp.Rpad * a.D * 4;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  kp.part_o = reinterpret_cast<float*>(ws);
  kp.part_ml = reinterpret_cast<float2*>(ws + ((o_bytes + 255) & ~size_t(255)));
  if (plan.tc) return a.D == 128 ? launch_tc<128>(mk, mv, kp, plan, s) : launch_tc<64>(mk, mv, kp, plan, s);
  if (a.D == 128)
    return plan.warps == 4 ? launch_d<128, 4>(mk, mv, kp, plan, s)
                           : launch_d<128, 8>(mk, mv, kp, plan, s);
  return plan.warps == 4 ? launch_d<64, 4>(mk, mv, kp, plan, s)
                         : launch_d<64, 8>(mk, mv, kp, plan, s);
}

}  // namespace spectree
