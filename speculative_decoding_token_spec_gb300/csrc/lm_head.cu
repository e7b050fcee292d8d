// The target model's LM head fused with the statistics verification reads (sm_103a).
//
// Method: EAGLE explainer (the target forward over the draft tree yields next-token logits per
// node); survey explainer, Formal Definition, 検証フェーズ (q_j = softmax of node j's target logits;
// each draft token x~ is tested against q_j(x~)).  Verification needs per row only the max m,
// S = sum_y exp((l_y - m) / T), the argmax (T = 0) and the logits of the tokens it tests, so
// q_j(x~) = exp((l_x~ - m) / T) / S.  Here logits = hidden @ W^T are computed on the tensor cores and
// reduced in the epilogue: the fp32 logit matrix is never written or read.
//
// lm_head_kernel: one CTA per (128-row tile, vocabulary tile of 128..256 entries).  Warp 0 streams the
// 64-wide hidden slices of hidden [M, H] and W [V, H] (bf16, 128-byte swizzle) through a 4-stage
// TMA ring; warp 1 issues tcgen05.mma (M = 128, N = the tile width, K = 16; fp32 accumulator in
// TMEM) over the whole hidden dimension; warps 4-7 read their row's accumulators from TMEM
// and write the tile's max, sum of exp and argmax.  Tested tokens are read from a copy of the tile
// in the (then idle) stage memory.  lm_head_combine_kernel merges the tiles of each row.
// Row passes (launch_lm_head_rows, for verification driven by these statistics) write the full
// logits of the few rows whose destination is given, and leave at once when none is requested.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace spectree {

namespace {

extern "C" typedef CUresult (*PFN_encodeTiledLm)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                                 void*, const cuuint64_t*, const cuuint64_t*,
                                                 const cuuint32_t*, const cuuint32_t*,
                                                 CUtensorMapInterleave, CUtensorMapSwizzle,
                                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver (looked up once; null if unavailable).
PFN_encodeTiledLm lm_encode_fn() {
  static PFN_encodeTiledLm fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiledLm>(p);
  });
  return fn;
}

// A 2-D bf16 tensor map with 128-byte swizzle: `inner` elements per row (a multiple of 8), `rows`
// rows, boxes of box_inner x box_rows (box_inner * 2 = 128 bytes); zero fill outside.
bool encode_bf16_2d(CUtensorMap* m, const void* ptr, long long inner, long long rows,
                    int box_inner, int box_rows) {
  PFN_encodeTiledLm fn = lm_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kLM = 128;                        // rows per tile (the MMA's M)
constexpr int kLN = 256;                        // vocabulary entries per tile at most (MMA N)
constexpr int kLK = 64;                         // hidden elements per stage: one 128-byte row
constexpr int kStages = 4;
constexpr int kABytes = kLM * kLK * 2;          // 16 KB
constexpr int kBBytes = kLN * kLK * 2;          // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;  // 48 KB
constexpr int kTileStride = kLN + 1;            // fp32 tile copy: odd row stride, no conflicts
constexpr int kLThreads = 256;
constexpr int kSmemBytes = kStages * kStageBytes + 1024;  // + alignment slack
static_assert(kLM * kTileStride * 4 <= kStages * kStageBytes, "tile copy fits the stages");

__global__ void __launch_bounds__(kLThreads, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap tmap_h,
                   const __grid_constant__ CUtensorMap tmap_w, int M, int H, int V, int G, int tn,
                   int packed,
                   const int32_t* __restrict__ gather_idx, float k2, LmPartial* __restrict__ part,
                   float* __restrict__ out_gather, int32_t* flag,
                   const long long* __restrict__ row_dst, float* __restrict__ out_rows,
                   const int32_t* active) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bars[2 * kStages + 1];  // full[s], empty[s], accumulator
  __shared__ uint32_t tmem_s;
  __shared__ int issued_s, timeout_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.x * kLM, v0 = blockIdx.y * tn;  // tn: this launch's tile width
  const int vend = min(V, v0 + tn);
  const int nk = (H + kLK - 1) / kLK;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  if (tid == 0) {
    prefetch_tmap(&tmap_h);
    prefetch_tmap(&tmap_w);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(s), 1);
      mbar_init(bar(kStages + s), 1);
    }
    mbar_init(bar(2 * kStages), 1);
    mbar_fence_init();
    issued_s = 0;
    timeout_s = 0;
  }
  griddep_wait();  // the hidden states may come from the preceding kernel
  griddep_launch_dependents();
  // a row pass with no row requested (uniform over the grid: nothing allocated or issued yet)
  if (active && *reinterpret_cast<const volatile int32_t*>(active) == 0) return;
  if (warp == 1) tmem_alloc(smem_u32(&tmem_s), kLN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_s;

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer
      int kc = 0;
      for (; kc < nk; ++kc) {
        const int s = kc % kStages;
        if (kc >= kStages && !mbar_wait(bar(kStages + s), ((kc / kStages) - 1) & 1)) {
          timeout_s = 1;
          break;
        }
        const uint32_t a = smem_u32(smem + s * kStageBytes);
        mbar_arrive_expect_tx(bar(s), kABytes + tn * kLK * 2);
        tma_load_2d(a, &tmap_h, bar(s), kc * kLK, m0);
        if (packed)  // tile-major head: box (vocabulary tile, hidden slice) is one contiguous block
          tma_load_2d(a + kABytes, &tmap_w, bar(s), 0, (blockIdx.y * nk + kc) * kLN);
        else
          tma_load_2d(a + kABytes, &tmap_w, bar(s), kc * kLK, v0);
      }
      issued_s = kc;
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer
      const uint32_t IDESC = idesc_bf16_f32(kLM, tn, false);
      int kc = 0;
      for (; kc < nk; ++kc) {
        const int s = kc % kStages;
        if (!mbar_wait(bar(s), (kc / kStages) & 1)) {
          timeout_s = 1;
          break;
        }
        tc_fence_after();
        const uint32_t a = smem_u32(smem + s * kStageBytes), b = a + kABytes;
#pragma unroll
        for (int ks = 0; ks < kLK / 16; ++ks)
          tc_mma_bf16(tmem, smem_desc_sw128(a + ks * 32, 16, 1024),
                      smem_desc_sw128(b + ks * 32, 16, 1024), IDESC, (kc > 0 || ks > 0) ? 1u : 0u);
        tc_commit(bar(kStages + s));  // the stage is free once these MMAs completed
      }
      tc_commit(bar(2 * kStages));  // the accumulator is final (or abandoned)
    }
  } else if (warp >= 4) {
    // ---- epilogue: thread r holds row m0 + r (TMEM lane r)
    const int r = 32 * (warp & 3) + lane, row = m0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const bool ok = mbar_wait(bar(2 * kStages), 0);
    if (!ok) timeout_s = 1;
    tc_fence_after();
    float mx = -INFINITY;
    int am = 0x7fffffff;
    float sum = 0.f;
    if (ok) {
      const int nch = (tn + 31) / 32;  // 32-column chunks (the last may pass the tile: skipped)
#pragma unroll 1
      for (int c = 0; c < nch; ++c) {  // max and argmax (ascending columns: lowest index)
        float v[32];
        tmem_ld32(lane_base + (uint32_t)(32 * c), v);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int col = v0 + 32 * c + q;
          if (col < vend && v[q] > mx) {
            mx = v[q];
            am = col;
          }
        }
      }
      const float mk = __fmul_rn(mx, k2);
      float* tile = reinterpret_cast<float*>(smem);  // the stages are idle now
      float* dst = nullptr;  // this row's full logits (row passes)
      if (out_rows && row < M) {
        const long long o = row_dst[row];
        if (o >= 0) dst = out_rows + o;
      }
#pragma unroll 1
      for (int c = 0; c < nch; ++c) {  // sum of exp((l - max) / T); copy for the gathers
        float v[32];
        tmem_ld32(lane_base + (uint32_t)(32 * c), v);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int col = v0 + 32 * c + q;
          if (col < vend) sum += exp2f(fmaf(v[q], k2, -mk));
          if (G > 0) tile[r * kTileStride + 32 * c + q] = v[q];
          if (dst && col < vend) dst[col] = v[q];
        }
      }
      if (row < M) {
        LmPartial p;
        p.m = mx;
        p.s = sum;
        p.arg = am;
        p.pad = 0;
        if (part) part[(size_t)blockIdx.y * M + row] = p;
        if (G > 0 && out_gather) {
          for (int g = 0; g < G; ++g) {
            const int tok = __ldg(gather_idx + (size_t)row * G + g);
            if (tok >= v0 && tok < vend)
              out_gather[(size_t)row * G + g] = tile[r * kTileStride + (tok - v0)];
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (timeout_s && tid == 0) {
    // wait (bounded) for the copies this CTA still has in flight before its memory goes away
    const int issued = issued_s;
    for (int s = 0; s < kStages; ++s) {
      int last = -1;
      for (int t = s; t < issued; t += kStages) last = t;
      if (last >= 0) mbar_wait(bar(s), (last / kStages) & 1);
    }
    if (flag) atomicOr(flag, SPEC_ST_TIMEOUT);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kLN);
  }
}

// The head in tile-major order: block (t, c) = rows 256 t .. 256 t + 255, hidden elements
// 64 c .. 64 c + 63, stored contiguously (zero past V and H).  One CTA per block.
__global__ void __launch_bounds__(256) lm_head_pack_kernel(const uint16_t* __restrict__ w, int V,
                                                           int H, int nk,
                                                           uint16_t* __restrict__ packed) {
  const int t = blockIdx.x / nk, c = blockIdx.x % nk;
  uint16_t* dst = packed + (size_t)blockIdx.x * kLN * kLK;
  for (int e = threadIdx.x; e < kLN * kLK; e += blockDim.x) {
    const int r = e / kLK, k = e % kLK;
    const int v = t * kLN + r, h = c * kLK + k;
    dst[e] = (v < V && h < H) ? w[(size_t)v * H + h] : (uint16_t)0;
  }
}

// Per row: merge the vocabulary tiles' (max, sum of exp, argmax).  One warp per row; lane l takes
// tiles l, l + 32, ... so that all of a row's partials are loaded at once (one thread walking the
// tiles in turn waits on one L2 load per tile), then the lanes combine by shuffles: the larger max,
// the lower index among equal maxima (tiles ascend in vocabulary order, so the lowest index wins).
constexpr int kCombineRows = 8;  // rows (warps) per 256-thread block
__global__ void __launch_bounds__(256) lm_head_combine_kernel(const LmPartial* __restrict__ part,
                                                              int M, int ntiles, float k2,
                                                              float* out_max, float* out_sumexp,
                                                              int32_t* out_argmax) {
  griddep_wait();
  griddep_launch_dependents();
  const int row = blockIdx.x * kCombineRows + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= M) return;
  float m = -INFINITY;
  int am = 0x7fffffff;
#pragma unroll 4
  for (int t = lane; t < ntiles; t += 32) {
    const LmPartial p = part[(size_t)t * M + row];
    if (p.m > m) {
      m = p.m;
      am = p.arg;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const int oa = __shfl_xor_sync(0xffffffffu, am, o);
    if (om > m || (om == m && oa < am)) {
      m = om;
      am = oa;
    }
  }
  float s = 0.f;
  const float mk = __fmul_rn(m, k2);
#pragma unroll 4
  for (int t = lane; t < ntiles; t += 32) {
    const LmPartial p = part[(size_t)t * M + row];
    if (p.m > -INFINITY) s += p.s * exp2f(fmaf(p.m, k2, -mk));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) {
    if (out_max) out_max[row] = m;
    if (out_sumexp) out_sumexp[row] = s;
    if (out_argmax) out_argmax[row] = am;
  }
}

}  // namespace

// Tile width: 256 vocabulary entries.  Narrower tiles that spread a single row tile over every SM
// (224 wide at V = 32000: 143 CTAs instead of 125) measured no faster: a CTA streams at about the
// same rate either way (each box reads 128-byte pieces of rows 2 H bytes apart).
static int tile_width(int M, int V, int num_sms) {
  (void)M;
  (void)V;
  (void)num_sms;
  return kLN;
}

size_t lm_head_workspace_bytes(int M, int V) {  // one partial per (tile, row); tiles >= 128 wide
  return (size_t)((V + 127) / 128) * (size_t)M * sizeof(LmPartial);
}

size_t lm_head_packed_bytes(int V, int H) {
  return (size_t)((V + kLN - 1) / kLN) * (size_t)((H + kLK - 1) / kLK) * kLN * kLK * 2;
}

cudaError_t launch_lm_head_pack(const void* weight, int V, int H, void* packed, cudaStream_t s) {
  const int nk = (H + kLK - 1) / kLK, nvt = (V + kLN - 1) / kLN;
  lm_head_pack_kernel<<<nvt * nk, 256, 0, s>>>(static_cast<const uint16_t*>(weight), V, H, nk,
                                               static_cast<uint16_t*>(packed));
  return cudaGetLastError();
}

cudaError_t launch_lm_head(const void* hidden, const void* weight, const int32_t* gather_idx, int M,
                           int H, int V, int G, float T, float* out_max, float* out_sumexp,
                           int32_t* out_argmax, float* out_gather, void* workspace,
                           int32_t* flag, int num_sms, bool packed, cudaStream_t s) {
  const int tn = packed ? kLN : tile_width(M, V, num_sms);
  const int nk = (H + kLK - 1) / kLK;
  CUtensorMap mh, mw;
  const bool wmap = packed ? encode_bf16_2d(&mw, weight, kLK,
                                            (long long)((V + kLN - 1) / kLN) * nk * kLN, kLK, kLN)
                           : encode_bf16_2d(&mw, weight, H, V, kLK, tn);
  if (!encode_bf16_2d(&mh, hidden, H, M, kLK, kLM) || !wmap) return cudaErrorInvalidValue;
  const float k2 = (float)(1.4426950408889634 / (double)T);
  const int ntiles = (V + tn - 1) / tn;
  cudaError_t e = cudaFuncSetAttribute(lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((M + kLM - 1) / kLM), (unsigned)ntiles);
  cfg.blockDim = dim3(kLThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  LmPartial* part = static_cast<LmPartial*>(workspace);
  e = cudaLaunchKernelEx(&cfg, lm_head_kernel, mh, mw, M, H, V, G, tn, packed ? 1 : 0, gather_idx,
                         k2, part, out_gather, flag, (const long long*)nullptr, (float*)nullptr,
                         (const int32_t*)nullptr);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t c2 = {};
  c2.gridDim = dim3((unsigned)((M + kCombineRows - 1) / kCombineRows));
  c2.blockDim = dim3(256);
  c2.stream = s;
  c2.attrs = attr;
  c2.numAttrs = 1;
  return cudaLaunchKernelEx(&c2, lm_head_combine_kernel, (const LmPartial*)part, M, ntiles, k2,
                            out_max, out_sumexp, out_argmax);
}

cudaError_t launch_lm_head_rows(const void* hidden, const void* weight, int M, int H, int V,
                                const long long* row_dst, float* out_rows, const int32_t* active,
                                int32_t* flag, bool packed, cudaStream_t s) {
  const int tn = kLN;
  const int nk = (H + kLK - 1) / kLK;
  CUtensorMap mh, mw;
  const bool wmap = packed ? encode_bf16_2d(&mw, weight, kLK,
                                            (long long)((V + kLN - 1) / kLN) * nk * kLN, kLK, kLN)
                           : encode_bf16_2d(&mw, weight, H, V, kLK, tn);
  if (!encode_bf16_2d(&mh, hidden, H, M, kLK, kLM) || !wmap) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((M + kLM - 1) / kLM), (unsigned)((V + tn - 1) / tn));
  cfg.blockDim = dim3(kLThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float k2 = 1.4426950408889634f;  // the statistics of a row pass are not kept
  return cudaLaunchKernelEx(&cfg, lm_head_kernel, mh, mw, M, H, V, 0, tn, packed ? 1 : 0,
                            (const int32_t*)nullptr, k2, (LmPartial*)nullptr, (float*)nullptr, flag,
                            row_dst, out_rows, active);
}

}  // namespace spectree
