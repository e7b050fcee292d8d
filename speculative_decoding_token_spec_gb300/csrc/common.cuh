// Device helpers shared by the tree-attention and tree-verify kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "spectree.h"

namespace spectree {

constexpr int kMaxNodes = 64;            // tree nodes per sequence (root included)
constexpr uint32_t kSpinLimit = 1u << 22;  // polls before a device-side wait gives up

// ------------------------------------------------------------------------------------------------
// shared-memory address helpers
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------------------------------------
// mbarrier (CTA scope) with bounded waits
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of the barrier; false if it did not complete within kSpinLimit polls.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// ------------------------------------------------------------------------------------------------
// TMA (tensor) loads
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int x,
                                            int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ------------------------------------------------------------------------------------------------
// tree helpers
// ------------------------------------------------------------------------------------------------
// Validates tree_parent[b][0..N) held in shared memory and builds each node's ancestor bitmask
// (bit j of anc[i] is set iff j is i or an ancestor of i).  Returns SPEC_ST_BAD_TREE or 0.
// Run by one thread.
__device__ __forceinline__ int build_ancestors(const int* par, int N, unsigned long long* anc) {
  if (par[0] != -1) return SPEC_ST_BAD_TREE;
  anc[0] = 1ull;
  for (int i = 1; i < N; ++i) {
    int p = par[i];
    if (p < 0 || p >= i) return SPEC_ST_BAD_TREE;
    anc[i] = anc[p] | (1ull << i);
  }
  return 0;
}

// ------------------------------------------------------------------------------------------------
// Knuth's TwoSum: s + e == a + b exactly (round-to-nearest fp32, no FMA contraction involved).
// ------------------------------------------------------------------------------------------------
struct CompSum {
  float hi = 0.f, lo = 0.f;
  __device__ __forceinline__ void add(float b) {
    float s = __fadd_rn(hi, b);
    float bb = __fsub_rn(s, hi);
    float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    hi = s;
    lo = __fadd_rn(lo, e);
  }
  __device__ __forceinline__ double value() const { return (double)hi + (double)lo; }
};

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace spectree
