// Post-accept KV compaction (sm_103a).
//
// Method: the target model keeps the accepted draft tokens' keys and values (EAGLE paper explainer,
// vLLM usage section: tree verification holds the tree's extra KV entries in the cache; survey
// explainer, "vLLMでの実装状況": speculative decoding runs on a paged KV cache).  After verification
// accepted the root-to-node path nodes[0..len-1], the root stays at slot L_b and slot L_b + 1 + k
// receives what slot L_b + nodes[k] held before the call; the committed length becomes
// L_b + 1 + len.  A sequence whose verification failed (len = -1) is left alone.
//
// One CTA per (KV head, sequence).  Node ids of a path increase (parents precede children), so a
// destination slot L_b + 1 + k is never above its source, but it can be another move's source
// (path 2, 3: slot L_b + 2 is read by the first move and written by the second): every source row
// is read into registers before any destination row is written.
#include "common.cuh"
#include "internal.h"

namespace spectree {

namespace {

constexpr int kCThreads = 256;

// Row (in units of D elements) of sequence b's slot s, head h; -1 if the page is not a real page.
__device__ __forceinline__ int slot_row(const CompactArgs& a, int b, int h, int s) {
  if (a.page_size == 0) return (b * a.Hkv + h) * a.Lmax + s;
  const int lp = s / a.page_size;
  if (lp >= a.max_pages) return -1;
  const int pg = __ldg(a.block_table + (size_t)b * a.max_pages + lp);
  if (pg < 0 || pg >= a.num_pages) return -1;
  return (pg * a.Hkv + h) * a.page_size + s % a.page_size;
}

template <int D>
__global__ void __launch_bounds__(kCThreads) kv_compact_kernel(const CompactArgs a) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  constexpr int MAXU = (2 * (kMaxNodes - 1) * CH + kCThreads - 1) / kCThreads;
  __shared__ int src_s[kMaxNodes], dst_s[kMaxNodes];
  __shared__ int bad_s;
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  griddep_wait();  // the cache and the verification outputs may come from the preceding kernel
  griddep_launch_dependents();
  if (tid == 0) bad_s = 0;
  const int L = __ldg(a.prefix_lens + b), len = __ldg(a.accept_len + b);
  __syncthreads();
  const bool skip = len < 0;
  if (!skip) {
    if (len > a.N - 1 || L < 0 || (long long)L + 1 + len > a.Lmax) {
      if (tid == 0) atomicOr(&bad_s, SPEC_ST_BAD_PATH);
    } else if (tid < len) {
      const int x = __ldg(a.accepted_nodes + (size_t)b * a.N + tid);
      const int prev = tid == 0 ? 0 : __ldg(a.accepted_nodes + (size_t)b * a.N + tid - 1);
      if (!(prev < x && x < a.N)) {
        atomicOr(&bad_s, SPEC_ST_BAD_PATH);
      } else {
        const int sr = slot_row(a, b, h, L + x), dr = slot_row(a, b, h, L + 1 + tid);
        if (sr < 0 || dr < 0) atomicOr(&bad_s, SPEC_ST_BAD_PAGE);
        src_s[tid] = sr;
        dst_s[tid] = dr;
      }
    }
  }
  __syncthreads();
  const int flags = bad_s;
  if (h == 0 && tid == 0) {
    if (a.new_prefix_lens) a.new_prefix_lens[b] = (skip || flags) ? L : L + 1 + len;
    if (flags && a.status) atomicOr(a.status + b, flags);
  }
  if (skip || flags || len == 0) return;
  const int per = len * CH;  // chunks of one tensor
  uint4 v[MAXU];
#pragma unroll
  for (int u = 0; u < MAXU; ++u) {
    const int idx = tid + u * kCThreads;
    if (idx < 2 * per) {
      const int t = idx / per, rem = idx % per;
      const uint4* src = reinterpret_cast<const uint4*>(t ? a.v : a.k) +
                         (size_t)src_s[rem / CH] * CH + rem % CH;
      v[u] = *src;
    }
  }
  __syncthreads();  // every source chunk of this (sequence, head) has been read
#pragma unroll
  for (int u = 0; u < MAXU; ++u) {
    const int idx = tid + u * kCThreads;
    if (idx < 2 * per) {
      const int t = idx / per, rem = idx % per;
      uint4* dst = reinterpret_cast<uint4*>(t ? a.v : a.k) + (size_t)dst_s[rem / CH] * CH + rem % CH;
      *dst = v[u];
    }
  }
}

}  // namespace

cudaError_t launch_compact(const CompactArgs& a, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hkv, a.B, 1);
  cfg.blockDim = dim3(kCThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return a.D == 128 ? cudaLaunchKernelEx(&cfg, kv_compact_kernel<128>, a)
                    : cudaLaunchKernelEx(&cfg, kv_compact_kernel<64>, a);
}

}  // namespace spectree
