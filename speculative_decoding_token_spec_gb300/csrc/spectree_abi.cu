// C ABI of libspectree: argument checks, launch planning and kernel launches (host code).
// Declarations and their documentation: include/spectree.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "spectree.h"

using namespace spectree;

namespace {

int sm_count() {
  static int cache[64] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// First-attempt polls of the verification kernels' bounded waits (spec_debug_set_verify_wait_polls).
std::atomic<uint32_t> g_verify_first_polls{kSpinLimit};

// Argument checks shared by the verification entry points (everything but the workspace).
int verify_check(const float* target_logits, const float* draft_probs, const int32_t* tree_tokens,
                 const int32_t* tree_parent, const float* uniforms, float temperature, int B,
                 int N, int V, const int32_t* out_accept_len, const int32_t* out_accepted_tokens,
                 const int32_t* out_bonus_token) {
  if (!target_logits || !tree_tokens || !tree_parent || !uniforms || !out_accept_len ||
      !out_accepted_tokens || !out_bonus_token)
    return SPEC_ERR_INVALID_ARG;
  if (!std::isfinite(temperature) || temperature < 0.f) return SPEC_ERR_INVALID_ARG;
  if (temperature > 0.f && !draft_probs) return SPEC_ERR_INVALID_ARG;
  if (B < 1 || B > 65535 || N < 1 || N > kMaxNodes || V < 1) return SPEC_ERR_INVALID_ARG;
  if (!verify_supported(V)) return SPEC_ERR_UNSUPPORTED;
  if (!aligned16(target_logits) || (draft_probs && !aligned16(draft_probs)))
    return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}

// The filtered logits follow the verification scratch in the filtered entry's workspace.
size_t filtered_logits_offset(int B, int N, int V) {
  return (verify_workspace_bytes(B, N, V) + 15) & ~size_t(15);
}

}  // namespace

extern "C" {

size_t spec_tree_attention_workspace(int B, int N, int Hq, int Hkv, int D, int Lmax) {
  AttnPlan plan;
  if (!attn_plan(B, N, Hq, Hkv, D, Lmax, sm_count(), &plan)) return 0;
  return plan.ws_bytes;
}

int spec_tree_attention(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* prefix_lens, const int32_t* tree_parent, void* out,
                        float* out_lse, int B, int N, int Hq, int Hkv, int D, int Lmax,
                        float softmax_scale, void* workspace, size_t workspace_bytes,
                        int32_t* status, void* stream) {
  if (!q || !k_cache || !v_cache || !prefix_lens || !tree_parent || !out) return SPEC_ERR_INVALID_ARG;
  if (B < 1 || B > 65535 || N < 1 || N > kMaxNodes || Hkv < 1 || Hq < 1 || Hq % Hkv != 0 ||
      Lmax < N || !std::isfinite(softmax_scale) || !(softmax_scale > 0.f))
    return SPEC_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return SPEC_ERR_UNSUPPORTED;
  if ((long long)B * Hkv * (long long)Lmax >= (1ll << 31)) return SPEC_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return SPEC_ERR_INVALID_ARG;
  const int sms = sm_count();
  if (sms <= 0) return SPEC_ERR_CUDA;
  AttnPlan plan;
  if (!attn_plan(B, N, Hq, Hkv, D, Lmax, sms, &plan)) return SPEC_ERR_INVALID_ARG;
  if (plan.ws_bytes > 0 && (!workspace || workspace_bytes < plan.ws_bytes || !aligned16(workspace)))
    return SPEC_ERR_WORKSPACE;
  AttnArgs a{q, k_cache, v_cache, prefix_lens, tree_parent, out, out_lse, B, N, Hq, Hkv, D,
             Lmax, softmax_scale, status, workspace, workspace_bytes};
  cudaError_t e = launch_attention(a, plan, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

static bool page_size_ok(int P) { return P >= 16 && P <= 1024 && (P & (P - 1)) == 0; }

int spec_tree_attention_paged(const void* q, const void* k_pages, const void* v_pages,
                              const int32_t* block_table, int page_size, int max_pages,
                              int num_pages, const int32_t* prefix_lens,
                              const int32_t* tree_parent, void* out, float* out_lse, int B, int N,
                              int Hq, int Hkv, int D, float softmax_scale, int32_t* status,
                              void* stream) {
  if (!q || !k_pages || !v_pages || !block_table || !prefix_lens || !tree_parent || !out)
    return SPEC_ERR_INVALID_ARG;
  if (B < 1 || B > 65535 || N < 1 || N > kMaxNodes || Hkv < 1 || Hq < 1 || Hq % Hkv != 0 ||
      max_pages < 1 || num_pages < 1 || !std::isfinite(softmax_scale) || !(softmax_scale > 0.f))
    return SPEC_ERR_INVALID_ARG;
  if (!page_size_ok(page_size)) return SPEC_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return SPEC_ERR_UNSUPPORTED;
  const long long lmax = (long long)max_pages * page_size;
  if (lmax < N) return SPEC_ERR_INVALID_ARG;
  if (lmax >= (1ll << 31) || (long long)num_pages * Hkv * page_size >= (1ll << 31))
    return SPEC_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out))
    return SPEC_ERR_INVALID_ARG;
  const int sms = sm_count();
  if (sms <= 0) return SPEC_ERR_CUDA;
  AttnPlan plan;
  if (!attn_plan(B, N, Hq, Hkv, D, (int)lmax, sms, &plan)) return SPEC_ERR_INVALID_ARG;
  if (plan.ws_bytes > 0) return SPEC_ERR_UNSUPPORTED;  // this path takes no workspace
  AttnArgs a{q, k_pages, v_pages, prefix_lens, tree_parent, out, out_lse, B, N, Hq, Hkv, D,
             (int)lmax, softmax_scale, status, nullptr, 0};
  a.page_size = page_size;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.block_table = block_table;
  cudaError_t e = launch_attention(a, plan, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

static int compact_common(CompactArgs& a, void* stream) {
  if (!a.k || !a.v || !a.prefix_lens || !a.accept_len || !a.accepted_nodes)
    return SPEC_ERR_INVALID_ARG;
  if (a.new_prefix_lens && a.new_prefix_lens == a.prefix_lens) return SPEC_ERR_INVALID_ARG;
  if (a.B < 1 || a.B > 65535 || a.N < 1 || a.N > kMaxNodes || a.Hkv < 1 || a.Hkv > 65535 ||
      a.Lmax < 1)
    return SPEC_ERR_INVALID_ARG;
  if (a.D != 64 && a.D != 128) return SPEC_ERR_UNSUPPORTED;
  if (!aligned16(a.k) || !aligned16(a.v)) return SPEC_ERR_INVALID_ARG;
  cudaError_t e = launch_compact(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

int spec_kv_compact(void* k_cache, void* v_cache, const int32_t* prefix_lens,
                    const int32_t* accept_len, const int32_t* accepted_nodes,
                    int32_t* new_prefix_lens, int B, int N, int Hkv, int D, int Lmax,
                    int32_t* status, void* stream) {
  if ((long long)B * Hkv * (long long)Lmax >= (1ll << 31)) return SPEC_ERR_UNSUPPORTED;
  CompactArgs a;
  a.k = k_cache;
  a.v = v_cache;
  a.prefix_lens = prefix_lens;
  a.accept_len = accept_len;
  a.accepted_nodes = accepted_nodes;
  a.new_prefix_lens = new_prefix_lens;
  a.status = status;
  a.B = B;
  a.N = N;
  a.Hkv = Hkv;
  a.D = D;
  a.Lmax = Lmax;
  return compact_common(a, stream);
}

int spec_kv_compact_paged(void* k_pages, void* v_pages, const int32_t* block_table, int page_size,
                          int max_pages, int num_pages, const int32_t* prefix_lens,
                          const int32_t* accept_len, const int32_t* accepted_nodes,
                          int32_t* new_prefix_lens, int B, int N, int Hkv, int D,
                          int32_t* status, void* stream) {
  if (!block_table || page_size < 1 || max_pages < 1 || num_pages < 1) return SPEC_ERR_INVALID_ARG;
  const long long lmax = (long long)max_pages * page_size;
  if (lmax >= (1ll << 31) || (long long)num_pages * Hkv * page_size >= (1ll << 31))
    return SPEC_ERR_UNSUPPORTED;
  CompactArgs a;
  a.k = k_pages;
  a.v = v_pages;
  a.prefix_lens = prefix_lens;
  a.accept_len = accept_len;
  a.accepted_nodes = accepted_nodes;
  a.new_prefix_lens = new_prefix_lens;
  a.status = status;
  a.B = B;
  a.N = N;
  a.Hkv = Hkv;
  a.D = D;
  a.Lmax = (int)lmax;
  a.page_size = page_size;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.block_table = block_table;
  return compact_common(a, stream);
}

size_t spec_tree_verify_workspace(int B, int N, int V) {
  if (B < 1 || N < 1 || N > kMaxNodes || V < 1) return 0;
  return verify_workspace_bytes(B, N, V);
}

int spec_tree_verify(const float* target_logits, const float* draft_probs,
                     const int32_t* tree_tokens, const int32_t* tree_parent,
                     const float* uniforms, float temperature, int B, int N, int V,
                     int32_t* out_accept_len, int32_t* out_accepted_tokens,
                     int32_t* out_bonus_token, int32_t* out_accepted_nodes, float* out_child_q,
                     void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
  const int rc = verify_check(target_logits, draft_probs, tree_tokens, tree_parent, uniforms,
                              temperature, B, N, V, out_accept_len, out_accepted_tokens,
                              out_bonus_token);
  if (rc != SPEC_OK) return rc;
  const size_t need = verify_workspace_bytes(B, N, V);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return SPEC_ERR_WORKSPACE;
  const int sms = sm_count();
  if (sms <= 0) return SPEC_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  VerifyArgs a;
  a.logits = target_logits;
  a.probs = draft_probs;
  a.tokens = tree_tokens;
  a.parent = tree_parent;
  a.uniforms = uniforms;
  a.T = temperature;
  a.B = B;
  a.N = N;
  a.V = V;
  a.accept_len = out_accept_len;
  a.acc_tokens = out_accepted_tokens;
  a.bonus = out_bonus_token;
  a.acc_nodes = out_accepted_nodes;
  a.child_q = out_child_q;
  a.status = status;
  a.stats = reinterpret_cast<NodeStat*>(ws);
  a.counters = reinterpret_cast<unsigned long long*>(ws + (size_t)B * N * sizeof(NodeStat));
  a.handover = a.counters + B;
  a.walk_done = a.handover + (size_t)B * N;
  static std::atomic<unsigned long long> call_gen{1};
  a.gen = call_gen.fetch_add(1) & 0xFFFFFFFFull;
  a.first_polls = g_verify_first_polls.load(std::memory_order_relaxed);
  cudaError_t e = launch_verify(a, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

size_t spec_tree_verify_filtered_workspace(int B, int N, int V) {
  if (B < 1 || N < 1 || N > kMaxNodes || V < 1) return 0;
  return filtered_logits_offset(B, N, V) + (size_t)B * N * V * sizeof(float);
}

int spec_tree_verify_filtered(const float* target_logits, const float* draft_probs,
                              const int32_t* tree_tokens, const int32_t* tree_parent,
                              const float* uniforms, float temperature, int top_k, float top_p,
                              int B, int N, int V, int32_t* out_accept_len,
                              int32_t* out_accepted_tokens, int32_t* out_bonus_token,
                              int32_t* out_accepted_nodes, float* out_child_q, void* workspace,
                              size_t workspace_bytes, int32_t* status, void* stream) {
  const int rc = verify_check(target_logits, draft_probs, tree_tokens, tree_parent, uniforms,
                              temperature, B, N, V, out_accept_len, out_accepted_tokens,
                              out_bonus_token);
  if (rc != SPEC_OK) return rc;
  if (top_k < 0 || !(top_p > 0.f && top_p <= 1.f)) return SPEC_ERR_INVALID_ARG;
  if (!filter_supported(V)) return SPEC_ERR_UNSUPPORTED;
  const bool active = temperature > 0.f && ((top_k > 0 && top_k < V) || top_p < 1.f);
  if (!active)
    return spec_tree_verify(target_logits, draft_probs, tree_tokens, tree_parent, uniforms,
                            temperature, B, N, V, out_accept_len, out_accepted_tokens,
                            out_bonus_token, out_accepted_nodes, out_child_q, workspace,
                            workspace_bytes, status, stream);
  const size_t off = filtered_logits_offset(B, N, V);
  if (!workspace || workspace_bytes < off + (size_t)B * N * V * sizeof(float) ||
      !aligned16(workspace))
    return SPEC_ERR_WORKSPACE;
  float* filtered = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + off);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int sms = sm_count();
  if (sms <= 0) return SPEC_ERR_CUDA;
  if (launch_filter(target_logits, filtered, B * N, V, temperature, top_k, top_p, sms, s) !=
      cudaSuccess)
    return SPEC_ERR_CUDA;
  return spec_tree_verify(filtered, draft_probs, tree_tokens, tree_parent, uniforms, temperature,
                          B, N, V, out_accept_len, out_accepted_tokens, out_bonus_token,
                          out_accepted_nodes, out_child_q, workspace, off, status, stream);
}

// ---- dynamic tree construction
namespace {
bool tree_shape_ok(int B, int K, int D) {
  if (B < 1 || K < 1 || K > kMaxTreeK || D < 1 || D > 16) return false;
  return 1 + K + (long long)(D - 1) * K * K <= kMaxTreePool;
}
}  // namespace

size_t spec_tree_build_workspace(int B, int K, int D) {
  if (!tree_shape_ok(B, K, D)) return 0;
  return (size_t)B * tree_build_stride(K, D);
}

int spec_tree_expand(const float* draft_logits, int B, int V, int K, int D, int level,
                     void* workspace, size_t workspace_bytes, int32_t* out_frontier_tokens,
                     int32_t* out_frontier_parent_slot, int32_t* status, void* stream) {
  if (!draft_logits || !tree_shape_ok(B, K, D) || V < K || level < 1 || level > D)
    return SPEC_ERR_INVALID_ARG;
  const int R = level == 1 ? 1 : K;
  if ((long long)B * R > 0x7fffffffLL) return SPEC_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < spec_tree_build_workspace(B, K, D) || !aligned16(workspace))
    return SPEC_ERR_WORKSPACE;
  const cudaError_t e =
      launch_tree_expand(draft_logits, B, R, V, K, D, level, workspace, out_frontier_tokens,
                         out_frontier_parent_slot, status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

int spec_tree_finalize(const void* workspace, size_t workspace_bytes, const int32_t* root_tokens,
                       int B, int K, int D, int N, int32_t* out_tree_tokens,
                       int32_t* out_tree_parent, int32_t* out_node_row, float* out_node_value,
                       int32_t* status, void* stream) {
  if (!root_tokens || !out_tree_tokens || !out_tree_parent || !tree_shape_ok(B, K, D))
    return SPEC_ERR_INVALID_ARG;
  if (N < 1 || N > kMaxNodes || N > 1 + K + (D - 1) * K * K) return SPEC_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < spec_tree_build_workspace(B, K, D) || !aligned16(workspace))
    return SPEC_ERR_WORKSPACE;
  const cudaError_t e = launch_tree_finalize(workspace, B, K, D, root_tokens, N, out_tree_tokens,
                                             out_tree_parent, out_node_row, out_node_value, status,
                                             static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// ---- fused LM head
size_t spec_lm_head_stats_workspace(int M, int V) {
  if (M < 1 || V < 1) return 0;
  return lm_head_workspace_bytes(M, V);
}

namespace {
int lm_head_common(const void* hidden, const void* weight, const int32_t* gather_idx, int M, int H,
                   int V, int G, float temperature, float* out_max, float* out_sumexp,
                   int32_t* out_argmax, float* out_gather, void* workspace,
                   size_t workspace_bytes, int32_t* status, void* stream, bool packed) {
  if (!hidden || !weight || M < 1 || H < 8 || (H & 7) || V < 1 || G < 0)
    return SPEC_ERR_INVALID_ARG;
  if (!std::isfinite(temperature) || !(temperature > 0.f)) return SPEC_ERR_INVALID_ARG;
  if (G > 0 && (!gather_idx || !out_gather)) return SPEC_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(weight)) return SPEC_ERR_INVALID_ARG;
  if ((long long)(V + 127) / 128 > 65535 || (long long)M * V > (1ll << 40))
    return SPEC_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < lm_head_workspace_bytes(M, V) || !aligned16(workspace))
    return SPEC_ERR_WORKSPACE;
  const int sms = sm_count();
  if (sms <= 0) return SPEC_ERR_CUDA;
  const cudaError_t e = launch_lm_head(hidden, weight, gather_idx, M, H, V, G, temperature, out_max,
                                       out_sumexp, out_argmax, out_gather, workspace, status, sms,
                                       packed, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidValue) return SPEC_ERR_INVALID_ARG;  // tensor maps refused
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
}  // namespace

int spec_lm_head_stats(const void* hidden, const void* weight, const int32_t* gather_idx, int M,
                       int H, int V, int G, float temperature, float* out_max, float* out_sumexp,
                       int32_t* out_argmax, float* out_gather, void* workspace,
                       size_t workspace_bytes, int32_t* status, void* stream) {
  return lm_head_common(hidden, weight, gather_idx, M, H, V, G, temperature, out_max, out_sumexp,
                        out_argmax, out_gather, workspace, workspace_bytes, status, stream, false);
}

size_t spec_lm_head_packed_bytes(int V, int H) {
  if (V < 1 || H < 8 || (H & 7)) return 0;
  return lm_head_packed_bytes(V, H);
}

int spec_lm_head_pack(const void* weight, int V, int H, void* packed, size_t packed_bytes,
                      void* stream) {
  if (!weight || V < 1 || H < 8 || (H & 7)) return SPEC_ERR_INVALID_ARG;
  if (!packed || packed_bytes < lm_head_packed_bytes(V, H) || !aligned16(packed))
    return SPEC_ERR_WORKSPACE;
  return launch_lm_head_pack(weight, V, H, packed, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

int spec_lm_head_stats_packed(const void* hidden, const void* packed, const int32_t* gather_idx,
                              int M, int H, int V, int G, float temperature, float* out_max,
                              float* out_sumexp, int32_t* out_argmax, float* out_gather,
                              void* workspace, size_t workspace_bytes, int32_t* status,
                              void* stream) {
  return lm_head_common(hidden, packed, gather_idx, M, H, V, G, temperature, out_max, out_sumexp,
                        out_argmax, out_gather, workspace, workspace_bytes, status, stream, true);
}

int spec_tree_verify_greedy(const int32_t* node_argmax, const int32_t* tree_tokens,
                            const int32_t* tree_parent, int B, int N, int V,
                            int32_t* out_accept_len, int32_t* out_accepted_tokens,
                            int32_t* out_bonus_token, int32_t* out_accepted_nodes, int32_t* status,
                            void* stream) {
  if (!node_argmax || !tree_tokens || !tree_parent || !out_accept_len || !out_accepted_tokens ||
      !out_bonus_token)
    return SPEC_ERR_INVALID_ARG;
  if (B < 1 || B > (1 << 24) || N < 1 || N > kMaxNodes || V < 1) return SPEC_ERR_INVALID_ARG;
  return launch_verify_greedy(node_argmax, tree_tokens, tree_parent, B, N, V, out_accept_len,
                              out_accepted_tokens, out_bonus_token, out_accepted_nodes, status,
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

size_t spec_tree_verify_head_workspace(int B, int N, int H, int V, int max_depth) {
  if (B < 1 || N < 1 || N > kMaxNodes || H < 8 || (H & 7) || V < 1 || max_depth < 0 ||
      max_depth >= N)
    return 0;
  return verify_head_workspace_bytes(B, N, H, V, max_depth);
}

int spec_tree_verify_head(const void* hidden, const void* head, int head_packed,
                          const float* draft_probs, const int32_t* tree_tokens,
                          const int32_t* tree_parent, const float* uniforms, float temperature,
                          int B, int N, int H, int V, int max_depth, int32_t* out_accept_len,
                          int32_t* out_accepted_tokens, int32_t* out_bonus_token,
                          int32_t* out_accepted_nodes, void* workspace, size_t workspace_bytes,
                          int32_t* status, void* stream) {
  if (!hidden || !head || !tree_tokens || !tree_parent || !uniforms || !out_accept_len ||
      !out_accepted_tokens || !out_bonus_token)
    return SPEC_ERR_INVALID_ARG;
  if (!std::isfinite(temperature) || temperature < 0.f) return SPEC_ERR_INVALID_ARG;
  if (temperature > 0.f && (!draft_probs || !aligned16(draft_probs))) return SPEC_ERR_INVALID_ARG;
  if (B < 1 || B > 65535 || N < 1 || N > kMaxNodes || V < 1 || H < 8 || (H & 7))
    return SPEC_ERR_INVALID_ARG;
  if (max_depth < 0 || max_depth >= N) return SPEC_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(head)) return SPEC_ERR_INVALID_ARG;
  if (!verify_supported(V) || (long long)(V + 127) / 128 > 65535 ||
      (long long)B * N * V > (1ll << 40))
    return SPEC_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < verify_head_workspace_bytes(B, N, H, V, max_depth))
    return SPEC_ERR_WORKSPACE;
  const int sms = sm_count();
  if (sms <= 0) return SPEC_ERR_CUDA;
  HeadVerifyArgs a;
  a.hidden = hidden;
  a.head = head;
  a.packed = head_packed != 0;
  a.probs = draft_probs;
  a.tokens = tree_tokens;
  a.parent = tree_parent;
  a.uniforms = uniforms;
  a.T = temperature;
  a.B = B;
  a.N = N;
  a.H = H;
  a.V = V;
  a.max_depth = max_depth;
  a.accept_len = out_accept_len;
  a.acc_tokens = out_accepted_tokens;
  a.bonus = out_bonus_token;
  a.acc_nodes = out_accepted_nodes;
  a.status = status;
  a.workspace = workspace;
  a.first_polls = g_verify_first_polls.load(std::memory_order_relaxed);
  const cudaError_t e = launch_verify_head(a, sms, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidValue) return SPEC_ERR_INVALID_ARG;  // tensor maps refused
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

int spec_debug_set_verify_wait_polls(long long polls) {
  const uint32_t v = polls < 0 || polls > (long long)kSpinLimit ? kSpinLimit : (uint32_t)polls;
  g_verify_first_polls.store(v, std::memory_order_relaxed);
  return SPEC_OK;
}

const char* spec_status_string(int code) {
  switch (code) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument (shape, pointer, alignment or temperature)";
    case SPEC_ERR_UNSUPPORTED: return "shape not supported by the kernels";
    case SPEC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SPEC_ERR_CUDA: return "CUDA runtime or launch failure";
    case SPEC_ERR_NOALLOC_LIMIT:
      return "B * N exceeds SPEC_NOALLOC_MAX_NODES, the fixed scratch of spec_tree_verify_noalloc";
    case SPEC_ST_BAD_TREE: return "bad tree: parent[0] != -1 or parent[i] not in [0, i)";
    case SPEC_ST_BAD_LEN: return "bad prefix length: L_b < 0 or L_b + N > Lmax";
    case SPEC_ST_BAD_TOKEN: return "draft token outside [0, V)";
    case SPEC_ST_NONFINITE: return "NaN/Inf in a target-logit row or a bad draft probability";
    case SPEC_ST_TIMEOUT: return "a bounded device-side wait gave up";
    case SPEC_ST_BAD_PAGE: return "block-table entry outside [0, num_pages) for a slot the call uses";
    case SPEC_ST_BAD_PATH:
      return "accepted nodes not increasing inside [1, N), or L_b + 1 + accept_len > Lmax";
    default: return "unknown status code";
  }
}

}  // extern "C"
