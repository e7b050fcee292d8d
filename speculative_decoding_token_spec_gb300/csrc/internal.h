// Internal interface between the C-ABI host code and the verify / attention kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace spectree {

// Per (sequence, node) record written by the node's cluster and read by the walk.
struct NodeStat {
  float m;        // max target logit of the row (raw logit units)
  int argmax;     // lowest index attaining the max
  float s_hi;     // sum_y exp((l_y - m) / T), as a double-float
  float s_lo;
  int first_acc;  // accepted child, or -1 when every child was rejected
  int nrej;       // children rejected before first_acc (all of them if none was accepted)
  int flags;      // SPEC_ST_NONFINITE / SPEC_ST_TIMEOUT met while processing the node
  int bonus;      // token drawn if the walk stops at this node (-1: not a possible stop)
};
static_assert(sizeof(NodeStat) == 32, "NodeStat layout");

// Walk state of one sequence in verification driven by the LM head's statistics
// (verify_head.cu): the walk stands at `cur`; `pending` is the node whose full logit row the next
// node step processes (-1: none).
constexpr int kHeadMaxNodes = 64;
struct HeadWalk {
  int cur;
  int pending;
  int len;   // accepted nodes so far, in path[0 .. len)
  int done;  // the sequence's outputs are written
  int path[kHeadMaxNodes];
};

// Slot of node j's logit row in that verification's row buffer: sequence b's stretch of V + 4
// floats, shifted so that the row has the 16-byte phase of draft row (b, j) (the node step stages
// both with the same slice bounds).
__host__ __device__ inline long long head_row_offset(int b, int j, int N, int V) {
  const unsigned long long e = ((unsigned long long)b * (unsigned)N + (unsigned)j) * (unsigned)V;
  const unsigned long long base = (unsigned long long)b * (unsigned)(V + 4);
  return (long long)(base + ((e - base) & 3ull));  // == e (mod 4), within [base, base + 4)
}

// What the statistics walk of the head-driven verification reads and writes (verify_head.cu; the
// node step continues the walk in its tail, tree_verify.cu).
struct HeadWalkIn {
  const uint16_t* hidden = nullptr;  // bf16 [B * N, H]
  const int32_t* fchild = nullptr;   // [B, N] first child (-1: leaf)
  const float* stat_m = nullptr;     // [B, N] row max, sum of exp, first child's logit
  const float* stat_s = nullptr;
  const float* gath = nullptr;
  long long* row_dst = nullptr;  // [B] row slot of the pending node (-1: none)
  int32_t* active = nullptr;     // the next row pass's flag (null: no next pass)
  uint16_t* hrow = nullptr;      // bf16 [B, H] hidden states of the pending nodes
  double invT = 0.0;
  int H = 0;
};

struct VerifyArgs {
  const float* logits;
  const float* probs;
  const int32_t* tokens;
  const int32_t* parent;
  const float* uniforms;
  float T;
  int B, N, V;
  int32_t* accept_len;
  int32_t* acc_tokens;
  int32_t* bonus;
  int32_t* acc_nodes;
  float* child_q;
  int32_t* status;
  NodeStat* stats;  // [B, N]
  // [B] arrival counters: (generation << 32) | (tag << 16) | arrivals; in the every-node form
  // without per-child q, call tickets: (generation << 32) | tickets taken
  unsigned long long* counters;
  // [B, N] walk hand-over words and [B] walk-done words of the every-node form without per-child
  // q: (tag << 32) | state, the tag derived from the generation and the call's ticket epoch
  // (see tree_verify.cu); words of other calls carry other tags, so none is ever cleared
  unsigned long long* handover;
  unsigned long long* walk_done;
  unsigned long long gen;        // this call's generation (32 bits)
  int p_global = 0;  // set by launch_verify: draft rows read from global memory, not staged
  // polls of the first attempt of each bounded wait (row copies, cluster exchanges); a wait that
  // gives up flags SPEC_ST_TIMEOUT and then drains with the full limit.  Normally the full limit;
  // lowered only through spec_debug_set_verify_wait_polls (tests of the timeout path).
  uint32_t first_polls = 0;
  // node steps of the head-driven verification: row (b, j) lives at head_rows + head_row_offset
  const float* head_rows = nullptr;
  HeadWalk* head_state = nullptr;
  const int32_t* head_flag = nullptr;  // non-zero: an LM-head pass gave up (SPEC_ST_TIMEOUT)
  HeadWalkIn head_walk;                // the walk continued after an accepted child
};
uint32_t verify_first_polls();  // the current first-attempt limit (spectree_abi.cu)

size_t verify_workspace_bytes(int B, int N, int V);
bool verify_supported(int V);  // the row slices of a cluster fit in shared memory
cudaError_t launch_verify(const VerifyArgs& a, int num_sms, cudaStream_t s);
// one node step per sequence whose head_state[b].pending >= 0 (T > 0), tree_verify.cu
cudaError_t launch_verify_head_step(const VerifyArgs& a, int num_sms, cudaStream_t s);
// rows of V target logits -> the same rows with -inf outside the top-k / top-p set (T > 0)
// fused LM head (lm_head.cu)
struct LmPartial {
  float m, s;  // a vocabulary tile's max and sum of exp((l - m) / T)
  int arg;     // its argmax (lowest index)
  int pad;
};
size_t lm_head_workspace_bytes(int M, int V);
cudaError_t launch_lm_head(const void* hidden, const void* weight, const int32_t* gather_idx, int M,
                           int H, int V, int G, float T, float* out_max, float* out_sumexp,
                           int32_t* out_argmax, float* out_gather, void* workspace,
                           int32_t* flag, int num_sms, bool packed, cudaStream_t s);
size_t lm_head_packed_bytes(int V, int H);
// Full logit rows of M hidden rows: row r goes to out_rows + row_dst[r] (skipped when negative);
// every CTA returns at once when *active == 0.  No statistics are kept.
cudaError_t launch_lm_head_rows(const void* hidden, const void* weight, int M, int H, int V,
                                const long long* row_dst, float* out_rows, const int32_t* active,
                                int32_t* flag, bool packed, cudaStream_t s);
// Greedy verification from each node's argmax token (verify_greedy.cu).
cudaError_t launch_verify_greedy(const int32_t* node_argmax, const int32_t* tokens,
                                 const int32_t* parent, int B, int N, int V, int32_t* accept_len,
                                 int32_t* acc_tokens, int32_t* bonus, int32_t* acc_nodes,
                                 int32_t* status, cudaStream_t s);
cudaError_t launch_lm_head_pack(const void* weight, int V, int H, void* packed, cudaStream_t s);

// Verification driven by the LM head's statistics (verify_head.cu).
struct HeadVerifyArgs {
  const void* hidden;  // bf16 [B * N, H]
  const void* head;    // bf16 [V, H], or packed (lm_head_packed_bytes)
  bool packed;
  const float* probs;  // [B, N, V] (T > 0)
  const int32_t* tokens;
  const int32_t* parent;
  const float* uniforms;
  float T;
  int B, N, H, V, max_depth;
  int32_t* accept_len;
  int32_t* acc_tokens;
  int32_t* bonus;
  int32_t* acc_nodes;
  int32_t* status;
  void* workspace;
  uint32_t first_polls;
};
size_t verify_head_workspace_bytes(int B, int N, int H, int V, int max_depth);
cudaError_t launch_verify_head(const HeadVerifyArgs& a, int num_sms, cudaStream_t s);

// dynamic tree construction (tree_build.cu)
constexpr int kMaxTreeK = 16;       // candidates per expanded node, frontier size
constexpr int kMaxTreePool = 2048;  // drafted nodes per sequence: 1 + K + (D - 1) K^2
size_t tree_build_stride(int K, int D);  // workspace bytes per sequence
cudaError_t launch_tree_expand(const float* logits, int B, int R, int V, int K, int D, int level,
                               void* state, int32_t* ftok, int32_t* fslot, int32_t* status,
                               cudaStream_t s);
cudaError_t launch_tree_finalize(const void* state, int B, int K, int D, const int32_t* root_tokens,
                                 int N, int32_t* tree_tokens, int32_t* tree_parent,
                                 int32_t* node_row, float* node_value, int32_t* status,
                                 cudaStream_t s);

bool filter_supported(int V);  // a row fits the filter kernel's clusters
cudaError_t launch_filter(const float* in, float* out, int rows, int V, float T, int top_k,
                          float top_p, int num_sms, cudaStream_t s);

struct AttnArgs {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* prefix_lens;
  const int32_t* parent;
  void* out;
  float* lse;
  int B, N, Hq, Hkv, D, Lmax;
  float scale;
  int32_t* status;
  void* workspace;
  size_t ws_bytes;
  // paged cache (page_size > 0): k / v are pages [num_pages][Hkv][page_size][D], Lmax =
  // max_pages * page_size, block_table [B][max_pages]
  int page_size = 0, max_pages = 0, num_pages = 0;
  const int32_t* block_table = nullptr;
};

struct AttnPlan {
  int kg;               // key groups per 128-row MMA block: 2 when the head's R <= 64 rows
  int row_blocks;       // CTAs along the query rows of one KV head
  int splits;           // split-KV factor = cluster size (<= 8)
  int tiles;            // 64-key tiles covering Lmax
  int tiles_per_split;
  size_t ws_bytes;      // device scratch needed (0: the splits are combined on chip)
};

bool attn_plan(int B, int N, int Hq, int Hkv, int D, int Lmax, int num_sms, AttnPlan* plan);
cudaError_t launch_attention(const AttnArgs& a, const AttnPlan& plan, cudaStream_t s);

// post-accept compaction (contiguous when page_size == 0)
struct CompactArgs {
  void* k;
  void* v;
  const int32_t* prefix_lens;
  const int32_t* accept_len;
  const int32_t* accepted_nodes;
  int32_t* new_prefix_lens;
  int32_t* status;
  int B, N, Hkv, D, Lmax;
  int page_size = 0, max_pages = 0, num_pages = 0;
  const int32_t* block_table = nullptr;
};
cudaError_t launch_compact(const CompactArgs& a, cudaStream_t s);

}  // namespace spectree
