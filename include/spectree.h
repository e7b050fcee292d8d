/*
 * spectree.h -- C ABI of the GB300 (sm_103a) token-tree verification library (libspectree.so).
 *
 * The library computes the verification step of EAGLE-style speculative decoding:
 *
 *   1. spec_tree_attention: tree-masked attention.  Every node of the draft tree attends to its
 *      sequence's KV-cache prefix and to its own ancestors (itself included), as given by parent
 *      indices.  Defined by the EAGLE paper explainer, "Static tree" section (all tree paths are
 *      verified in one forward pass under a tree attention mask) and the speculative-decoding
 *      survey explainer, verification taxonomy ("Token Tree verification").
 *
 *   2. spec_tree_verify: speculative-sampling accept/reject over the tree.  Survey explainer,
 *      "Formal Definition": draft x~_i is accepted if r < min(1, q_i(x~_i) / p_i(x~_i)); at the first
 *      rejection c the next token is drawn from norm(max(0, q_c - p_c)); with temperature 0 the test
 *      is greedy argmax matching (taxonomy table, "Greedy verification").
 *
 * Conventions shared by every entry point
 *   - All array arguments are DEVICE pointers (cudaMalloc'd or managed memory) owned by the caller.
 *     The library never allocates, frees or retains them and keeps no state between calls.
 *   - Every call is asynchronous on `stream` (a cudaStream_t, NULL = legacy default stream) and
 *     performs no host<->device synchronisation.  Calls on different streams are independent as
 *     long as they do not share output or workspace buffers.
 *   - Argument errors are reported synchronously, before anything is launched, by a negative
 *     return value (spec_err_t).  A launch failure returns SPEC_ERR_CUDA.
 *   - Content errors found on the device are reported per sequence in `status[b]` (SPEC_ST_* bits;
 *     `status` may be NULL).  Bits are OR-ed into status[b] with atomics and never cleared by the
 *     library (sticky, like an error flag): zero the array before the first call and whenever the
 *     caller has handled the errors.  A flagged sequence gets -1 in its integer outputs and zeros
 *     in its attention rows; other sequences are unaffected.
 *   - No kernel traps, asserts or waits without bound: every device-side wait gives up after a
 *     fixed number of polls and sets SPEC_ST_TIMEOUT.
 *   - Node 0 of every tree is the root (the last committed token, whose key/value is written at
 *     cache slot L_b like every other node).  tree_parent[b][0] == -1 and
 *     0 <= tree_parent[b][i] < i for i >= 1 (parents precede children).  1 <= N <= 64.
 */
#ifndef SPECTREE_H
#define SPECTREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = -1, /* bad shape, NULL required pointer, T < 0 or non-finite, ... */
  SPEC_ERR_UNSUPPORTED = -2, /* shape outside what the kernels implement (e.g. D not 64/128)  */
  SPEC_ERR_WORKSPACE = -3,   /* workspace NULL or smaller than the *_workspace() query        */
  SPEC_ERR_CUDA = -4,        /* a CUDA runtime / driver call or a launch failed               */
  SPEC_ERR_NOALLOC_LIMIT = -5 /* B * N above SPEC_NOALLOC_MAX_NODES (spec_tree_verify_noalloc)  */
} spec_err_t;

/* per-sequence status bits (int32 status[B]) */
#define SPEC_ST_BAD_TREE 1   /* tree_parent[b][0] != -1, or tree_parent[b][i] outside [0, i)       */
#define SPEC_ST_BAD_LEN 2    /* prefix_lens[b] < 0 or prefix_lens[b] + N > Lmax                    */
#define SPEC_ST_BAD_TOKEN 4  /* a draft token tree_tokens[b][i >= 1] outside [0, V)                */
#define SPEC_ST_NONFINITE 8  /* NaN or +Inf in a target-logit row that was read, or a bad p value  */
#define SPEC_ST_TIMEOUT 16   /* a bounded device-side wait gave up                                 */
#define SPEC_ST_BAD_PAGE 32  /* paged cache: a block-table entry a call needs is outside [0, pages) */
#define SPEC_ST_BAD_PATH 64  /* compaction: accepted nodes not increasing in [1, N), or L+1+len>Lmax */

/* ------------------------------------------------------------------------------------------------
 * Tree attention
 * ------------------------------------------------------------------------------------------------
 * Workspace bytes spec_tree_attention needs for these sizes on the current device.  This
 * implementation combines its split-KV partial results on chip and returns 0 (as it does for
 * invalid sizes); callers that pass a buffer of the returned size keep working if a later version
 * needs scratch.
 */
size_t spec_tree_attention_workspace(int B, int N, int Hq, int Hkv, int D, int Lmax);

/*
 * Tree-masked attention of the draft tree's queries (one layer).
 *
 *   q           bf16 [B, N, Hq, D]      query of node i, head h (RoPE already applied)
 *   k_cache     bf16 [B, Hkv, Lmax, D]  keys; prefix at slots 0..L_b-1, node i's key at slot L_b+i
 *   v_cache     bf16 [B, Hkv, Lmax, D]  values, same slots
 *   prefix_lens int32 [B]               L_b, the committed prefix length of sequence b
 *   tree_parent int32 [B, N]            parent index of every node (see conventions)
 *   out         bf16 [B, N, Hq, D]      attention output
 *   out_lse     fp32 [B, Hq, N] or NULL natural-log sum-exp of the scaled scores per row
 *   softmax_scale                       score scale, finite and > 0 (usually 1/sqrt(D))
 *   workspace   device scratch of at least spec_tree_attention_workspace(...) bytes, 16-byte
 *               aligned (NULL when that is 0); contents need not be initialised and are garbage
 *               afterwards
 *   status      int32 [B] or NULL       SPEC_ST_BAD_TREE / SPEC_ST_BAD_LEN / SPEC_ST_TIMEOUT (OR-ed)
 *
 * Node i, query head h sees the keys {0..L_b-1} U {L_b + j : j ancestor of i or j == i}, using KV
 * head h / (Hq/Hkv).  Supported: D in {64, 128}, Hq % Hkv == 0, Lmax >= N, B * Hkv * Lmax < 2^31.
 * q, k_cache, v_cache, out and workspace must be 16-byte aligned.  Cache slots past L_b + N are
 * never used and may hold any bits (NaN included).
 */
int spec_tree_attention(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* prefix_lens, const int32_t* tree_parent, void* out,
                        float* out_lse, int B, int N, int Hq, int Hkv, int D, int Lmax,
                        float softmax_scale, void* workspace, size_t workspace_bytes,
                        int32_t* status, void* stream);

/* ------------------------------------------------------------------------------------------------
 * Speculative-sampling verification
 * ------------------------------------------------------------------------------------------------
 * Workspace bytes spec_tree_verify needs (per-node statistics and decisions).  0 if invalid.
 */
size_t spec_tree_verify_workspace(int B, int N, int V);

/*
 * Accept/reject the draft tree of every sequence and draw its bonus token.
 *
 *   target_logits fp32 [B, N, V]  row j: target logits for the token after node j's path
 *   draft_probs   fp32 [B, N, V]  row j: draft distribution p_j the children of j were drawn from
 *                                 (already tempered by the caller); may be NULL iff temperature==0
 *   tree_tokens   int32 [B, N]    token of node i (entry 0, the root, is not read)
 *   tree_parent   int32 [B, N]
 *   uniforms      fp32 [B, N]     entry i >= 1: the test uniform r_i of node i, in [0, 1);
 *                                 entry 0: the uniform u of the bonus-token draw
 *   temperature   >= 0; q_j = softmax(l_j / T); 0 selects greedy verification
 *   out_accept_len      int32 [B]        accepted drafts (depth of the last accepted node)
 *   out_accepted_tokens int32 [B, N]     tokens on the accepted path (root excluded), -1 padded
 *   out_bonus_token     int32 [B]        token drawn where the walk stopped
 *   out_accepted_nodes  int32 [B, N] or NULL   node indices of the accepted path, -1 padded
 *   out_child_q         fp32 [B, N] or NULL    q value used in node i's own test (the current
 *                                 residual's probability of x~_i); -1 where node i was not tested
 *                                 (an earlier sibling was accepted) and at the root; at T == 0 it
 *                                 is 1 or 0 (token equals / differs from the parent's argmax)
 *   workspace     at least spec_tree_verify_workspace(B, N, V) bytes, 16-byte aligned
 *   status        int32 [B] or NULL  SPEC_ST_BAD_TREE / SPEC_ST_BAD_TOKEN / SPEC_ST_NONFINITE
 *                                 (OR-ed); target_logits, draft_probs and workspace must be 16-byte
 *                                 aligned; B <= 65535
 *
 * Tree rule (the pages give the chain form only): the children of the current node are tried in
 * ascending index against the current target distribution, which is replaced by its normalised
 * residual norm(max(0, q - p)) after each rejection (kept if that residual is all zero).  The
 * emitted tokens of the step are the accepted tokens followed by the bonus token.
 *
 * Rows read.  Small problems (B * N * V * 4 <= 64 MiB) process every node at once; large ones
 * process every internal node when out_child_q is given, and otherwise only the nodes the walk
 * reaches (the root, then each accepted child, one step per level).  Without out_child_q the small
 * form's walk starts as soon as the root's outcome is known and follows each accepted child as its
 * outcome is published; once it ends, nodes still in their residual rounds stop.  The results are
 * the same in every form.  SPEC_ST_NONFINITE reports NaN / +Inf in a row the walk depends on;
 * a non-finite row off the walk flags the sequence only when out_child_q is given (every internal
 * node is then processed in full).
 */
int spec_tree_verify(const float* target_logits, const float* draft_probs,
                     const int32_t* tree_tokens, const int32_t* tree_parent,
                     const float* uniforms, float temperature, int B, int N, int V,
                     int32_t* out_accept_len, int32_t* out_accepted_tokens,
                     int32_t* out_bonus_token, int32_t* out_accepted_nodes, float* out_child_q,
                     void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* ------------------------------------------------------------------------------------------------
 * Verification without a workspace argument
 * ------------------------------------------------------------------------------------------------
 * The pages have no counterpart to this entry point; it exists for callers that cannot allocate
 * device scratch memory -- for example a serving engine that hands all free GPU memory to its
 * KV cache at start-up and allows no cudaMalloc afterwards, or a plugin host that gives a kernel
 * only its input and output buffers.
 *
 * Same arguments, outputs and results as spec_tree_verify, minus the workspace.  The scratch lives
 * in one fixed device array inside the library (SPEC_NOALLOC_MAX_NODES * 56 bytes, 224 KB,
 * held on every GPU that loads the library until the process exits).  Calls with
 * B * N > SPEC_NOALLOC_MAX_NODES return SPEC_ERR_NOALLOC_LIMIT.  Every call made outside stream
 * capture looks up the array's device address with the caller's device current; a call made while
 * its stream is being captured reuses the last such address, so make one call on the device before
 * capturing.  All calls share the array (it keeps the last call's contents, none of which needs to
 * start at zero), so calls whose kernels may overlap on the GPU race: serialise them on one stream.
 * Allocates nothing (no cudaMalloc / cudaFree / allocating library call).
 */
#define SPEC_NOALLOC_MAX_NODES 4096
int spec_tree_verify_noalloc(const float* target_logits, const float* draft_probs,
                             const int32_t* tree_tokens, const int32_t* tree_parent,
                             const float* uniforms, float temperature, int B, int N, int V,
                             int32_t* out_accept_len, int32_t* out_accepted_tokens,
                             int32_t* out_bonus_token, int32_t* out_accepted_nodes,
                             float* out_child_q, int32_t* status, void* stream);

/* ------------------------------------------------------------------------------------------------
 * Verification against a top-k / top-p filtered target distribution
 * ------------------------------------------------------------------------------------------------
 * Survey explainer, verification taxonomy (sampling paragraph): speculative sampling carries over
 * to top-k and top-p sampling when the accept/reject test and the residual use the filtered target
 * distribution.  Reading (the pages give no procedure): per target row, temperature first, then
 * top-k on the logits (every token whose logit is >= the k-th largest is kept, ties included), then
 * top-p on the renormalised top-k distribution (token y is kept when the probability mass of the
 * tokens strictly more probable than y is < top_p; ties are kept or dropped together, the most
 * probable token always stays).  The filtered target q'_j = softmax(l_j / T) over the kept tokens,
 * renormalised, replaces q_j everywhere in spec_tree_verify's rule.  draft_probs is the drafter's
 * own distribution (filtered or not, as it sampled).
 *
 *   top_k  >= 0; 0 or >= V: no top-k filter
 *   top_p  in (0, 1]; 1: no top-p filter
 * Top-p masses come from single-precision exponentials summed exactly in 2^-40 fixed point
 * (relative error a few 1e-7), so a top_p within about 2e-6 of the mass above a tie group may
 * keep or drop that group; top-k decisions are exact.
 * At temperature 0 both filters keep the argmax, and the call is spec_tree_verify (greedy); with
 * both filters off it is spec_tree_verify as well, and needs only spec_tree_verify_workspace
 * bytes.  Otherwise the workspace must hold spec_tree_verify_filtered_workspace(B, N, V) bytes:
 * the verification scratch followed by the filtered logits (B * N * V fp32, -inf outside the kept
 * sets), written by one kernel and read by the verification kernel on the same stream.  A row of
 * target_logits holding NaN or +Inf is passed through unfiltered (verification flags it
 * SPEC_ST_NONFINITE when it reads it).
 * The other arguments, outputs and the status bits are spec_tree_verify's.
 */
size_t spec_tree_verify_filtered_workspace(int B, int N, int V);
int spec_tree_verify_filtered(const float* target_logits, const float* draft_probs,
                              const int32_t* tree_tokens, const int32_t* tree_parent,
                              const float* uniforms, float temperature, int top_k, float top_p,
                              int B, int N, int V, int32_t* out_accept_len,
                              int32_t* out_accepted_tokens, int32_t* out_bonus_token,
                              int32_t* out_accepted_nodes, float* out_child_q, void* workspace,
                              size_t workspace_bytes, int32_t* status, void* stream);

/* ------------------------------------------------------------------------------------------------
 * Dynamic draft-tree construction
 * ------------------------------------------------------------------------------------------------
 * EAGLE-3 explainer, 背景と動機 and EAGLE-2との統合: EAGLE-2 builds the draft tree at inference
 * time from the draft head's outputs instead of using a fixed shape.  The pages give no procedure;
 * this follows EAGLE-2's expand-then-rerank construction (a reading):
 *   - a drafted node's value is the sum of the draft log-probabilities log softmax(l)[token] along
 *     its path from the root, under each parent's draft logits l (root value 0);
 *   - level d expands the frontier (the root at level 1): frontier slot i's K highest draft logits
 *     (ties: lower token id) become candidates, candidate order i K + r; the K candidates of the
 *     level with the highest values (ties: lower order) are the next frontier, best first;
 *   - spec_tree_finalize returns the root plus the N - 1 best candidates of all levels (ties:
 *     shallower, then lower order), numbered by depth then candidate order, so every parent comes
 *     before its children: the tree_parent / tree_tokens that spec_tree_verify and
 *     spec_tree_attention take.
 * The draft model runs between the levels: after level d the caller drafts the frontier nodes
 * (their tokens and the slot of the row they came from are returned) and passes their logits as
 * level d + 1.
 *
 * Workspace: spec_tree_build_workspace(B, K, D) bytes, 16-byte aligned, holding each sequence's
 * construction state; level 1 starts a new construction in it.  0 if the shape is unsupported.
 * Supported: 1 <= K <= SPEC_TREE_MAX_K, 1 <= D <= 16, 1 + K + (D - 1) K^2 <= SPEC_TREE_MAX_POOL.
 */
#define SPEC_TREE_MAX_K 16
#define SPEC_TREE_MAX_POOL 2048
size_t spec_tree_build_workspace(int B, int K, int D);

/*
 * One level of the construction.
 *   draft_logits  fp32 [B, R, V], R = 1 at level 1 (the root's draft logits), else K (row i: the
 *                 draft logits at frontier slot i of the previous level).  -inf entries are
 *                 allowed (masked tokens); V >= K.
 *   level         1 .. D, called in order for each construction (a call out of order sets
 *                 SPEC_ST_BAD_TREE for every sequence and leaves the state unchanged)
 *   out_frontier_tokens       int32 [B, K] or NULL: the new frontier's tokens, best first
 *   out_frontier_parent_slot  int32 [B, K] or NULL: the row i of this level each came from
 *   status        int32 [B] or NULL: SPEC_ST_NONFINITE (NaN or +Inf in one of the sequence's rows:
 *                 its construction stops, spec_tree_finalize returns the root alone),
 *                 SPEC_ST_BAD_TREE (out-of-order level); OR-ed in
 * Draft row numbering across levels (node_row below): row 0 is the root's, row 1 + (d - 2) K + i
 * is frontier slot i's at level d >= 2.
 */
int spec_tree_expand(const float* draft_logits, int B, int V, int K, int D, int level,
                     void* workspace, size_t workspace_bytes, int32_t* out_frontier_tokens,
                     int32_t* out_frontier_parent_slot, int32_t* status, void* stream);

/*
 * The tree of the root and the N - 1 best candidates (1 <= N <= 64, N <= 1 + K + (D - 1) K^2).
 *   root_tokens     int32 [B]: token of node 0 (the last committed token)
 *   out_tree_tokens int32 [B, N], out_tree_parent int32 [B, N]: the tree, parents first; entries
 *                   past the nodes a construction produced (fewer levels run than D, or a stopped
 *                   construction) are -1
 *   out_node_row    int32 [B, N] or NULL: node j's own draft row (numbering above) if it was
 *                   expanded, else -1 -- a node with children always has one; gather those rows
 *                   for spec_tree_verify's draft_probs
 *   out_node_value  fp32 [B, N] or NULL: node values (fp32 arithmetic; log-sum-exp from a
 *                   compensated fp32 sum), NaN past the produced nodes
 */
int spec_tree_finalize(const void* workspace, size_t workspace_bytes, const int32_t* root_tokens,
                       int B, int K, int D, int N, int32_t* out_tree_tokens,
                       int32_t* out_tree_parent, int32_t* out_node_row, float* out_node_value,
                       int32_t* status, void* stream);

/* ------------------------------------------------------------------------------------------------
 * LM head fused with the statistics verification reads
 * ------------------------------------------------------------------------------------------------
 * EAGLE explainer (the target forward over the tree gives each node's next-token logits); survey
 * explainer, Formal Definition, 検証フェーズ (q_j = softmax(l_j / T); a draft token x~ is tested
 * against q_j(x~)).  Verification needs per row only m = max_y l_y, S = sum_y exp((l_y - m) / T),
 * the argmax and the logits of the tokens it tests: q_j(x~) = exp((l_x~ - m) / T) / S.  This call
 * computes logits = hidden @ weight^T on the tensor cores and reduces them on chip; the fp32 logit
 * matrix is never written.
 *   hidden      bf16 [M, H] (row-major; H a multiple of 8), 16-byte aligned
 *   weight      bf16 [V, H] (the LM head, one row per vocabulary entry), 16-byte aligned
 *   gather_idx  int32 [M, G] or NULL (G = 0): token ids whose logits to return (-1: none)
 *   temperature > 0 (for the sum only; max and argmax do not depend on it)
 *   out_max     fp32 [M] or NULL, out_sumexp fp32 [M] or NULL, out_argmax int32 [M] or NULL
 *               (lowest index among equal maxima), out_gather fp32 [M, G] (entries whose id is -1
 *               or outside [0, V) are left as they are)
 *   workspace   spec_lm_head_stats_workspace(M, V) bytes, 16-byte aligned
 *   status      int32 [1] or NULL: SPEC_ST_TIMEOUT if a bounded wait gave up (OR-ed in)
 * Precision: bf16 products accumulated in fp32 over H.  NaN / Inf inputs give unspecified results.
 */
size_t spec_lm_head_stats_workspace(int M, int V);
int spec_lm_head_stats(const void* hidden, const void* weight, const int32_t* gather_idx, int M,
                       int H, int V, int G, float temperature, float* out_max, float* out_sumexp,
                       int32_t* out_argmax, float* out_gather, void* workspace,
                       size_t workspace_bytes, int32_t* status, void* stream);

/*
 * The head in tile-major order, made once (it is a model weight): block (t, c) holds rows
 * 256 t .. 256 t + 255 and hidden elements 64 c .. 64 c + 63, contiguous, zero past V and H, so
 * that spec_lm_head_stats_packed reads every tile as one contiguous 32 KB block (the row-major head
 * gives 128-byte pieces of 256 rows).  packed: spec_lm_head_packed_bytes(V, H) bytes, 16-byte
 * aligned.  spec_lm_head_stats_packed: spec_lm_head_stats on a packed head, same results bit for
 * bit.
 */
size_t spec_lm_head_packed_bytes(int V, int H);
int spec_lm_head_pack(const void* weight, int V, int H, void* packed, size_t packed_bytes,
                      void* stream);
int spec_lm_head_stats_packed(const void* hidden, const void* packed, const int32_t* gather_idx,
                              int M, int H, int V, int G, float temperature, float* out_max,
                              float* out_sumexp, int32_t* out_argmax, float* out_gather,
                              void* workspace, size_t workspace_bytes, int32_t* status,
                              void* stream);

/*
 * Greedy verification (T = 0) from each node's argmax token: survey explainer, Formal Definition,
 * 検証フェーズ at temperature 0 -- from the root, move to the first child (ascending index) whose
 * draft token equals the argmax of the current node's target logits; stop where no child does; the
 * bonus token is the argmax there.  The results equal spec_tree_verify at temperature 0 on logits
 * with those argmaxes; with spec_lm_head_stats's out_argmax (row b * N + i = node i of sequence b)
 * no logit row is ever written.
 *   node_argmax  int32 [B, N]: the argmax of node i's target logits (lowest index among equal
 *                maxima); a value outside [0, V) at a node the walk reaches means that row had no
 *                maximum: the sequence gets SPEC_ST_NONFINITE
 *   tree_tokens, tree_parent, outputs, status: as in spec_tree_verify (out_accepted_nodes may be
 *                NULL; a flagged sequence gets accept_len = bonus = -1 and -1 rows)
 * No workspace; B <= 2^24, N <= 64.  Returns SPEC_OK or a negative spec_err_t before any launch.
 */
int spec_tree_verify_greedy(const int32_t* node_argmax, const int32_t* tree_tokens,
                            const int32_t* tree_parent, int B, int N, int V,
                            int32_t* out_accept_len, int32_t* out_accepted_tokens,
                            int32_t* out_bonus_token, int32_t* out_accepted_nodes, int32_t* status,
                            void* stream);

/*
 * Tree verification from the target's final hidden states and LM head, without the logit matrix:
 * survey explainer, Formal Definition, 検証フェーズ (child x~ of node c accepted iff
 * r < min(1, q_c(x~) / p_c(x~)); after a rejection the next sibling is tested against
 * norm(max(0, q - p_c)); the bonus token is drawn where the walk stops); EAGLE explainer (q_c is the
 * softmax of the target LM head's logits at node c).  The results are those of spec_tree_verify on
 * the logits hidden @ head^T (bf16 products, fp32 sums over H), computed as follows.  Every node's
 * max m, S = sum_y exp((l_y - m) / T) and its first child's logit come from the fused LM head
 * (spec_lm_head_stats); from the root the walk accepts first children while
 * r p(x~) S < exp((l_x~ - m) / T) (evaluated in fp64) holds; where it stops (a rejected first
 * child, or a leaf), one more pass of the LM head writes that node's full logit row and the node
 * is processed as in spec_tree_verify (its children re-tested in order from that row, residual
 * rounds, the bonus draw); an accepted child continues the walk.  Per sequence, one full row per
 * such stop, against every internal node's row for spec_tree_verify.  A first test decided from
 * the statistics can differ from spec_tree_verify's only when |r - q(x~) / p(x~)| is within the
 * rounding of S (fp32 sums: about 1e-5 relative).  At T = 0 the walk follows each node's argmax
 * (spec_tree_verify_greedy on the LM head's argmax).
 *   hidden      bf16 [B, N, H]: node i's final hidden state (the target's input to the LM head)
 *   head        bf16 [V, H] (head_packed = 0) or spec_lm_head_pack's tile-major copy (1)
 *   draft_probs, tree_tokens, tree_parent, uniforms, temperature, outputs, status: as in
 *               spec_tree_verify (out_accepted_nodes may be NULL; no per-child q); a bad draft
 *               probability is detected where it is read
 *   max_depth   >= the depth of every tree (root: 0); the call makes max_depth + 1 row passes at
 *               T > 0 (those with no node to process end after one flag read); a deeper tree is
 *               flagged SPEC_ST_BAD_TREE (T > 0)
 *   workspace   spec_tree_verify_head_workspace(B, N, H, V, max_depth) bytes, 16-byte aligned
 * H % 8 == 0; hidden, head and draft_probs 16-byte aligned; N <= 64; the V limits of
 * spec_tree_verify.  Returns SPEC_OK or a negative spec_err_t before any launch.
 */
size_t spec_tree_verify_head_workspace(int B, int N, int H, int V, int max_depth);
int spec_tree_verify_head(const void* hidden, const void* head, int head_packed,
                          const float* draft_probs, const int32_t* tree_tokens,
                          const int32_t* tree_parent, const float* uniforms, float temperature,
                          int B, int N, int H, int V, int max_depth, int32_t* out_accept_len,
                          int32_t* out_accepted_tokens, int32_t* out_bonus_token,
                          int32_t* out_accepted_nodes, void* workspace, size_t workspace_bytes,
                          int32_t* status, void* stream);

/* ------------------------------------------------------------------------------------------------
 * Tree attention over a paged KV cache
 * ------------------------------------------------------------------------------------------------
 * Survey explainer, "vLLMでの実装状況" section: serving stacks run speculative decoding on
 * PagedAttention; EAGLE explainer, vLLM usage section: the tree's nodes take extra KV-cache slots.
 * Layout (a reading; the pages give none): the cache is cut into pages of page_size slots,
 *   k_pages, v_pages  bf16 [num_pages, Hkv, page_size, D]
 *   block_table       int32 [B, max_pages]: slot s of sequence b lives in page
 *                     block_table[b][s / page_size], row s % page_size
 * Lmax = max_pages * page_size.  The other arguments, the visibility rule and the outputs are those
 * of spec_tree_attention (node i's key and value at slot L_b + i, written by the caller).  Every
 * page holding a slot below L_b + N must be a real page; otherwise the sequence gets
 * SPEC_ST_BAD_PAGE and unspecified output rows (no out-of-bounds access happens: such pages read as
 * zeros).  Table entries past the pages a sequence uses are never read for keys.
 * Supported: page_size a power of two in [16, 1024]; num_pages * Hkv * page_size < 2^31.
 * No workspace.  Returns SPEC_OK or a negative spec_err_t before any launch.
 */
int spec_tree_attention_paged(const void* q, const void* k_pages, const void* v_pages,
                              const int32_t* block_table, int page_size, int max_pages,
                              int num_pages, const int32_t* prefix_lens,
                              const int32_t* tree_parent, void* out, float* out_lse, int B, int N,
                              int Hq, int Hkv, int D, float softmax_scale, int32_t* status,
                              void* stream);

/* ------------------------------------------------------------------------------------------------
 * Post-accept KV compaction
 * ------------------------------------------------------------------------------------------------
 * After spec_tree_verify accepted the path accepted_nodes[b][0 .. accept_len[b] - 1] (node ids,
 * root excluded), commit it: the root stays at slot L_b, and slot L_b + 1 + k receives, for every
 * KV head, the key and value that slot L_b + accepted_nodes[b][k] held before the call (in place;
 * overlapping moves read the old values).  Other slots are untouched.
 *   k_cache, v_cache  bf16 [B, Hkv, Lmax, D], updated in place
 *   prefix_lens       int32 [B]  L_b
 *   accept_len        int32 [B]  from spec_tree_verify: -1 (verification failed) leaves the
 *                                sequence alone, 0 commits the root only
 *   accepted_nodes    int32 [B, N] from spec_tree_verify (out_accepted_nodes)
 *   new_prefix_lens   int32 [B] or NULL: L_b + 1 + accept_len[b] (L_b if nothing was committed);
 *                     must not alias prefix_lens (other CTAs of the call still read it)
 *   status            int32 [B] or NULL: SPEC_ST_BAD_PATH when the node ids are not strictly
 *                     increasing inside [1, N) or L_b + 1 + accept_len > Lmax (the sequence is
 *                     then left unchanged); OR-ed
 * Supported: D in {64, 128}, N <= 64, B * Hkv * Lmax < 2^31; k_cache and v_cache 16-byte aligned.
 */
int spec_kv_compact(void* k_cache, void* v_cache, const int32_t* prefix_lens,
                    const int32_t* accept_len, const int32_t* accepted_nodes,
                    int32_t* new_prefix_lens, int B, int N, int Hkv, int D, int Lmax,
                    int32_t* status, void* stream);

/* The same moves on the paged layout of spec_tree_attention_paged (any page_size >= 1 here); a
 * sequence whose table maps a moved slot outside [0, num_pages) gets SPEC_ST_BAD_PAGE and is left
 * unchanged.  Destination pages must not be shared with another sequence of the call. */
int spec_kv_compact_paged(void* k_pages, void* v_pages, const int32_t* block_table, int page_size,
                          int max_pages, int num_pages, const int32_t* prefix_lens,
                          const int32_t* accept_len, const int32_t* accepted_nodes,
                          int32_t* new_prefix_lens, int B, int N, int Hkv, int D,
                          int32_t* status, void* stream);

/* ------------------------------------------------------------------------------------------------
 * Debugging: the timeout path of the verification kernels
 * ------------------------------------------------------------------------------------------------
 * The pages have no counterpart; this exists so that tests can make a bounded device-side wait run
 * out without hanging or faulting a GPU.  Every bounded wait of the verification kernels (the row
 * copies into shared memory and the cluster exchanges of spec_tree_verify, and so of
 * spec_tree_verify_noalloc and spec_tree_verify_filtered) first polls at most `polls` times; a wait
 * that gives up there sets SPEC_ST_TIMEOUT for its sequence (whose outputs become -1) and then
 * waits for the copies and stores still in flight with the normal limit, so that nothing is left
 * in flight and the results of later calls are unaffected.  polls = 0 makes every such wait give up
 * at once; a negative value restores the normal limit (the default).  The setting is process-wide
 * and is read when a call is made: calls made before it keep theirs, a captured CUDA graph keeps
 * the value of its capture.  Always returns SPEC_OK.
 */
int spec_debug_set_verify_wait_polls(long long polls);

/* Human-readable text for a spec_err_t return value or a SPEC_ST_* bit. */
const char* spec_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* SPECTREE_H */
