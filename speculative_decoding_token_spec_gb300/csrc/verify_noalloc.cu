// spec_tree_verify_noalloc: tree verification without a caller-provided workspace.
//
// Some callers cannot hand the library device scratch memory.  Examples: a serving engine that
// reserves all free GPU memory for its KV cache at start-up and forbids cudaMalloc afterwards, or
// a plugin host that passes a kernel only its input and output buffers.  For them this entry point
// keeps the per-node statistics and arrival counters that spec_tree_verify otherwise writes to its
// workspace in one fixed, file-scope device array instead.
//
// Properties of that array:
//   * Size: room for B * N <= SPEC_NOALLOC_MAX_NODES tree nodes per call (224 KB).  Every
//     GPU on which the library is loaded holds it until the process exits.
//   * Set-up: every call made outside stream capture looks up the array's device address
//     (cudaGetSymbolAddress, a host-side lookup) with the caller's device current, so a module
//     that was reloaded at another address (after cudaDeviceReset, say) is followed.  A call made
//     while its stream is being captured uses the address of the last uncaptured call on that
//     device (looking it up if there was none); make one call before capturing.
//   * Sharing: all calls share the one array and it keeps the previous call's contents.  Nothing in
//     it has to start at zero: each call writes every statistics entry it reads, a per-sequence
//     arrival counter is trusted only when it carries the generation and tag of the call itself,
//     and a hand-over or walk-done word only when it carries the call's generation, so counts,
//     node records and words left by earlier calls are reset or ignored.  Calls whose
//     kernels may overlap on the GPU (different streams, or concurrent host threads) race on it.
//   * No allocation: no cudaMalloc, cudaFree or allocating library routine is called.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "spectree.h"

using namespace spectree;

namespace {

// per node: its statistics record and hand-over word; per sequence (B <= B * N): an arrival
// counter and a walk-done word
constexpr size_t kPerNode = sizeof(NodeStat) + 3 * sizeof(unsigned long long);
constexpr size_t kScratchBytes = (size_t)SPEC_NOALLOC_MAX_NODES * kPerNode;

// The fixed scratch.  In host code `g_verify_scratch` names a host-side stand-in, not device
// memory: its device address must come from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_verify_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device: looked up on every call outside
// stream capture, the last such address reused while `stream` is being captured.
int scratch_on_current_device(cudaStream_t stream, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  const bool capturing =
      cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!capturing || g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_verify_scratch);
    if (e != cudaSuccess || p == nullptr) return SPEC_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SPEC_OK;
}

}  // namespace

extern "C" int spec_tree_verify_noalloc(const float* target_logits, const float* draft_probs,
                                        const int32_t* tree_tokens, const int32_t* tree_parent,
                                        const float* uniforms, float temperature, int B, int N,
                                        int V, int32_t* out_accept_len,
                                        int32_t* out_accepted_tokens, int32_t* out_bonus_token,
                                        int32_t* out_accepted_nodes, float* out_child_q,
                                        int32_t* status, void* stream) {
  if (B < 1 || N < 1 || N > kMaxNodes) return SPEC_ERR_INVALID_ARG;
  if ((long long)B * N > SPEC_NOALLOC_MAX_NODES) return SPEC_ERR_NOALLOC_LIMIT;
  void* scratch = nullptr;
  int rc = scratch_on_current_device(static_cast<cudaStream_t>(stream), &scratch);
  if (rc != SPEC_OK) return rc;
  return spec_tree_verify(target_logits, draft_probs, tree_tokens, tree_parent, uniforms,
                          temperature, B, N, V, out_accept_len, out_accepted_tokens,
                          out_bonus_token, out_accepted_nodes, out_child_q, scratch,
                          kScratchBytes, status, stream);
}
