// Attention tree verify with its scratch in a fixed device array instead of
// a caller-supplied workspace.  The kernels are the bf16 split / tail pair of
// the ordinary entry point; only where the per-split partial states live
// differs.  The pages describe no such variant: it exists for callers that
// cannot hand over device scratch (see the declaration in tv.h).
#include <mutex>

#include "common.cuh"
#include "host.hpp"

using namespace tv;

namespace {

constexpr size_t kScratchBytes = TV_STATIC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte granularity");

// One copy per device (a __device__ variable lives in every context that
// loads this module).  Nothing in it needs to start at any value: each
// partial-state record a call reads was written earlier in the same call.
static __device__ __align__(256) float g_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ptr[kMaxDevices];

// Device address of g_scratch on the current device, looked up once per
// device (the lookup loads the module, so the first call must not be inside
// a stream capture).
tv_status scratch_ptr(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return TV_ERR_CUDA;
    g_ptr[dev] = p;
  }
  *out = g_ptr[dev];
  return TV_OK;
}

}  // namespace

extern "C" size_t tv_attn_static_scratch_bytes(void) { return kScratchBytes; }

extern "C" tv_status tv_attn_tree_verify_static(const tv_plan* plan, const tv_attn_layer* layer,
                                                const tv_tree* tree, const int32_t* len, int32_t max_len,
                                                const void* q, const void* k_t, const void* v_t, void* out,
                                                float scale, tv_stream stream) {
  if (!tree || !layer) return TV_ERR_ARG;
  // host-only size check first, so an oversized request enqueues nothing
  if (tv_attn_workspace_bytes(plan, layer, tree->n_seq, tree->n_max, max_len) > kScratchBytes)
    return TV_ERR_SCRATCH;
  void* ws = nullptr;
  const tv_status s = scratch_ptr(&ws);
  if (s != TV_OK) return s;
  return tv_attn_tree_verify(plan, layer, tree, len, max_len, q, k_t, v_t, out, scale, ws, kScratchBytes, stream);
}
