// Attention tree verify with its scratch in a fixed device array instead of
// a caller-supplied workspace.  The kernels are the bf16 split / tail pair of
// the ordinary entry point; only where the per-split partial states live
// differs.  The pages describe no such variant: it exists for callers that
// cannot hand over device scratch (see the declaration in tv.h).
#include <cuda.h>
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
struct Cached {
  void* ptr;
  unsigned long long ctx_id;  // context the address belongs to (0: not known)
};
Cached g_cache[kMaxDevices];

// Id of the calling thread's current context, through the driver's entry
// points (the library does not link the driver); 0 when unavailable.
unsigned long long current_ctx_id() {
  typedef CUresult (*GetCurrent)(CUcontext*);
  typedef CUresult (*GetId)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
    cudaGetLastError();
    looked_up = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_scratch on the current device.  Looked up once per
// device and context: a device reset (cudaDeviceReset) makes a new context,
// and the address is looked up again there.  The first lookup loads the
// module, so the first call on a device must not be inside a stream capture.
tv_status scratch_ptr(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return TV_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  // cudaGetDevice does not create the context; the symbol lookup does, so a
  // first call reads the id after its lookup
  const unsigned long long ctx = current_ctx_id();
  Cached& c = g_cache[dev];
  if (!c.ptr || (ctx != 0 && c.ctx_id != ctx)) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
      cudaGetLastError();  // the next call of any entry point starts clean
      c.ptr = nullptr;
      return TV_ERR_CUDA;
    }
    c.ptr = p;
    c.ctx_id = current_ctx_id();
  }
  *out = c.ptr;
  return TV_OK;
}

}  // namespace

extern "C" size_t tv_attn_static_scratch_bytes(void) { return kScratchBytes; }

extern "C" tv_status tv_attn_tree_verify_static(const tv_plan* plan, const tv_attn_layer* layer,
                                                const tv_tree* tree, const int32_t* len, int32_t max_len,
                                                const void* q, const void* k_t, const void* v_t, void* out,
                                                float scale, tv_stream stream) {
  // an ill-formed tree or length bound is an argument error, as for the
  // workspace call; the size check below reads n_seq, n_max and max_len
  if (!tree_ok(tree) || !layer || max_len < 0) return TV_ERR_ARG;
  // host-only size check next, so an oversized request enqueues nothing
  if (tv_attn_workspace_bytes(plan, layer, tree->n_seq, tree->n_max, max_len) > kScratchBytes)
    return TV_ERR_SCRATCH;
  void* ws = nullptr;
  const tv_status s = scratch_ptr(&ws);
  if (s != TV_OK) return s;
  return tv_attn_tree_verify(plan, layer, tree, len, max_len, q, k_t, v_t, out, scale, ws, kScratchBytes, stream);
}
