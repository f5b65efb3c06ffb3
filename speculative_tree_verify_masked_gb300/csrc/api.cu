// C-ABI entry points that dispatch on element type: attention verify and
// single-token decode, plus status strings.
#include <cmath>

#include "common.cuh"
#include "host.hpp"
#include "launchers.hpp"

#include "ptx.cuh"

using namespace tv;

namespace {

// The bounded waits of the pipelined kernels, run against barriers that
// nothing arrives at: each must give up after `limit` clocks, raise the
// shared give-up flag and let the kernel report TV_ERR_TIMEOUT.  Warp 0
// first waits on a barrier that has completed (must succeed), then on one
// that never completes with the warp-wide wait; thread 32 does the same
// with the single-thread wait; thread 64 uses the plain wait.
__global__ void __launch_bounds__(96) wait_selftest_kernel(int32_t* status, int32_t* result, long long limit) {
  __shared__ __align__(8) uint64_t bars[4];
  __shared__ int abort_flag;
  const uint32_t done_bar = smem_u32(&bars[0]), never0 = smem_u32(&bars[1]), never1 = smem_u32(&bars[2]),
                 never2 = smem_u32(&bars[3]);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; i++) mbar_init(smem_u32(&bars[i]), 1);
    abort_flag = 0;
    fence_mbar_init();
    mbar_arrive(done_bar);  // phase 0 of this one completes
  }
  __syncthreads();
  volatile int* flag = &abort_flag;
  if (threadIdx.x < 32) {
    const bool a = wait_warp(done_bar, 0, flag, limit);
    const bool b = wait_warp(never0, 0, flag, limit);
    if (threadIdx.x == 0) {
      result[0] = a ? 1 : 0;
      result[1] = b ? 1 : 0;
    }
  } else if (threadIdx.x == 32) {
    result[2] = wait_role(never1, 0, flag, limit) ? 1 : 0;
  } else if (threadIdx.x == 64) {
    result[3] = mbar_wait(never2, 0, limit) ? 1 : 0;
  }
  __syncthreads();
  if (threadIdx.x == 0 && (result[1] == 0 || result[2] == 0 || result[3] == 0)) set_status(status, TV_ERR_TIMEOUT);
}

tv_status attn_layer_check(const tv_attn_layer* l, int n_seq) {
  if (!l || !l->K || !l->V) return TV_ERR_ARG;
  if (l->dtype != TV_F32 && l->dtype != TV_BF16) return TV_ERR_DTYPE;
  if (l->Hq < 1 || l->Hkv < 1 || l->Hq % l->Hkv || l->Hq / l->Hkv > 128) return TV_ERR_SHAPE;
  if (l->D != 64 && l->D != 128 && l->D != 256) return TV_ERR_SHAPE;
  if (l->cap < 1) return TV_ERR_ARG;
  for (int s = 0; s < n_seq; s++) {
    if (!l->K[s] || !l->V[s]) return TV_ERR_ARG;
    if (!aligned16(l->K[s]) || !aligned16(l->V[s])) return TV_ERR_ALIGN;
  }
  return TV_OK;
}

}  // namespace

extern "C" const char* tv_status_string(tv_status s) {
  switch (s) {
    case TV_OK: return "ok";
    case TV_ERR_ARG: return "invalid argument";
    case TV_ERR_SHAPE: return "unsupported shape";
    case TV_ERR_DTYPE: return "unsupported element type";
    case TV_ERR_ALIGN: return "pointer not 16-byte aligned";
    case TV_ERR_TREE: return "malformed draft tree";
    case TV_ERR_CAPACITY: return "cache capacity exceeded";
    case TV_ERR_CUDA: return "CUDA runtime error";
    case TV_ERR_WORKSPACE: return "workspace too small";
    case TV_ERR_TIMEOUT: return "bounded device wait expired";
    case TV_ERR_LEN: return "sequence length above max_len";
    case TV_ERR_SCRATCH: return "request exceeds the fixed static scratch (TV_STATIC_SCRATCH_BYTES)";
  }
  return "unknown status";
}

extern "C" const char* tv_version(void) { return "treeverify 0.1 (sm_103a)"; }

extern "C" size_t tv_attn_workspace_bytes(const tv_plan* plan, const tv_attn_layer* layer, int32_t n_seq,
                                          int32_t n_max, int32_t max_len) {
  if (!layer || layer->dtype != TV_BF16) return 0;
  return attn_tc_ws_bytes(plan, layer, n_seq, n_max, max_len);
}

extern "C" tv_status tv_attn_tree_verify(const tv_plan* plan, const tv_attn_layer* l, const tv_tree* t,
                                         const int32_t* len, int32_t max_len, const void* q, const void* k_t,
                                         const void* v_t, void* out, float scale, void* ws, size_t ws_bytes,
                                         tv_stream stream) {
  if (!tree_ok(t) || !len || !q || !k_t || !v_t || !out) return TV_ERR_ARG;
  const tv_status ls = attn_layer_check(l, t->n_seq);
  if (ls != TV_OK) return ls;
  if (max_len < 0 || max_len > l->cap || !(scale > 0.f) || !std::isfinite(scale)) return TV_ERR_ARG;
  if (!aligned16(len) || !aligned16(q) || !aligned16(k_t) || !aligned16(v_t) || !aligned16(out)) return TV_ERR_ALIGN;
  AttnCall c{l, t->n_seq, t->n_total, t->n_max, t->node_off, t->meta, len, max_len, q, k_t, v_t, out, scale,
             t->status, 0, tree_overlap(t)};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (l->dtype == TV_F32) return attn_f32_launch(c, st);
  return attn_tc_launch(plan, c, ws, ws_bytes, st);
}

extern "C" tv_status tv_decode_step(const tv_plan* plan, const tv_attn_layer* attn, const tv_gdn_layer* gdn,
                                    int32_t n_seq, const int32_t* len, int32_t max_len, const void* q, const void* k,
                                    const void* v, const float* alpha, const float* beta, void* out, float scale,
                                    void* ws, size_t ws_bytes, int32_t* status, tv_stream stream) {
  if ((attn == nullptr) == (gdn == nullptr)) return TV_ERR_ARG;
  if (n_seq < 1 || n_seq > TV_MAX_SEQ || !status || !q || !k || !v || !out) return TV_ERR_ARG;
  if (!aligned16(status)) return TV_ERR_ALIGN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (gdn) return gdn_decode_launch(gdn, n_seq, q, k, v, alpha, beta, out, scale, status, st);
  const tv_status ls = attn_layer_check(attn, n_seq);
  if (ls != TV_OK) return ls;
  if (!len || max_len < 0 || max_len > attn->cap || !(scale > 0.f) || !std::isfinite(scale)) return TV_ERR_ARG;
  if (!aligned16(len) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return TV_ERR_ALIGN;
  AttnCall c{attn, n_seq, n_seq, 1, nullptr, nullptr, len, max_len, q, k, v, out, scale, status, 1, false};
  if (attn->dtype == TV_F32) return attn_f32_launch(c, st);
  return attn_tc_launch(plan, c, ws, ws_bytes, st);
}

extern "C" tv_status tv_attn_tree_verify_gated(const tv_plan* plan, const tv_attn_layer* l, const tv_tree* t,
                                               const int32_t* len, int32_t max_len, const void* q, const void* k_t,
                                               const void* v_t, const void* gate, void* out, float scale, void* ws,
                                               size_t ws_bytes, tv_stream stream) {
  if (!tree_ok(t) || !len || !q || !k_t || !v_t || !gate || !out) return TV_ERR_ARG;
  const tv_status ls = attn_layer_check(l, t->n_seq);
  if (ls != TV_OK) return ls;
  if (max_len < 0 || max_len > l->cap || !(scale > 0.f) || !std::isfinite(scale)) return TV_ERR_ARG;
  if (!aligned16(len) || !aligned16(q) || !aligned16(k_t) || !aligned16(v_t) || !aligned16(gate) || !aligned16(out))
    return TV_ERR_ALIGN;
  AttnCall c{l, t->n_seq, t->n_total, t->n_max, t->node_off, t->meta, len, max_len, q, k_t, v_t, out, scale,
             t->status, 0, tree_overlap(t), gate};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (l->dtype == TV_F32) return attn_f32_launch(c, st);
  return attn_tc_launch(plan, c, ws, ws_bytes, st);
}

extern "C" tv_status tv_attn_decode_gated(const tv_plan* plan, const tv_attn_layer* attn, int32_t n_seq,
                                          const int32_t* len, int32_t max_len, const void* q, const void* k,
                                          const void* v, const void* gate, void* out, float scale, void* ws,
                                          size_t ws_bytes, int32_t* status, tv_stream stream) {
  if (n_seq < 1 || n_seq > TV_MAX_SEQ || !status || !q || !k || !v || !gate || !out || !len) return TV_ERR_ARG;
  if (!aligned16(status)) return TV_ERR_ALIGN;
  const tv_status ls = attn_layer_check(attn, n_seq);
  if (ls != TV_OK) return ls;
  if (max_len < 0 || max_len > attn->cap || !(scale > 0.f) || !std::isfinite(scale)) return TV_ERR_ARG;
  if (!aligned16(len) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(gate) || !aligned16(out))
    return TV_ERR_ALIGN;
  AttnCall c{attn, n_seq, n_seq, 1, nullptr, nullptr, len, max_len, q, k, v, out, scale, status, 1, false, gate};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (attn->dtype == TV_F32) return attn_f32_launch(c, st);
  return attn_tc_launch(plan, c, ws, ws_bytes, st);
}

extern "C" tv_status tv_wait_selftest(int32_t* status, int32_t* result, int64_t limit_cycles, tv_stream stream) {
  if (!status || !result || limit_cycles < 1 || limit_cycles > kWaitCycles) return TV_ERR_ARG;
  if (!aligned16(status) || !aligned16(result)) return TV_ERR_ALIGN;
  wait_selftest_kernel<<<1, 96, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status, result, limit_cycles);
  return launch_status();
}
