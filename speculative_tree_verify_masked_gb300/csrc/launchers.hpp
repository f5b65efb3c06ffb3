// Internal launchers shared between the C-ABI entry points.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "tv.h"

namespace tv {

// Attention rows over (context + ancestors-or-self); `decode` != 0 means one
// token per sequence whose own row sits at position len[s] and is appended to
// the cache.  For verify, `meta` is the prepared tree table.
struct AttnCall {
  const tv_attn_layer* layer;
  int n_seq, n_total, n_max;
  const int32_t* node_off;
  const void* meta;
  const int32_t* len;
  int max_len;
  const void* q;
  const void* kt;
  const void* vt;
  void* out;
  float scale;
  int32_t* status;
  int decode;
  bool overlap;  // programmatic dependent launch (TV_TREE_OVERLAP)
  const void* gate = nullptr;  // [rows][Hq][D] in the KV type: out *= sigmoid(gate), or none
};

tv_status attn_f32_launch(const AttnCall& c, cudaStream_t st);
tv_status attn_tc_launch(const tv_plan* plan, const AttnCall& c, void* ws, size_t ws_bytes, cudaStream_t st);
size_t attn_tc_ws_bytes(const tv_plan* plan, const tv_attn_layer* layer, int n_seq, int n_max, int max_len);

// A front-end layer descriptor the front-end kernels accept.
bool front_layer_ok(const tv_gdn_front_layer* f);

tv_status gdn_decode_launch(const tv_gdn_layer* l, int32_t n_seq, const void* q, const void* k, const void* v,
                            const float* alpha, const float* beta, void* out, float scale, int32_t* status,
                            cudaStream_t st);

}  // namespace tv
