// Attention front end: rotary position embedding of the tree's queries and
// keys at each row's logical position ("Adding a model", "What is still
// specific to Qwen3.8": attention with partial rotary).
//
// A tree node at depth d sits at logical position L + d, where decoding its
// root path token by token would have put it; a decode token sits at L.  The
// first rot_dims dimensions of each head turn as rot_dims / 2 planes: plane
// j pairs dimension j with j + rot_dims / 2 and turns by the angle
// pos * theta^(-2j / rot_dims); the other dimensions pass through.  The
// angle and its sine and cosine are formed in fp64 (positions reach 2^17 and
// more, where an fp32 angle would be off by ~1e-2 rad), the rotation in
// fp32, the result rounded to the row type.  A row's bits depend only on its
// input row and its position, so a verified row and the same token decoded
// later are rotated identically.
#include <cmath>

#include "common.cuh"
#include "host.hpp"

namespace tv {

struct RopeParams {
  const void* q_raw;
  const void* k_raw;
  void* q;
  void* k;
  const int32_t* len;
  const int32_t* node_off;
  const void* meta;
  int32_t* status;
  int n_rows;  // nodes (verify) or sequences (decode)
  int n_seq, n_total, Hq, Hkv, D, rot, max_len, decode;
  double theta;
};

template <typename T>
__global__ void __launch_bounds__(128) rope_kernel(const RopeParams p) {
  const int warp = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  const int H = p.Hq + p.Hkv;
  if (warp >= p.n_rows * H || status_bad(p.status)) return;
  const int node = warp / H, hh = warp % H;
  int s = node, depth = 0;
  if (!p.decode) {
    s = 0;
    while (s < p.n_seq - 1 && node >= p.node_off[s + 1]) s++;
    const MetaView mv = meta_view(const_cast<void*>(p.meta), p.n_total);
    depth = mv.depth[node];
  }
  const int L = p.len[s];
  if (L < 0 || L > p.max_len) {
    if (lane == 0) set_status(p.status, TV_ERR_LEN);
    return;
  }
  const double pos = static_cast<double>(L + depth);
  const bool is_q = hh < p.Hq;
  const size_t row = is_q ? static_cast<size_t>(node) * p.Hq + hh : static_cast<size_t>(node) * p.Hkv + (hh - p.Hq);
  const T* src = static_cast<const T*>(is_q ? p.q_raw : p.k_raw) + row * p.D;
  T* dst = static_cast<T*>(is_q ? p.q : p.k) + row * p.D;
  const int half = p.rot / 2;
  // each lane reads both halves of its planes before writing them, so the
  // rotation may run in place
  for (int j = lane; j < half; j += 32) {
    const double ang = pos * pow(p.theta, -2.0 * j / p.rot);
    double sn, cs;
    sincos(ang, &sn, &cs);
    const float c = static_cast<float>(cs), sf = static_cast<float>(sn);
    const float a = to_f32(src[j]), b = to_f32(src[j + half]);
    const float ra = __fmaf_rn(a, c, -__fmul_rn(b, sf));
    const float rb = __fmaf_rn(b, c, __fmul_rn(a, sf));
    dst[j] = from_f32<T>(ra);
    dst[j + half] = from_f32<T>(rb);
  }
  if (dst != src)
    for (int j = p.rot + lane; j < p.D; j += 32) dst[j] = src[j];
}

}  // namespace tv

using namespace tv;

extern "C" tv_status tv_attn_rope(const tv_attn_layer* l, const tv_tree* t, int32_t n_seq, const int32_t* len,
                                  int32_t max_len, int32_t rot_dims, float theta, const void* q_raw,
                                  const void* k_raw, void* q, void* k, int32_t* status, tv_stream stream) {
  if (!l || !len || !q_raw || !k_raw || !q || !k) return TV_ERR_ARG;
  if (l->dtype != TV_F32 && l->dtype != TV_BF16) return TV_ERR_DTYPE;
  if (l->Hq < 1 || l->Hkv < 1 || l->Hq % l->Hkv || (l->D != 64 && l->D != 128 && l->D != 256)) return TV_ERR_SHAPE;
  if (rot_dims < 0 || rot_dims > l->D || rot_dims % 2 || !(theta > 1.f) || !std::isfinite(theta)) return TV_ERR_ARG;
  if (max_len < 0 || max_len > l->cap) return TV_ERR_ARG;
  if (!aligned16(len) || !aligned16(q_raw) || !aligned16(k_raw) || !aligned16(q) || !aligned16(k)) return TV_ERR_ALIGN;
  RopeParams p{};
  if (t) {
    if (!tree_ok(t)) return TV_ERR_ARG;
    p.n_rows = t->n_total;
    p.n_seq = t->n_seq;
    p.n_total = t->n_total;
    p.node_off = t->node_off;
    p.meta = t->meta;
    p.status = t->status;
    p.decode = 0;
  } else {
    if (n_seq < 1 || n_seq > TV_MAX_SEQ || !status) return TV_ERR_ARG;
    if (!aligned16(status)) return TV_ERR_ALIGN;
    p.n_rows = n_seq;
    p.n_seq = n_seq;
    p.status = status;
    p.decode = 1;
  }
  p.q_raw = q_raw;
  p.k_raw = k_raw;
  p.q = q;
  p.k = k;
  p.len = len;
  p.Hq = l->Hq;
  p.Hkv = l->Hkv;
  p.D = l->D;
  p.rot = rot_dims;
  p.max_len = max_len;
  p.theta = static_cast<double>(theta);
  const int warps = p.n_rows * (l->Hq + l->Hkv);
  const int grid = (warps + 3) / 4;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (l->dtype == TV_BF16) rope_kernel<__nv_bfloat16><<<grid, 128, 0, st>>>(p);
  else rope_kernel<float><<<grid, 128, 0, st>>>(p);
  return launch_status();
}
