// Gated DeltaNet front end and output norm ("Adding a model", "What is still
// specific to Qwen3.8": the Gated DeltaNet layer with its gated norm; "The
// model layer": per-sequence state includes the convolution tails).
//
// Channels are the layer's raw query, key and value projections side by
// side: C = 2 Hk dk + Hv dv per token.
//   * short convolution: depthwise and causal, width W.  A token's output at
//     channel c is sum_j w[c][j] x[t - (W-1) + j][c] over the token's root
//     path, continuing past the root into the committed tail (the last W-1
//     inputs of the context, oldest first); then SiLU.  A tree node at depth
//     d reads window element j from its ancestor at depth d + j - (W-1), or
//     from tail row d + j while that depth is negative: exactly the inputs
//     decoding its root path token by token would read.
//   * q and k: divided per head by sqrt(sum of squares + 1e-6).
//   * gates: beta = sigmoid(b_raw), alpha = exp(-softplus(a_raw)).
//   * output: o / sqrt(mean(o^2) + 1e-6) * w_norm * SiLU(z).
// Every value is formed in fp32 in a fixed order (the window in j order, the
// sums of squares per lane in channel order then a butterfly), so a verified
// row and the same token decoded later get the same bits.
#include <cmath>

#include "common.cuh"
#include "front_gdn.cuh"
#include "host.hpp"
#include "launchers.hpp"

namespace tv {

struct GdnFrontParams {
  const void* x;
  const float* a_raw;
  const float* b_raw;
  void* q;
  void* k;
  void* v;
  float* alpha;
  float* beta;
  const float* wconv;
  const void* tail[TV_MAX_SEQ];
  const int32_t* node_off;
  const void* meta;
  int32_t* status;
  int n_rows, n_seq, n_total, Hk, Hv, dk, dv, W, decode;
};

// One warp per (row, head unit): units 0..Hk-1 are query heads, Hk..2Hk-1
// key heads, then Hv value heads; the last warps of the grid do the gates.
template <typename T, int DH>
__global__ void __launch_bounds__(128) gdn_front_kernel(const GdnFrontParams p) {
  constexpr int CPL = DH / 32;  // channels per lane
  const int warp = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  const int units = 2 * p.Hk + p.Hv;
  const int C = 2 * p.Hk * p.dk + p.Hv * p.dv;
  if (status_bad(p.status)) return;
  if (warp >= p.n_rows * units) {
    // gates: one thread per (row, value head)
    const int gi = (warp - p.n_rows * units) * 32 + lane;
    if (gi < p.n_rows * p.Hv) front_gates(p.a_raw[gi], p.b_raw[gi], p.alpha[gi], p.beta[gi]);
    return;
  }
  const int row = warp / units, u = warp % units;
  int s = row, depth = 0, off = row;
  const int8_t* anc = nullptr;
  if (!p.decode) {
    s = 0;
    while (s < p.n_seq - 1 && row >= p.node_off[s + 1]) s++;
    off = p.node_off[s];
    const MetaView mv = meta_view(const_cast<void*>(p.meta), p.n_total);
    depth = mv.depth[row];
    anc = mv.anc_at + static_cast<size_t>(row) * TV_MAX_PATH;
  }
  const int c0 = u < 2 * p.Hk ? u * p.dk : 2 * p.Hk * p.dk + (u - 2 * p.Hk) * p.dv;
  const T* x = static_cast<const T*>(p.x);
  const T* tail = static_cast<const T*>(p.tail[s]);
  // the rows of the window: node rows (global) or tail rows (negative: -1 - r)
  int src[kMaxConvWidth];
  conv_window(src, p.W, depth, off, anc, row);
  float val[CPL];
#pragma unroll
  for (int e = 0; e < CPL; e++) val[e] = conv_silu(x, tail, p.wconv, C, p.W, src, c0 + lane + 32 * e);
  T* dst;
  float scale = 1.f;
  if (u < 2 * p.Hk) {
    scale = warp_l2_scale<CPL>(val);
    const int hk = u < p.Hk ? u : u - p.Hk;
    dst = static_cast<T*>(u < p.Hk ? p.q : p.k) + (static_cast<size_t>(row) * p.Hk + hk) * p.dk;
  } else {
    dst = static_cast<T*>(p.v) + (static_cast<size_t>(row) * p.Hv + (u - 2 * p.Hk)) * p.dv;
  }
#pragma unroll
  for (int e = 0; e < CPL; e++) dst[lane + 32 * e] = from_f32<T>(u < 2 * p.Hk ? __fmul_rn(val[e], scale) : val[e]);
}

// Gated RMS norm: one warp per (row, value head).
template <typename T, int DV>
__global__ void __launch_bounds__(128) gdn_out_norm_kernel(const void* o_, const void* z_, const float* w_norm,
                                                           void* out_, int n_units) {
  constexpr int CPL = DV / 32;
  const int warp = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  if (warp >= n_units) return;
  const T* o = static_cast<const T*>(o_) + static_cast<size_t>(warp) * DV;
  const T* z = static_cast<const T*>(z_) + static_cast<size_t>(warp) * DV;
  T* out = static_cast<T*>(out_) + static_cast<size_t>(warp) * DV;
  float ov[CPL], zv[CPL], wn[CPL];
#pragma unroll
  for (int e = 0; e < CPL; e++) {
    ov[e] = to_f32(o[lane + 32 * e]);
    zv[e] = to_f32(z[lane + 32 * e]);
    wn[e] = w_norm[lane + 32 * e];
  }
  gated_norm_vals<T, CPL>(ov, zv, wn, out, lane);
}

struct ConvCommitParams {
  void* tail[TV_MAX_SEQ];
  const void* x;
  const int32_t* path;
  const int32_t* acc_len;
  const int32_t* node_off;
  int32_t* status;
  int C, W, decode;
};

// One thread per (sequence, channel): the last W-1 of (old tail, new inputs).
template <typename T>
__global__ void __launch_bounds__(256) gdn_conv_commit_kernel(const ConvCommitParams p) {
  const int s = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= p.C || status_bad(p.status)) return;
  const int W1 = p.W - 1;
  T* tail = static_cast<T*>(p.tail[s]);
  const T* x = static_cast<const T*>(p.x);
  const int a = p.decode ? 1 : p.acc_len[s];
  if (a < 1 || a > TV_MAX_PATH) return;
  T seq[kMaxConvWidth - 1 + TV_MAX_PATH];
  for (int r = 0; r < W1; r++) seq[r] = tail[static_cast<size_t>(r) * p.C + c];
  for (int j = 0; j < a; j++) {
    const int node = p.decode ? s : p.node_off[s] + p.path[s * TV_MAX_PATH + j];
    seq[W1 + j] = x[static_cast<size_t>(node) * p.C + c];
  }
  for (int r = 0; r < W1; r++) tail[static_cast<size_t>(r) * p.C + c] = seq[a + r];
}

bool front_layer_ok(const tv_gdn_front_layer* f) {
  return f && (f->dtype == TV_F32 || f->dtype == TV_BF16) && f->Hk >= 1 && f->Hv >= 1 &&
         (f->dk == 64 || f->dk == 128) && f->dv == f->dk && f->width >= 1 && f->width <= kMaxConvWidth &&
         f->wconv && f->tail;
}

}  // namespace tv

using namespace tv;

extern "C" tv_status tv_gdn_front(const tv_gdn_front_layer* f, const tv_tree* t, int32_t n_seq, const void* x,
                                  const float* a_raw, const float* b_raw, void* q, void* k, void* v, float* alpha,
                                  float* beta, int32_t* status, tv_stream stream) {
  if (!f || !x || !a_raw || !b_raw || !q || !k || !v || !alpha || !beta) return TV_ERR_ARG;
  if (f->dtype != TV_F32 && f->dtype != TV_BF16) return TV_ERR_DTYPE;
  if (!front_layer_ok(f)) return TV_ERR_SHAPE;
  GdnFrontParams p{};
  if (t) {
    if (!tree_ok(t)) return TV_ERR_ARG;
    p.n_rows = t->n_total;
    p.n_seq = t->n_seq;
    p.n_total = t->n_total;
    p.node_off = t->node_off;
    p.meta = t->meta;
    p.status = t->status;
  } else {
    if (n_seq < 1 || n_seq > TV_MAX_SEQ || !status) return TV_ERR_ARG;
    if (!aligned16(status)) return TV_ERR_ALIGN;
    p.n_rows = n_seq;
    p.n_seq = n_seq;
    p.status = status;
    p.decode = 1;
  }
  for (int s = 0; s < p.n_seq; s++) {
    if (f->width > 1 && !f->tail[s]) return TV_ERR_ARG;
    p.tail[s] = f->tail[s];
  }
  p.x = x; p.a_raw = a_raw; p.b_raw = b_raw; p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta;
  p.wconv = f->wconv;
  p.Hk = f->Hk; p.Hv = f->Hv; p.dk = f->dk; p.dv = f->dv; p.W = f->width;
  const int warps = p.n_rows * (2 * f->Hk + f->Hv) + (p.n_rows * f->Hv + 31) / 32;
  const int grid = (warps + 3) / 4;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool bf = f->dtype == TV_BF16;
  if (f->dk == 128) {
    if (bf) gdn_front_kernel<__nv_bfloat16, 128><<<grid, 128, 0, st>>>(p); else gdn_front_kernel<float, 128><<<grid, 128, 0, st>>>(p);
  } else {
    if (bf) gdn_front_kernel<__nv_bfloat16, 64><<<grid, 128, 0, st>>>(p); else gdn_front_kernel<float, 64><<<grid, 128, 0, st>>>(p);
  }
  return launch_status();
}

extern "C" tv_status tv_gdn_out_norm(const tv_gdn_front_layer* f, int32_t rows, const void* o, const void* z,
                                     const float* w_norm, void* out, tv_stream stream) {
  if (!f || !o || !z || !w_norm || !out || rows < 0) return TV_ERR_ARG;
  if (f->dtype != TV_F32 && f->dtype != TV_BF16) return TV_ERR_DTYPE;
  if (f->dv != 64 && f->dv != 128) return TV_ERR_SHAPE;
  if (rows == 0) return TV_OK;
  const int units = rows * f->Hv;
  const int grid = (units + 3) / 4;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool bf = f->dtype == TV_BF16;
  if (f->dv == 128) {
    if (bf) gdn_out_norm_kernel<__nv_bfloat16, 128><<<grid, 128, 0, st>>>(o, z, w_norm, out, units);
    else gdn_out_norm_kernel<float, 128><<<grid, 128, 0, st>>>(o, z, w_norm, out, units);
  } else {
    if (bf) gdn_out_norm_kernel<__nv_bfloat16, 64><<<grid, 128, 0, st>>>(o, z, w_norm, out, units);
    else gdn_out_norm_kernel<float, 64><<<grid, 128, 0, st>>>(o, z, w_norm, out, units);
  }
  return launch_status();
}

extern "C" tv_status tv_gdn_conv_commit(const tv_gdn_front_layer* f, const tv_tree* t, int32_t n_seq, const void* x,
                                        const int32_t* path, const int32_t* acc_len, int32_t* status,
                                        tv_stream stream) {
  if (!f || !x) return TV_ERR_ARG;
  if (f->dtype != TV_F32 && f->dtype != TV_BF16) return TV_ERR_DTYPE;
  if (!front_layer_ok(f)) return TV_ERR_SHAPE;
  ConvCommitParams p{};
  if (t) {
    if (!tree_ok(t) || !path || !acc_len) return TV_ERR_ARG;
    n_seq = t->n_seq;
    p.node_off = t->node_off;
    p.path = path;
    p.acc_len = acc_len;
    p.status = t->status;
  } else {
    if (n_seq < 1 || n_seq > TV_MAX_SEQ || !status) return TV_ERR_ARG;
    p.status = status;
    p.decode = 1;
  }
  if (f->width == 1) return TV_OK;  // no tail
  for (int s = 0; s < n_seq; s++) {
    if (!f->tail[s]) return TV_ERR_ARG;
    p.tail[s] = f->tail[s];
  }
  p.x = x;
  p.C = 2 * f->Hk * f->dk + f->Hv * f->dv;
  p.W = f->width;
  const dim3 grid((p.C + 255) / 256, n_seq);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (f->dtype == TV_BF16) gdn_conv_commit_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(p);
  else gdn_conv_commit_kernel<float><<<grid, 256, 0, st>>>(p);
  return launch_status();
}
