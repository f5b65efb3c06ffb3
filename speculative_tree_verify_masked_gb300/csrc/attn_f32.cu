// Tree-masked attention for fp32 caches on the CUDA cores.
//
// One warp owns one (node, query head) row and walks its visible positions
// 0 .. L+d in tiles of 32 aligned at absolute position 0: lane j scores
// position 32t+j (a sequential fp32 dot product), the tile's maximum and
// probability sum are butterfly reductions (identical bits on every lane),
// and the value rows are accumulated in position order.  Everything depends
// only on the row's query and its logical key sequence, so a node verified in
// a tree and the same token decoded after its ancestors were committed give
// the same bits ("Adding a model", step 4).
#include <cmath>

#include "common.cuh"
#include "host.hpp"
#include "launchers.hpp"
#include "ptx.cuh"

namespace tv {

struct AttnF32Params {
  float* K[TV_MAX_SEQ];
  float* V[TV_MAX_SEQ];
  const float* q;
  const float* kt;
  const float* vt;
  float* out;
  const float* gate;  // output gate of the front end, or null
  const int32_t* len;
  const int32_t* node_off;
  const void* meta;
  int32_t* status;
  int n_total, n_seq, Hq, Hkv, G, cap, max_len, decode;
  float c;  // scale * log2(e)
};

template <int D>
__global__ void __launch_bounds__(128) attn_f32_kernel(const AttnF32Params p) {
  constexpr int CPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + warp;
  const int nrows = (p.decode ? p.n_seq : p.n_total) * p.Hq;
  __shared__ __align__(16) float qs[4][D];
  if (row >= nrows || status_bad(p.status)) return;
  const int node = row / p.Hq, h = row % p.Hq, g = h / p.G;
  int s = 0, off = 0, depth = 0;
  const int8_t* anc = nullptr;
  if (p.decode) {
    s = node;
  } else {
    while (s < p.n_seq - 1 && node >= p.node_off[s + 1]) s++;
    off = p.node_off[s];
    MetaView mv = meta_view(const_cast<void*>(p.meta), p.n_total);
    depth = mv.depth[node];
    anc = mv.anc_at + static_cast<size_t>(node) * TV_MAX_PATH;
  }
  const int L = p.len[s];
  if (L < 0 || L > p.max_len) {
    set_status(p.status, TV_ERR_LEN);
    return;
  }
  if (p.decode && L >= p.cap) {
    set_status(p.status, TV_ERR_CAPACITY);
    return;
  }
  const int P = L + depth + 1;  // visible positions
#pragma unroll
  for (int c = 0; c < CPL; c++) qs[warp][lane + 32 * c] = p.q[static_cast<size_t>(row) * D + lane + 32 * c];
  __syncwarp();
  const float* Kb = p.K[s] + static_cast<size_t>(g) * p.cap * D;
  const float* Vb = p.V[s] + static_cast<size_t>(g) * p.cap * D;
  float m = -INFINITY, l = 0.f;
  float acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; c++) acc[c] = 0.f;
  for (int t0 = 0; t0 < P; t0 += 32) {
    const int pos = t0 + lane;
    const bool valid = pos < P;
    const float* krow = nullptr;
    const float* vrow = nullptr;
    if (pos < L) {
      krow = Kb + static_cast<size_t>(pos) * D;
      vrow = Vb + static_cast<size_t>(pos) * D;
    } else if (valid) {
      const int tn = p.decode ? s : off + anc[pos - L];
      krow = p.kt + (static_cast<size_t>(tn) * p.Hkv + g) * D;
      vrow = p.vt + (static_cast<size_t>(tn) * p.Hkv + g) * D;
    }
    float sc = -INFINITY;
    if (valid) {
      float a = 0.f;
      for (int d = 0; d < D; d++) a = __fmaf_rn(qs[warp][d], krow[d], a);
      sc = a;
    }
    float mx = sc;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float m_new = fmaxf(m, __fmul_rn(mx, p.c));
    const float alpha = (m_new == m) ? 1.f : ex2_approx(__fsub_rn(m, m_new));
    const float pj = valid ? ex2_approx(__fmaf_rn(sc, p.c, -m_new)) : 0.f;
    float ps = pj;
#pragma unroll
    for (int o = 1; o <= 16; o <<= 1) ps = __fadd_rn(ps, __shfl_xor_sync(0xffffffffu, ps, o));
    l = __fmaf_rn(l, alpha, ps);
#pragma unroll
    for (int c = 0; c < CPL; c++) acc[c] = __fmul_rn(acc[c], alpha);
    const int nv = min(32, P - t0);
    for (int jj = 0; jj < nv; jj++) {
      const float pw = __shfl_sync(0xffffffffu, pj, jj);
      const float* vr = reinterpret_cast<const float*>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(vrow), jj));
#pragma unroll
      for (int c = 0; c < CPL; c++) acc[c] = __fmaf_rn(pw, vr[lane + 32 * c], acc[c]);
    }
    m = m_new;
  }
#pragma unroll
  for (int c = 0; c < CPL; c++) {
    const size_t oi = static_cast<size_t>(row) * D + lane + 32 * c;
    const float y = __fdiv_rn(acc[c], l);
    p.out[oi] = p.gate ? gate_mul(y, p.gate[oi]) : y;
  }
  if (p.decode && h % p.G == 0) {
    // append this token's key/value at row L of its KV head
    float* kd = p.K[s] + (static_cast<size_t>(g) * p.cap + L) * D;
    float* vd = p.V[s] + (static_cast<size_t>(g) * p.cap + L) * D;
    const float* ks = p.kt + (static_cast<size_t>(s) * p.Hkv + g) * D;
    const float* vs = p.vt + (static_cast<size_t>(s) * p.Hkv + g) * D;
#pragma unroll
    for (int c = 0; c < CPL; c++) {
      kd[lane + 32 * c] = ks[lane + 32 * c];
      vd[lane + 32 * c] = vs[lane + 32 * c];
    }
  }
}

tv_status attn_f32_launch(const AttnCall& a, cudaStream_t st) {
  const tv_attn_layer* l = a.layer;
  AttnF32Params p{};
  for (int s = 0; s < a.n_seq; s++) {
    if (!l->K[s] || !l->V[s]) return TV_ERR_ARG;
    if (!aligned16(l->K[s]) || !aligned16(l->V[s])) return TV_ERR_ALIGN;
    p.K[s] = static_cast<float*>(l->K[s]);
    p.V[s] = static_cast<float*>(l->V[s]);
  }
  p.q = static_cast<const float*>(a.q);
  p.kt = static_cast<const float*>(a.kt);
  p.vt = static_cast<const float*>(a.vt);
  p.out = static_cast<float*>(a.out);
  p.gate = static_cast<const float*>(a.gate);
  p.len = a.len;
  p.node_off = a.node_off;
  p.meta = a.meta;
  p.status = a.status;
  p.n_total = a.n_total;
  p.n_seq = a.n_seq;
  p.Hq = l->Hq;
  p.Hkv = l->Hkv;
  p.G = l->Hq / l->Hkv;
  p.cap = l->cap;
  p.max_len = a.max_len;
  p.decode = a.decode;
  p.c = a.scale * 1.4426950408889634f;
  const int nrows = (a.decode ? a.n_seq : a.n_total) * l->Hq;
  const int grid = (nrows + 3) / 4;
  switch (l->D) {
    case 64: attn_f32_kernel<64><<<grid, 128, 0, st>>>(p); break;
    case 128: attn_f32_kernel<128><<<grid, 128, 0, st>>>(p); break;
    case 256: attn_f32_kernel<256><<<grid, 128, 0, st>>>(p); break;
    default: return TV_ERR_SHAPE;
  }
  return launch_status();
}

}  // namespace tv
