// Gated DeltaNet tree verify and single-token decode.
//
// Tree verify ("Adding a model", Gated DeltaNet layers; the gated delta rule
// applied along every node's root path): one CTA owns 16 state rows of one
// value head of one sequence and walks the tree in the order prepared by
// tv_tree_prepare.  A lane group of LPR lanes holds two state rows (the
// token's key and query are read once for both, and the two rows give two
// independent dependency chains); the few states that must outlive a subtree
// sit in shared-memory slots.  No per-node state is written to memory: the
// kernel reads the committed state once and writes one output value per
// (node, row).
//
// Work per (node, row): two dot products of length dk (s.k, s.q) and, for
// nodes with children, one rank-1 update of the row, in packed fp32x2
// arithmetic.  The kernel is bound by latency and shared-memory bandwidth,
// not by the 4 * Hv * dv * dk bytes of state it reads.
#include "common.cuh"
#include "gdn_step.cuh"
#include "host.hpp"
#include "launchers.hpp"

namespace tv {

constexpr int kGdnThreads = 64;

struct GdnVerifyParams {
  float* S[TV_MAX_SEQ];
  const void* q;
  const void* k;
  const void* v;
  const float* alpha;
  const float* beta;
  void* out;
  const void* meta;
  int32_t* status;
  int n_total, n_max, n_slots, Hk, Hv, dv;
  float scale;
};

// Slots for states that must outlive a subtree: at most floor(log2(n / 5)) + 1
// for a tree of n nodes (see tree.cu).
inline int slots_for(int n_max) {
  int k = 1;
  while ((5 << k) <= n_max) k++;
  return k;
}

template <int LPR>
struct GdnShape {
  static constexpr int DK = 16 * LPR;           // key dim
  static constexpr int NG = kGdnThreads / LPR;  // lane groups per CTA
  static constexpr int R = 2 * NG;              // state rows per CTA (two per group)
};

template <int LPR>
inline size_t gdn_verify_smem(int n_max, int n_slots) {
  using Sh = GdnShape<LPR>;
  const size_t n = static_cast<size_t>(n_max);
  return (2 * n * Sh::DK + 4 * n + n * Sh::R + static_cast<size_t>(n_slots) * Sh::R * Sh::DK) * 4 + 4 * n;
}

// Stage the tree's keys and queries (this CTA's key head, fp32), the values at
// this CTA's rows, alpha and beta of this value head and the traversal.
// Every load of a thread is issued before any of them is used.
template <typename T, int DK, int R>
__device__ __forceinline__ void stage_node_inputs(const GdnVerifyParams& p, const MetaView& mv, int n, int off, int g,
                                                  int h, int rb, float* kb, float* qb, float4* nc, float* vb,
                                                  int* sch) {
  constexpr int EPL = 16 / sizeof(T);  // elements per 16-byte load
  constexpr int CPR = DK / EPL;        // 16-byte chunks per key row
  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  const T* v = static_cast<const T*>(p.v);
  const int nchunks = n * CPR;
  for (int base = threadIdx.x; base < nchunks; base += 4 * blockDim.x) {
    uint4 kv[4], qv[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int idx = base + u * blockDim.x;
      if (idx < nchunks) {
        const size_t src = (static_cast<size_t>(off + idx / CPR) * p.Hk + g) * DK + (idx % CPR) * EPL;
        kv[u] = *reinterpret_cast<const uint4*>(k + src);
        qv[u] = *reinterpret_cast<const uint4*>(q + src);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int idx = base + u * blockDim.x;
      if (idx < nchunks) {
        const T* ke = reinterpret_cast<const T*>(&kv[u]);
        const T* qe = reinterpret_cast<const T*>(&qv[u]);
        float* kd = kb + (idx / CPR) * DK + (idx % CPR) * EPL;
        float* qd = qb + (idx / CPR) * DK + (idx % CPR) * EPL;
#pragma unroll
        for (int e = 0; e < EPL; e++) {
          kd[e] = to_f32(ke[e]);
          qd[e] = to_f32(qe[e]);
        }
      }
    }
  }
  for (int base = threadIdx.x; base < n * R; base += 4 * blockDim.x) {
    float vv[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int idx = base + u * blockDim.x;
      const int row = rb * R + idx % R;
      vv[u] = (idx < n * R && row < p.dv)
                  ? to_f32(v[(static_cast<size_t>(off + idx / R) * p.Hv + h) * p.dv + row])
                  : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; u++)
      if (base + u * blockDim.x < n * R) vb[base + u * blockDim.x] = vv[u];
  }
  for (int idx = threadIdx.x; idx < n; idx += blockDim.x) {
    const size_t ah = static_cast<size_t>(off + idx) * p.Hv + h;
    const float a = p.alpha[ah], b = p.beta[ah];
    sch[idx] = mv.sched[off + idx];
    nc[idx] = make_float4(a, b, 0.f, 0.f);
  }
}

template <typename T, int LPR>
__global__ void __launch_bounds__(kGdnThreads) gdn_verify_kernel(const GdnVerifyParams p) {
  using Sh = GdnShape<LPR>;
  constexpr int DK = Sh::DK, NG = Sh::NG, R = Sh::R;
  const int s = blockIdx.y;
  const int rb_per_head = (p.dv + R - 1) / R;
  const int h = blockIdx.x / rb_per_head;
  const int rb = blockIdx.x % rb_per_head;
  if (status_bad(p.status)) return;
  MetaView mv = meta_view(const_cast<void*>(p.meta), p.n_total);
  const SeqInfo info = mv.seq[s];
  const int n = info.n, off = info.off;
  if (n <= 0 || n > p.n_max) return;
  if (info.max_slot > p.n_slots) {
    if (threadIdx.x == 0) set_status(p.status, TV_ERR_TREE);
    return;
  }
  const int g = h / (p.Hv / p.Hk);

  extern __shared__ float4 smem4[];
  float* kb = reinterpret_cast<float*>(smem4);                     // [n_max][DK] keys, fp32
  float* qb = kb + p.n_max * DK;                                   // [n_max][DK] queries
  float4* nc = reinterpret_cast<float4*>(qb + p.n_max * DK);       // [n_max] (alpha, beta, k.q, -)
  float* vb = reinterpret_cast<float*>(nc + p.n_max);              // [n_max][R] v at this CTA's rows
  float* slots = vb + p.n_max * R;                                 // [n_slots][R][DK]
  int* sch = reinterpret_cast<int*>(slots + p.n_slots * R * DK);   // [n_max] traversal

  // this group's two state rows first, so their loads overlap the staging
  const int gi = threadIdx.x / LPR, j = threadIdx.x % LPR;
  const int r0 = gi, r1 = gi + NG;
  const int row0 = rb * R + r0, row1 = rb * R + r1;
  const bool valid0 = row0 < p.dv, valid1 = row1 < p.dv;
  f2_t s0[8], s1[8];
  if (valid0) {
    load_row8<LPR>(s0, p.S[s] + (static_cast<size_t>(h) * p.dv + row0) * DK, j);
  } else {
#pragma unroll
    for (int e = 0; e < 8; e++) s0[e] = 0ull;
  }
  if (valid1) {
    load_row8<LPR>(s1, p.S[s] + (static_cast<size_t>(h) * p.dv + row1) * DK, j);
  } else {
#pragma unroll
    for (int e = 0; e < 8; e++) s1[e] = 0ull;
  }
  stage_node_inputs<T, DK, R>(p, mv, n, off, g, h, rb, kb, qb, nc, vb, sch);
  __syncthreads();
  // k . q of every node, one lane group per node.  Every group runs every
  // round (the lane reduction needs all lanes of the warp); a group past the
  // last node reduces zeros and writes nothing.
  for (int base = 0; base < n; base += NG) {
    const int node = base + gi;
    const bool act = node < n;
    f2_t k[8], q[8];
    if (act) {
      load_row8<LPR>(k, kb + node * DK, j);
      load_row8<LPR>(q, qb + node * DK, j);
    } else {
#pragma unroll
      for (int e = 0; e < 8; e++) k[e] = q[e] = 0ull;
    }
    const float kq = kq_group<LPR>(k, q);
    if (act && j == 0) nc[node].z = kq;
  }
  __syncthreads();

  T* out = static_cast<T*>(p.out);
  for (int step = 0; step < n; step++) {
    const int e = sch[step];
    const int node = e & 0xFF, src = (e >> 8) & 0xFF, save = (e >> 16) & 0xFF;
    const bool has_children = (e >> 24) & 1;
    if (src) {
      load_row8<LPR>(s0, slots + ((src - 1) * R + r0) * DK, j);
      load_row8<LPR>(s1, slots + ((src - 1) * R + r1) * DK, j);
    }
    f2_t k[8], q[8];
    load_row8<LPR>(k, kb + node * DK, j);
    load_row8<LPR>(q, qb + node * DK, j);
    const float4 c4 = nc[node];
    const float o0 =
        gdn_row_step<LPR, true>(s0, k, q, c4.z, vb[node * R + r0], c4.x, c4.y, p.scale, has_children);
    const float o1 =
        gdn_row_step<LPR, true>(s1, k, q, c4.z, vb[node * R + r1], c4.x, c4.y, p.scale, has_children);
    if (save) {
      store_row8<LPR>(slots + ((save - 1) * R + r0) * DK, s0, j);
      store_row8<LPR>(slots + ((save - 1) * R + r1) * DK, s1, j);
    }
    if (j == 0) {
      T* orow = out + (static_cast<size_t>(off + node) * p.Hv + h) * p.dv;
      if (valid0) orow[row0] = from_f32<T>(o0);
      if (valid1) orow[row1] = from_f32<T>(o1);
    }
  }
}

struct GdnDecodeParams {
  float* S[TV_MAX_SEQ];
  const void* q;
  const void* k;
  const void* v;
  const float* alpha;
  const float* beta;
  void* out;
  int32_t* status;
  int Hk, Hv, dv;
  float scale;
};

template <typename T, int LPR>
__global__ void __launch_bounds__(128) gdn_decode_kernel(const GdnDecodeParams p) {
  constexpr int DK = 16 * LPR;
  constexpr int R = 128 / LPR;
  const int s = blockIdx.y;
  const int rb_per_head = (p.dv + R - 1) / R;
  const int h = blockIdx.x / rb_per_head;
  const int rb = blockIdx.x % rb_per_head;
  if (status_bad(p.status)) return;
  const int g = h / (p.Hv / p.Hk);
  __shared__ __align__(16) float kb[DK];
  __shared__ __align__(16) float qb[DK];
  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  for (int e = threadIdx.x; e < DK; e += blockDim.x) {
    const size_t src = (static_cast<size_t>(s) * p.Hk + g) * DK + e;
    kb[e] = to_f32(k[src]);
    qb[e] = to_f32(q[src]);
  }
  __syncthreads();
  const int r = threadIdx.x / LPR, j = threadIdx.x % LPR;
  const int row = rb * R + r;
  const bool valid = row < p.dv;
  float* Srow = p.S[s] + (static_cast<size_t>(h) * p.dv + (valid ? row : 0)) * DK;
  f2_t st[8];
  if (valid) {
    load_row8<LPR>(st, Srow, j);
  } else {
#pragma unroll
    for (int e = 0; e < 8; e++) st[e] = 0ull;
  }
  f2_t kk[8], qq[8];
  load_row8<LPR>(kk, kb, j);
  load_row8<LPR>(qq, qb, j);
  const float kq = kq_group<LPR>(kk, qq);
  const size_t hi = static_cast<size_t>(s) * p.Hv + h;
  const float vv = valid ? to_f32(static_cast<const T*>(p.v)[hi * p.dv + row]) : 0.f;
  const float o = gdn_row_step<LPR, true>(st, kk, qq, kq, vv, p.alpha[hi], p.beta[hi], p.scale, true);
  if (valid) {
    store_row8<LPR>(Srow, st, j);
    if (j == 0) static_cast<T*>(p.out)[hi * p.dv + row] = from_f32<T>(o);
  }
}

static bool gdn_shape_ok(const tv_gdn_layer* l) {
  return l && (l->dtype == TV_F32 || l->dtype == TV_BF16) && l->Hk >= 1 && l->Hv >= l->Hk && l->Hv % l->Hk == 0 &&
         (l->dk == 64 || l->dk == 128) && l->dv >= 1 && l->dv <= 256 && l->S;
}

template <typename T, int LPR>
static void launch_verify(const GdnVerifyParams& p, int n_seq, cudaStream_t st) {
  constexpr int R = GdnShape<LPR>::R;
  static bool attrs = false;  // one-time, sized for the largest tree
  if (!attrs) {
    const int smem_max = static_cast<int>(gdn_verify_smem<LPR>(TV_MAX_NODES, slots_for(TV_MAX_NODES)));
    cudaFuncSetAttribute(gdn_verify_kernel<T, LPR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    attrs = true;
  }
  const dim3 grid(p.Hv * ((p.dv + R - 1) / R), n_seq);
  gdn_verify_kernel<T, LPR><<<grid, kGdnThreads, gdn_verify_smem<LPR>(p.n_max, p.n_slots), st>>>(p);
}

template <typename T, int LPR>
static void launch_decode(const GdnDecodeParams& p, int n_seq, cudaStream_t st) {
  constexpr int R = 128 / LPR;
  const dim3 grid(p.Hv * ((p.dv + R - 1) / R), n_seq);
  gdn_decode_kernel<T, LPR><<<grid, 128, 0, st>>>(p);
}

tv_status gdn_decode_launch(const tv_gdn_layer* l, int32_t n_seq, const void* q, const void* k, const void* v,
                            const float* alpha, const float* beta, void* out, float scale, int32_t* status,
                            cudaStream_t st) {
  if (!gdn_shape_ok(l) || n_seq < 1 || n_seq > TV_MAX_SEQ || !q || !k || !v || !alpha || !beta || !out || !status)
    return TV_ERR_ARG;
  GdnDecodeParams p{};
  for (int s = 0; s < n_seq; s++) {
    if (!l->S[s]) return TV_ERR_ARG;
    if (!aligned16(l->S[s])) return TV_ERR_ALIGN;
    p.S[s] = l->S[s];
  }
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(alpha) || !aligned16(beta))
    return TV_ERR_ALIGN;
  p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta; p.out = out; p.status = status;
  p.Hk = l->Hk; p.Hv = l->Hv; p.dv = l->dv; p.scale = scale;
  const bool bf = l->dtype == TV_BF16;
  if (l->dk == 128) {
    if (bf) launch_decode<__nv_bfloat16, 8>(p, n_seq, st); else launch_decode<float, 8>(p, n_seq, st);
  } else {
    if (bf) launch_decode<__nv_bfloat16, 4>(p, n_seq, st); else launch_decode<float, 4>(p, n_seq, st);
  }
  return launch_status();
}

}  // namespace tv

using namespace tv;

extern "C" tv_status tv_gdn_tree_verify(const tv_gdn_layer* l, const tv_tree* t, const void* q, const void* k,
                                        const void* v, const float* alpha, const float* beta, void* out,
                                        float scale, tv_stream stream) {
  if (!tree_ok(t)) return TV_ERR_ARG;
  if (!l || !l->S) return TV_ERR_ARG;
  if (l->dtype != TV_F32 && l->dtype != TV_BF16) return TV_ERR_DTYPE;
  if (!gdn_shape_ok(l)) return TV_ERR_SHAPE;
  if (!q || !k || !v || !alpha || !beta || !out) return TV_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(alpha) || !aligned16(beta))
    return TV_ERR_ALIGN;
  GdnVerifyParams p{};
  for (int s = 0; s < t->n_seq; s++) {
    if (!l->S[s]) return TV_ERR_ARG;
    if (!aligned16(l->S[s])) return TV_ERR_ALIGN;
    p.S[s] = l->S[s];
  }
  p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta; p.out = out;
  p.meta = t->meta; p.status = t->status;
  p.n_total = t->n_total; p.n_max = t->n_max; p.n_slots = slots_for(t->n_max);
  p.Hk = l->Hk; p.Hv = l->Hv; p.dv = l->dv; p.scale = scale;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool bf = l->dtype == TV_BF16;
  if (l->dk == 128) {
    if (bf) launch_verify<__nv_bfloat16, 8>(p, t->n_seq, st); else launch_verify<float, 8>(p, t->n_seq, st);
  } else {
    if (bf) launch_verify<__nv_bfloat16, 4>(p, t->n_seq, st); else launch_verify<float, 4>(p, t->n_seq, st);
  }
  return launch_status();
}
