// Gated DeltaNet tree verify and single-token decode.
//
// Tree verify ("Adding a model", Gated DeltaNet layers; the gated delta rule
// applied along every node's root path): one CTA owns a block of state rows of
// one value head of one sequence and walks the tree in the order prepared by
// tv_tree_prepare, keeping the current node's state rows in registers and
// the few states that must outlive a subtree in register slots.  No per-node
// state is ever written to memory; the kernel reads the committed state once
// and writes one output value per (node, row).
//
// Work per (node, row): two dot products of length dk (s.k, s.q) and, for
// nodes with children, one rank-1 update of the row; the kernel is bound by
// CUDA-core arithmetic, not by the 4 * Hv * dv * dk bytes of state it reads.
#include "common.cuh"
#include "gdn_step.cuh"
#include "host.hpp"
#include "launchers.hpp"

namespace tv {

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
  int n_total, n_max, Hk, Hv, dv;
  float scale;
};

__device__ __forceinline__ void copy16(float (&d)[16], const float (&s)[16]) {
#pragma unroll
  for (int e = 0; e < 16; e++) d[e] = s[e];
}

// Saved states live in registers: every access below uses a constant slot index.
__device__ __forceinline__ void slot_save(float (&sl)[kMaxSlots][16], const float (&st)[16], int k) {
  switch (k) {
    case 0: copy16(sl[0], st); break;
    case 1: copy16(sl[1], st); break;
    case 2: copy16(sl[2], st); break;
    case 3: copy16(sl[3], st); break;
    default: copy16(sl[4], st); break;
  }
}
__device__ __forceinline__ void slot_load(float (&st)[16], const float (&sl)[kMaxSlots][16], int k) {
  switch (k) {
    case 0: copy16(st, sl[0]); break;
    case 1: copy16(st, sl[1]); break;
    case 2: copy16(st, sl[2]); break;
    case 3: copy16(st, sl[3]); break;
    default: copy16(st, sl[4]); break;
  }
}

template <typename T, int LPR>
__global__ void __launch_bounds__(128) gdn_verify_kernel(const GdnVerifyParams p) {
  constexpr int DK = 16 * LPR;
  constexpr int R = 128 / LPR;  // state rows per CTA
  const int s = blockIdx.y;
  const int rb_per_head = (p.dv + R - 1) / R;
  const int h = blockIdx.x / rb_per_head;
  const int rb = blockIdx.x % rb_per_head;
  if (status_bad(p.status)) return;
  MetaView mv = meta_view(const_cast<void*>(p.meta), p.n_total);
  const SeqInfo info = mv.seq[s];
  const int n = info.n, off = info.off;
  if (n <= 0 || n > p.n_max) return;
  const int g = h / (p.Hv / p.Hk);

  extern __shared__ float4 smem4[];
  float* kb = reinterpret_cast<float*>(smem4);  // [n_max][DK] keys, fp32
  float* qb = kb + p.n_max * DK;                // [n_max][DK] queries
  float* vb = qb + p.n_max * DK;                // [n_max][R]  v at this CTA's rows
  float* ab = vb + p.n_max * R;                 // [n_max]
  float* bb = ab + p.n_max;                     // [n_max]
  float* kqb = bb + p.n_max;                    // [n_max]
  int* sch = reinterpret_cast<int*>(kqb + p.n_max);

  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  const T* v = static_cast<const T*>(p.v);
  for (int idx = threadIdx.x; idx < n * DK; idx += blockDim.x) {
    const int node = idx / DK, e = idx % DK;
    const size_t src = (static_cast<size_t>(off + node) * p.Hk + g) * DK + e;
    kb[idx] = to_f32(k[src]);
    qb[idx] = to_f32(q[src]);
  }
  for (int idx = threadIdx.x; idx < n * R; idx += blockDim.x) {
    const int node = idx / R, r = idx % R, row = rb * R + r;
    vb[idx] = row < p.dv ? to_f32(v[(static_cast<size_t>(off + node) * p.Hv + h) * p.dv + row]) : 0.f;
  }
  for (int idx = threadIdx.x; idx < n; idx += blockDim.x) {
    ab[idx] = p.alpha[static_cast<size_t>(off + idx) * p.Hv + h];
    bb[idx] = p.beta[static_cast<size_t>(off + idx) * p.Hv + h];
    sch[idx] = mv.sched[off + idx];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < n; idx += blockDim.x) kqb[idx] = dot_seq(kb + idx * DK, qb + idx * DK, DK);
  __syncthreads();

  const int r = threadIdx.x / LPR, j = threadIdx.x % LPR;
  const int row = rb * R + r;
  const bool valid = row < p.dv;
  float st[16];
  if (valid) {
    load_row16<LPR>(st, p.S[s] + (static_cast<size_t>(h) * p.dv + row) * DK, j);
  } else {
#pragma unroll
    for (int e = 0; e < 16; e++) st[e] = 0.f;
  }
  float sl[kMaxSlots][16];
  T* out = static_cast<T*>(p.out);
  for (int step = 0; step < n; step++) {
    const int e = sch[step];
    const int node = e & 0xFF, src = (e >> 8) & 0xFF, save = (e >> 16) & 0xFF;
    const bool has_children = (e >> 24) & 1;
    if (src) slot_load(st, sl, src - 1);
    const float o = gdn_row_step<LPR, true>(st, kb + node * DK, qb + node * DK, j, kqb[node], vb[node * R + r],
                                            ab[node], bb[node], p.scale, has_children);
    if (save) slot_save(sl, st, save - 1);
    if (valid && j == 0) out[(static_cast<size_t>(off + node) * p.Hv + h) * p.dv + row] = from_f32<T>(o);
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
  __shared__ float kq;
  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  for (int e = threadIdx.x; e < DK; e += blockDim.x) {
    const size_t src = (static_cast<size_t>(s) * p.Hk + g) * DK + e;
    kb[e] = to_f32(k[src]);
    qb[e] = to_f32(q[src]);
  }
  __syncthreads();
  if (threadIdx.x == 0) kq = dot_seq(kb, qb, DK);
  __syncthreads();
  const int r = threadIdx.x / LPR, j = threadIdx.x % LPR;
  const int row = rb * R + r;
  const bool valid = row < p.dv;
  float* Srow = p.S[s] + (static_cast<size_t>(h) * p.dv + (valid ? row : 0)) * DK;
  float st[16];
  if (valid) {
    load_row16<LPR>(st, Srow, j);
  } else {
#pragma unroll
    for (int e = 0; e < 16; e++) st[e] = 0.f;
  }
  const size_t hi = static_cast<size_t>(s) * p.Hv + h;
  const float vv = valid ? to_f32(static_cast<const T*>(p.v)[hi * p.dv + row]) : 0.f;
  const float o = gdn_row_step<LPR, true>(st, kb, qb, j, kq, vv, p.alpha[hi], p.beta[hi], p.scale, true);
  if (valid) {
    store_row16<LPR>(Srow, st, j);
    if (j == 0) static_cast<T*>(p.out)[hi * p.dv + row] = from_f32<T>(o);
  }
}

static bool gdn_shape_ok(const tv_gdn_layer* l) {
  return l && (l->dtype == TV_F32 || l->dtype == TV_BF16) && l->Hk >= 1 && l->Hv >= l->Hk && l->Hv % l->Hk == 0 &&
         (l->dk == 64 || l->dk == 128) && l->dv >= 1 && l->dv <= 256 && l->S;
}

template <typename T, int LPR>
static void launch_verify(const GdnVerifyParams& p, int n_seq, cudaStream_t st) {
  constexpr int DK = 16 * LPR, R = 128 / LPR;
  const size_t smem = (2 * static_cast<size_t>(p.n_max) * DK + static_cast<size_t>(p.n_max) * R + 4 * p.n_max) * 4;
  static bool attrs = false;  // one-time, sized for the largest tree
  if (!attrs) {
    const int smem_max = (2 * TV_MAX_NODES * DK + TV_MAX_NODES * R + 4 * TV_MAX_NODES) * 4;
    cudaFuncSetAttribute(gdn_verify_kernel<T, LPR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    attrs = true;
  }
  const dim3 grid(p.Hv * ((p.dv + R - 1) / R), n_seq);
  gdn_verify_kernel<T, LPR><<<grid, 128, smem, st>>>(p);
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
  p.n_total = t->n_total; p.n_max = t->n_max; p.Hk = l->Hk; p.Hv = l->Hv; p.dv = l->dv; p.scale = scale;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool bf = l->dtype == TV_BF16;
  if (l->dk == 128) {
    if (bf) launch_verify<__nv_bfloat16, 8>(p, t->n_seq, st); else launch_verify<float, 8>(p, t->n_seq, st);
  } else {
    if (bf) launch_verify<__nv_bfloat16, 4>(p, t->n_seq, st); else launch_verify<float, 4>(p, t->n_seq, st);
  }
  return launch_status();
}
