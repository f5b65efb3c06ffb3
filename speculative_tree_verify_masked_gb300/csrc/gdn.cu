// Gated DeltaNet tree verify and single-token decode.
//
// Tree verify ("Adding a model", Gated DeltaNet layers; the gated delta rule
// applied along every node's root path): a CTA of four warps owns
// 4 * 4 * 32/LPR state rows of one value head of one sequence (the warps share
// one staged copy of the tree's keys, queries and gates) and each warp walks
// the tree in the order prepared by tv_tree_prepare.  A lane group of LPR lanes holds four
// state rows, so each node's key and query, read once from shared memory (as
// bf16), serve four rows, and the eight dot products of a step (s.k and s.q
// of each row) are reduced together by one reduce-scatter.  The few states
// that must outlive a subtree sit in shared-memory slots.  No per-node state
// is written to memory: the kernel reads the committed state once and writes
// one output value per (node, row).
//
// Work per (node, row): two dot products of length dk and, for nodes with
// children, one rank-1 update of the row, in packed fp32x2 arithmetic.  The
// kernel is bound by the dependent chain of steps along the tree, not by the
// 4 * Hv * dv * dk bytes of state it reads.
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
  static constexpr int DK = 16 * LPR;  // key dim
  static constexpr int NG = 32 / LPR;  // lane groups per warp
  static constexpr int RPG = 4;        // state rows per lane group
  static constexpr int W = 4;          // warps per CTA (one per SM sub-partition)
  static constexpr int NGC = NG * W;   // lane groups per CTA
  static constexpr int R = NGC * RPG;  // state rows per CTA
  static constexpr int NV = 2 * RPG;   // dot products per step and group (s.k, s.q per row)
};

// Shared memory: slots [n_slots][R][DK] f32 | keys, queries [n_max][DK] T |
// (alpha, beta, k.q, -) [n_max] | v [n_max][R] f32 | schedule [n_max].
template <typename T, int LPR>
inline size_t gdn_verify_smem(int n_max, int n_slots) {
  using Sh = GdnShape<LPR>;
  const size_t n = static_cast<size_t>(n_max);
  size_t b = static_cast<size_t>(n_slots) * Sh::R * Sh::DK * 4;
  b += 2 * ((n * Sh::DK * sizeof(T) + 15) / 16 * 16);
  b += n * 16 + n * Sh::R * 4 + n * 4;
  return b;
}

__device__ __forceinline__ void cp_async16_g(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))), "l"(src) : "memory");
}

template <typename T, int LPR>
__global__ void __launch_bounds__(32 * GdnShape<LPR>::W) gdn_verify_kernel(const GdnVerifyParams p) {
  using Sh = GdnShape<LPR>;
  constexpr int DK = Sh::DK, R = Sh::R, RPG = Sh::RPG, NV = Sh::NV;
  const int s = blockIdx.y;
  const int rb_per_head = (p.dv + R - 1) / R;
  const int h = blockIdx.x / rb_per_head;
  const int rb = blockIdx.x % rb_per_head;
  const int tid = threadIdx.x, lane = tid & 31, j = lane % LPR;
  const int gi = (tid >> 5) * Sh::NG + lane / LPR;  // lane group within the CTA

  // this group's four state rows first (they do not depend on the tree, and
  // no kernel of the round before commit writes them), so their loads overlap
  // the previous kernel's end and everything up to the first step
  f2_t st[RPG][8];
  bool valid[RPG];
#pragma unroll
  for (int r = 0; r < RPG; r++) {
    const int row = rb * R + gi * RPG + r;
    valid[r] = row < p.dv;
    if (valid[r]) {
      load_row8<LPR>(st[r], p.S[s] + (static_cast<size_t>(h) * p.dv + row) * DK, j);
    } else {
#pragma unroll
      for (int e = 0; e < 8; e++) st[r][e] = 0ull;
    }
  }
  pdl_wait();  // tree tables, status and node inputs come from earlier kernels
  pdl_trigger();
  MetaView mv = meta_view(const_cast<void*>(p.meta), p.n_total);
  const SeqInfo info = mv.seq[s];
  if (status_bad(p.status)) return;
  const int n = info.n, off = info.off;
  if (n <= 0 || n > p.n_max) return;
  if (info.max_slot > p.n_slots) {
    if (tid == 0) set_status(p.status, TV_ERR_TREE);
    return;
  }
  const int g = h / (p.Hv / p.Hk);

  extern __shared__ float4 smem4[];
  float* slots = reinterpret_cast<float*>(smem4);  // [n_slots][R][DK]
  T* kb = reinterpret_cast<T*>(slots + static_cast<size_t>(p.n_slots) * R * DK);
  const size_t kq_bytes = (static_cast<size_t>(p.n_max) * DK * sizeof(T) + 15) / 16 * 16;
  T* qb = reinterpret_cast<T*>(reinterpret_cast<uint8_t*>(kb) + kq_bytes);
  float4* nc = reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(qb) + kq_bytes);  // [n_max]
  float* vb = reinterpret_cast<float*>(nc + p.n_max);                                // [n_max][R]
  int* sch = reinterpret_cast<int*>(vb + static_cast<size_t>(p.n_max) * R);          // [n_max]

  // stage the tree's keys and queries of this key head (raw, asynchronously),
  // then the values of this CTA's rows, alpha, beta and the traversal, with
  // every load issued before any is used
  {
    constexpr int CPR = DK * static_cast<int>(sizeof(T)) / 16;  // 16-byte chunks per key row
    const T* qg = static_cast<const T*>(p.q);
    const T* kg = static_cast<const T*>(p.k);
    for (int idx = tid; idx < n * CPR; idx += blockDim.x) {
      const size_t src = (static_cast<size_t>(off + idx / CPR) * p.Hk + g) * DK + (idx % CPR) * (16 / sizeof(T));
      cp_async16_g(kb + static_cast<size_t>(idx / CPR) * DK + (idx % CPR) * (16 / sizeof(T)), kg + src);
      cp_async16_g(qb + static_cast<size_t>(idx / CPR) * DK + (idx % CPR) * (16 / sizeof(T)), qg + src);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    const T* vg = static_cast<const T*>(p.v);
    for (int base = tid; base < n * R; base += 16 * blockDim.x) {
      float vv[16];
#pragma unroll
      for (int u = 0; u < 16; u++) {
        const int idx = base + u * blockDim.x;
        const int row = rb * R + idx % R;
        vv[u] = (idx < n * R && row < p.dv)
                    ? to_f32(vg[(static_cast<size_t>(off + idx / R) * p.Hv + h) * p.dv + row])
                    : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 16; u++)
        if (base + u * blockDim.x < n * R) vb[base + u * blockDim.x] = vv[u];
    }
    for (int idx = tid; idx < n; idx += blockDim.x) {
      const size_t ah = static_cast<size_t>(off + idx) * p.Hv + h;
      const float a = p.alpha[ah], b = p.beta[ah];
      sch[idx] = mv.sched[off + idx];
      nc[idx] = make_float4(a, b, 0.f, 0.f);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
  }
  // k . q of every node: each group takes eight nodes at a time, and one
  // reduce-scatter finishes all of them
  for (int base = 0; base < n; base += 8 * Sh::NGC) {
    float part[8];
#pragma unroll
    for (int m = 0; m < 8; m++) {
      const int node = base + gi * 8 + m;
      part[m] = 0.f;
      if (node < n) {
        f2_t kk[8], qq[8];
        load_row8_any<LPR>(kk, kb + static_cast<size_t>(node) * DK, j);
        load_row8_any<LPR>(qq, qb + static_cast<size_t>(node) * DK, j);
        part[m] = row_partial(kk, qq);
      }
    }
    reduce_scatter<LPR, 8>(part, j);
#pragma unroll
    for (int i = 0; i < rs_count<LPR, 8>(); i++) {
      const int m = rs_value<LPR, 8>(j, i);
      const int node = base + gi * 8 + m;
      const bool writer = rs_first<LPR, 8>(j);
      if (writer && node < n) nc[node].z = part[i];
    }
  }
  __syncthreads();

  T* out = static_cast<T*>(p.out);
  // The next node's schedule entry, key, query, gates and values do not depend
  // on the state: each step loads them for the step after, so only the state
  // chain (dots, reduce-scatter, update) is on the critical path.
  int e_nx = sch[0];
  f2_t k_nx[8], q_nx[8];
  float4 c_nx;
  float v_nx[RPG];
  {
    const int node = e_nx & 0xFF;
    load_row8_any<LPR>(k_nx, kb + static_cast<size_t>(node) * DK, j);
    load_row8_any<LPR>(q_nx, qb + static_cast<size_t>(node) * DK, j);
    c_nx = nc[node];
#pragma unroll
    for (int r = 0; r < RPG; r++) v_nx[r] = vb[node * R + gi * RPG + r];
  }
  for (int step = 0; step < n; step++) {
    const int e = e_nx;
    const int node = e & 0xFF, src = (e >> 8) & 0xFF, save = (e >> 16) & 0xFF;
    const bool has_children = (e >> 24) & 1;
    f2_t k[8], q[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
      k[i] = k_nx[i];
      q[i] = q_nx[i];
    }
    const float4 c4 = c_nx;
    float v[RPG];
#pragma unroll
    for (int r = 0; r < RPG; r++) v[r] = v_nx[r];
    if (step + 1 < n) {
      e_nx = sch[step + 1];
      const int nn = e_nx & 0xFF;
      load_row8_any<LPR>(k_nx, kb + static_cast<size_t>(nn) * DK, j);
      load_row8_any<LPR>(q_nx, qb + static_cast<size_t>(nn) * DK, j);
      c_nx = nc[nn];
#pragma unroll
      for (int r = 0; r < RPG; r++) v_nx[r] = vb[nn * R + gi * RPG + r];
    }
    if (src) {
#pragma unroll
      for (int r = 0; r < RPG; r++) load_row8<LPR>(st[r], slots + ((src - 1) * R + gi * RPG + r) * DK, j);
    }
    float part[NV];
#pragma unroll
    for (int r = 0; r < RPG; r++) {
      part[2 * r] = row_partial(st[r], k);
      part[2 * r + 1] = row_partial(st[r], q);
    }
    reduce_scatter<LPR, NV>(part, j);
    float c[RPG];
#pragma unroll
    for (int r = 0; r < RPG; r++) {
      const float x = __shfl_sync(0xffffffffu, part[rs_index<LPR, NV>(2 * r)], rs_lane<LPR, NV>(2 * r), LPR);
      c[r] = gdn_c(x, v[r], c4.x, c4.y);
    }
    if (has_children) {
#pragma unroll
      for (int r = 0; r < RPG; r++) gdn_update(st[r], k, c4.x, c[r]);
    }
    if (save) {
#pragma unroll
      for (int r = 0; r < RPG; r++) store_row8<LPR>(slots + ((save - 1) * R + gi * RPG + r) * DK, st[r], j);
    }
    // one lane holding y of a row writes that row's output
#pragma unroll
    for (int i = 0; i < rs_count<LPR, NV>(); i++) {
      const int m = rs_value<LPR, NV>(j, i);
      const bool writer = rs_first<LPR, NV>(j);
      if (writer && (m & 1)) {
        const int r = m >> 1;
        float cr = c[0];
#pragma unroll
        for (int rr = 1; rr < RPG; rr++)
          if (rr == r) cr = c[rr];
        bool vr = valid[0];
#pragma unroll
        for (int rr = 1; rr < RPG; rr++)
          if (rr == r) vr = valid[rr];
        if (vr)
          out[(static_cast<size_t>(off + node) * p.Hv + h) * p.dv + rb * R + gi * RPG + r] =
              from_f32<T>(gdn_o(cr, c4.z, c4.x, part[i], p.scale));
      }
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
static void launch_verify(const GdnVerifyParams& p, int n_seq, cudaStream_t st, bool ov) {
  constexpr int R = GdnShape<LPR>::R;
  static bool attrs = false;  // one-time, sized for the largest tree
  if (!attrs) {
    const int smem_max = static_cast<int>(gdn_verify_smem<T, LPR>(TV_MAX_NODES, slots_for(TV_MAX_NODES)));
    cudaFuncSetAttribute(gdn_verify_kernel<T, LPR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    attrs = true;
  }
  const dim3 grid(p.Hv * ((p.dv + R - 1) / R), n_seq);
  launch_k(ov, gdn_verify_kernel<T, LPR>, grid, dim3(32 * GdnShape<LPR>::W), gdn_verify_smem<T, LPR>(p.n_max, p.n_slots),
           st, p);
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
  const bool ov = tree_overlap(t);
  if (l->dk == 128) {
    if (bf) launch_verify<__nv_bfloat16, 8>(p, t->n_seq, st, ov); else launch_verify<float, 8>(p, t->n_seq, st, ov);
  } else {
    if (bf) launch_verify<__nv_bfloat16, 4>(p, t->n_seq, st, ov); else launch_verify<float, 4>(p, t->n_seq, st, ov);
  }
  return launch_status();
}
