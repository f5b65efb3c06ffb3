// Gated DeltaNet tree verify and single-token decode.
//
// Tree verify ("Adding a model", Gated DeltaNet layers; the gated delta rule
// applied along every node's root path).  A lane group of LPR lanes owns two
// state rows of one value head of one sequence, each with the lane layout
// and the step arithmetic of decode and commit (gdn_step.cuh), so a verified
// row is the decoded row bit for bit by construction.  A CTA of W warps
// owns W * 2 * 32/LPR consecutive rows of one value head and stages the
// tree's keys and queries (by cp.async), gates and values once.  The
// lane groups walk the tree in the order prepared by tv_tree_prepare, cut
// into segments that restore a saved state only at their start and save one
// only at their end.  Every lane group of a CTA visits the same node at the
// same time, so the one branch inside a segment, a leaf skipping its update,
// is uniform; a leaf leaves the state as it is, so its siblings still find
// their parent's state in registers.  The few states that must outlive a subtree
// sit in shared-memory slots.  No per-node state is written to memory: the
// kernel reads the committed state once and writes one output value per
// (node, row).
//
// Bound.  The chain of dependent steps along the tree, not the
// 4 * Hv * dv * dk bytes of state, sets the layer's time: every visit is a
// chain of dependent pieces (shared-memory loads, packed fp32 FMAs, the
// butterfly over the group, the update) that a warp issues in order, and
// the tree's visits run one after another.  Two rows per lane group (16
// columns per lane, one 16-byte bf16 load per chunk of the node's key or
// query serving both rows) and CTAs of four or eight warps that share one
// staged copy of the tree's inputs; leaves skip the update (nothing reads
// their state).
#include "common.cuh"
#include "front_gdn.cuh"
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
  // front end of the fused verify: raw projections [n_total][C], raw gates
  // [n_total][Hv], convolution weights [C][W] and each sequence's tail [W-1][C]
  const void* x;
  const float* a_raw;
  const float* b_raw;
  const float* wconv;
  const void* tail[TV_MAX_SEQ];
  int C, W;
};

// Slots for states that must outlive a subtree: at most floor(log2(n / 5)) + 1
// for a tree of n nodes (see tree.cu).
inline int slots_for(int n_max) {
  int k = 1;
  while ((5 << k) <= n_max) k++;
  return k;
}

// Layout of a verify CTA: WARPS warps, lane groups of LPR lanes, RPG state
// rows per lane group (each row with the lane layout of gdn_step.cuh).
template <int LPR, int RPG, int WARPS>
struct GdnShape {
  static constexpr int DK = 2 * kPairs * LPR;  // key dim
  static constexpr int W = WARPS;              // warps per CTA
  static constexpr int NG = W * 32 / LPR;      // lane groups per CTA
  static constexpr int R = NG * RPG;           // state rows per CTA
};
// The verify kernel runs two rows per lane group with CTAs of 4 or 8 warps:
// 8 when CTAs of 4 warps would number at most two per SM (then one CTA of 8
// warps per SM stages the tree once for twice the rows and keeps two warps
// per scheduler; measured on one GDN layer of the 64-layer workload, 15.2
// against 17.7 us), 4 otherwise (more sequences: 18.5 against 18.9 us on the
// four-sequence workload).
constexpr int kGdnRpg = 2;

// Shared memory: slots [n_slots][R][DK] f32 | keys, queries [n_max][DK] KQ |
// (alpha, beta, k.q, -) [n_max] | v [n_max][R] f32 | visits [n_max] | segments [n_max].
// KQ is the input type: staging keys and queries widened to fp32 measured
// no faster per visit and takes twice the shared memory.
template <typename KQ, typename Sh>
inline size_t gdn_verify_smem(int n_max, int n_slots) {
  const size_t n = static_cast<size_t>(n_max);
  size_t b = static_cast<size_t>(n_slots) * Sh::R * Sh::DK * 4;
  b += 2 * ((n * Sh::DK * sizeof(KQ) + 15) / 16 * 16);
  b += n * 16 + n * Sh::R * 4 + 2 * n * 4;
  return b;
}

__device__ __forceinline__ void cp_async16_g(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))), "l"(src) : "memory");
}

// Values of a lane group's RPG rows (consecutive fp32 in shared memory).
template <int N>
__device__ __forceinline__ void load_vals(float (&v)[N], const float* src) {
  if constexpr (N == 4) {
    const float4 t = *reinterpret_cast<const float4*>(src);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else if constexpr (N == 2) {
    const float2 t = *reinterpret_cast<const float2*>(src);
    v[0] = t.x; v[1] = t.y;
  } else {
#pragma unroll
    for (int i = 0; i < N; i++) v[i] = src[i];
  }
}

template <typename T, int LPR, int RPG, int WARPS, bool FRONT>
__global__ void __launch_bounds__(32 * WARPS) gdn_verify_kernel(const GdnVerifyParams p) {
  using KQ = T;
  using Sh = GdnShape<LPR, RPG, WARPS>;
  constexpr int DK = Sh::DK, R = Sh::R, NG = Sh::NG, NT = 32 * WARPS;
  const int s = blockIdx.y;
  const int rb_per_head = (p.dv + R - 1) / R;
  const int h = blockIdx.x / rb_per_head;
  const int rb = blockIdx.x % rb_per_head;
  const int tid = threadIdx.x, j = tid % LPR;
  const int gi = tid / LPR;                 // lane group within the CTA
  const int row0 = rb * R + RPG * gi;       // the group's rows: row0 .. row0 + RPG - 1

  // this group's state rows first (they do not depend on the tree, and no
  // kernel of the round before commit writes them), so their loads overlap
  // the previous kernel's end and everything up to the first step
  f2_t st[RPG][kPairs];
  {
    const float* S = p.S[s] + static_cast<size_t>(h) * p.dv * DK;
#pragma unroll
    for (int i = 0; i < RPG; i++) {
      if (row0 + i < p.dv) {
        load_row<LPR>(st[i], S + static_cast<size_t>(row0 + i) * DK, j);
      } else {
#pragma unroll
        for (int e = 0; e < kPairs; e++) st[i][e] = 0ull;
      }
    }
  }
  pdl_wait();  // tree tables, status and node inputs come from earlier kernels
  pdl_trigger();
  MetaView mv = meta_view(const_cast<void*>(p.meta), p.n_total);
  const SeqInfo info = mv.seq[s];
  if (status_bad(p.status)) return;
  const int n = info.n, off = info.off, n_seg = info.n_seg;
  if (n <= 0 || n > p.n_max || n_seg < 1 || n_seg > n) return;
  if (info.max_slot > p.n_slots) {
    if (tid == 0) set_status(p.status, TV_ERR_TREE);
    return;
  }
  const int g = h / (p.Hv / p.Hk);

  extern __shared__ float4 smem4[];
  float* slots = reinterpret_cast<float*>(smem4);  // [n_slots][R][DK]
  KQ* kb = reinterpret_cast<KQ*>(slots + static_cast<size_t>(p.n_slots) * R * DK);
  const size_t kq_bytes = (static_cast<size_t>(p.n_max) * DK * sizeof(KQ) + 15) / 16 * 16;
  KQ* qb = reinterpret_cast<KQ*>(reinterpret_cast<uint8_t*>(kb) + kq_bytes);
  float4* nc = reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(qb) + kq_bytes);  // [n_max]
  float* vb = reinterpret_cast<float*>(nc + p.n_max);                                // [n_max][R]
  int* sch = reinterpret_cast<int*>(vb + static_cast<size_t>(p.n_max) * R);          // [n_max] visits
  int* sgt = sch + p.n_max;                                                           // [n_max] segments

  if constexpr (FRONT) {
    // The front end, as tv_gdn_front forms it (front_gdn.cuh): this key
    // head's query and key of every node (one warp per node and vector:
    // convolution along the node's ancestor path into the committed tail,
    // SiLU, division by the head's L2 norm, rounding to the layer type), the
    // values of this CTA's rows (convolution, SiLU, rounding) and the gates.
    const T* x = static_cast<const T*>(p.x);
    const T* tail = static_cast<const T*>(p.tail[s]);
    const int warp = tid >> 5, lane = tid & 31;
    constexpr int CPL = DK / 32;
    auto window = [&](int node, int (&src)[kMaxConvWidth]) {
      const int row = off + node;
      conv_window(src, p.W, mv.depth[row], off, mv.anc_at + static_cast<size_t>(row) * TV_MAX_PATH, row);
    };
    for (int w = warp; w < 2 * n; w += WARPS) {
      const int node = w >> 1, is_k = w & 1;
      int src[kMaxConvWidth];
      window(node, src);
      const int c0 = (is_k ? p.Hk + g : g) * DK;
      float val[CPL];
#pragma unroll
      for (int e = 0; e < CPL; e++) val[e] = conv_silu(x, tail, p.wconv, p.C, p.W, src, c0 + lane + 32 * e);
      const float sc = warp_l2_scale<CPL>(val);
      KQ* dst = (is_k ? kb : qb) + static_cast<size_t>(node) * DK;
#pragma unroll
      for (int e = 0; e < CPL; e++) dst[lane + 32 * e] = from_f32<KQ>(__fmul_rn(val[e], sc));
    }
    for (int idx = tid; idx < n * R; idx += NT) {
      const int node = idx / R, rr = rb * R + idx % R;
      float vv = 0.f;
      if (rr < p.dv) {
        int src[kMaxConvWidth];
        window(node, src);
        vv = to_f32(from_f32<T>(conv_silu(x, tail, p.wconv, p.C, p.W, src, 2 * p.Hk * DK + h * p.dv + rr)));
      }
      vb[idx] = vv;
    }
    for (int idx = tid; idx < n; idx += NT) {
      const size_t ah = static_cast<size_t>(off + idx) * p.Hv + h;
      float a, b;
      front_gates(p.a_raw[ah], p.b_raw[ah], a, b);
      nc[idx] = make_float4(a, b, 0.f, 0.f);
      sch[idx] = mv.sched[off + idx];
      sgt[idx] = mv.seg[off + idx];
    }
    __syncthreads();
  } else {
  // Stage the tree's keys and queries of this key head (cp.async), the
  // values of this CTA's rows, alpha, beta and the steps.  Every global load
  // goes into registers (or a cp.async) before any shared-memory store, so
  // the stage costs one memory round trip.
  {
    const T* kg = static_cast<const T*>(p.k);
    const T* qg = static_cast<const T*>(p.q);
    const T* vg = static_cast<const T*>(p.v);
    constexpr int CPR = DK * static_cast<int>(sizeof(T)) / 16;  // 16-byte chunks of a source row
    constexpr int EPC = 16 / static_cast<int>(sizeof(T));       // elements per chunk
    for (int idx = tid; idx < n * CPR; idx += NT) {
      const int node = idx / CPR, c = idx % CPR;
      const size_t src = (static_cast<size_t>(off + node) * p.Hk + g) * DK + c * EPC;
      cp_async16_g(kb + static_cast<size_t>(node) * DK + c * EPC, kg + src);
      cp_async16_g(qb + static_cast<size_t>(node) * DK + c * EPC, qg + src);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    constexpr int UV = (32 * R + NT - 1) / NT;  // values of a 32-node tree in one batch
    float vv[UV];
#pragma unroll
    for (int u = 0; u < UV; u++) {
      const int idx = tid + u * NT;
      const int rr = rb * R + idx % R;
      vv[u] = (idx < n * R && rr < p.dv) ? to_f32(vg[(static_cast<size_t>(off + idx / R) * p.Hv + h) * p.dv + rr])
                                         : 0.f;
    }
    float a = 0.f, b = 0.f;
    int e = 0, rde = 0;
    if (tid < n) {
      const size_t ah = static_cast<size_t>(off + tid) * p.Hv + h;
      a = p.alpha[ah];
      b = p.beta[ah];
      e = mv.sched[off + tid];
      rde = mv.seg[off + tid];
    }
#pragma unroll
    for (int u = 0; u < UV; u++)
      if (tid + u * NT < n * R) vb[tid + u * NT] = vv[u];
    if (tid < n) {
      nc[tid] = make_float4(a, b, 0.f, 0.f);
      sch[tid] = e;
      sgt[tid] = rde;
    }
    // values and gates of larger trees
    for (int idx = UV * NT + tid; idx < n * R; idx += NT) {
      const int rr = rb * R + idx % R;
      vb[idx] = rr < p.dv ? to_f32(vg[(static_cast<size_t>(off + idx / R) * p.Hv + h) * p.dv + rr]) : 0.f;
    }
    for (int idx = NT + tid; idx < n; idx += NT) {
      const size_t ah = static_cast<size_t>(off + idx) * p.Hv + h;
      nc[idx] = make_float4(p.alpha[ah], p.beta[ah], 0.f, 0.f);
      sch[idx] = mv.sched[off + idx];
      sgt[idx] = mv.seg[off + idx];
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
  }
  }
  // k . q of every node, one node per lane group at a time (warp-uniform
  // trip count, so every lane of a warp takes part in each butterfly)
  for (int base = 0; base < n; base += NG) {
    const int node = base + gi;
    f2_t kk[kPairs], qq[kPairs];
    const int src = node < n ? node : 0;
    load_row_any<LPR>(kk, kb + static_cast<size_t>(src) * DK, j);
    load_row_any<LPR>(qq, qb + static_cast<size_t>(src) * DK, j);
    const float kq = kq_group<LPR>(kk, qq);
    __syncwarp();
    if (node < n && j == 0) nc[node].z = kq;
  }
  __syncthreads();

  T* out = static_cast<T*>(p.out) + (static_cast<size_t>(off) * p.Hv + h) * p.dv + row0;
  float* slot0 = slots + static_cast<size_t>(RPG * gi) * DK;  // the group's rows in slot 0
  const size_t out_stride = static_cast<size_t>(p.Hv) * p.dv;
  const bool vec_store = sizeof(T) == 2 && (RPG == 2 || RPG == 4) && row0 + RPG <= p.dv && (p.dv % RPG) == 0;
  // Outputs go out as explicit global stores: the compiler then knows they
  // cannot alias the shared-memory tables and may issue the next visit's
  // loads ahead of them.
  auto put = [&](int node, const float (&o)[RPG]) {
    T* dst = out + static_cast<size_t>(node) * out_stride;
    if (vec_store) {
      uint32_t w[RPG / 2 > 0 ? RPG / 2 : 1];
#pragma unroll
      for (int i = 0; i + 1 < RPG; i += 2)
        w[i / 2] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(o[i]))) |
                   (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(o[i + 1]))) << 16);
      if constexpr (RPG == 4) {
        asm volatile("st.global.v2.b32 [%0], {%1, %2};" ::"l"(dst), "r"(w[0]), "r"(w[1]));
      } else {
        asm volatile("st.global.b32 [%0], %1;" ::"l"(dst), "r"(w[0]));
      }
    } else {
#pragma unroll
      for (int i = 0; i < RPG; i++)
        if (row0 + i < p.dv) store_global(dst + i, from_f32<T>(o[i]));
    }
  };
  const float scale = p.scale;
  // the first visit's entry, key, query, gates and value; each visit then
  // loads the next one in visit order, across segment ends too (segments are
  // consecutive runs of the visits)
  int e = sch[0];
  f2_t k[kPairs], q[kPairs];
  load_row_any<LPR>(k, kb + static_cast<size_t>(e & 0xFF) * DK, j);
  load_row_any<LPR>(q, qb + static_cast<size_t>(e & 0xFF) * DK, j);
  float4 c4 = nc[e & 0xFF];
  float vv[RPG];
  load_vals<RPG>(vv, vb + (e & 0xFF) * R + RPG * gi);
  for (int sg = 0; sg < n_seg; sg++) {
    const int sw = sgt[sg];
    const int first = sw & 0xFF, cnt = (sw >> 8) & 0xFF, src = (sw >> 16) & 0xFF, save = (sw >> 24) & 0xFF;
    if (src) {
      const float* sl = slot0 + static_cast<size_t>(src - 1) * R * DK;
#pragma unroll
      for (int i = 0; i < RPG; i++) load_row<LPR>(st[i], sl + i * DK, j);
    }
    // the visits of the segment: no branch but the lane-0 store.  Each sum,
    // c and o is formed exactly as gdn_row_step forms it.  The next visit's
    // entry, key, query, gates and value are loaded during this one (the
    // index clamped at the last visit, so the loads need no branch).
    const int last = first + cnt - 1;
#pragma unroll 2
    for (int v = first; v <= last; v++) {
      const int node = e & 0xFF;
      const bool hc = (e >> 24) & 1;
      const int en = sch[v + 1 < n ? v + 1 : v];
      f2_t kn[kPairs], qn[kPairs];
      load_row_any<LPR>(kn, kb + static_cast<size_t>(en & 0xFF) * DK, j);
      load_row_any<LPR>(qn, qb + static_cast<size_t>(en & 0xFF) * DK, j);
      const float4 c4n = nc[en & 0xFF];
      float vn[RPG];
      load_vals<RPG>(vn, vb + (en & 0xFF) * R + RPG * gi);
      float d[2 * RPG];
#pragma unroll
      for (int i = 0; i < RPG; i++) {
        d[2 * i] = row_partial(st[i], k);
        d[2 * i + 1] = row_partial(st[i], q);
      }
      group_sum_n<LPR, 2 * RPG>(d);
      float c[RPG], o[RPG];
#pragma unroll
      for (int i = 0; i < RPG; i++) {
        c[i] = gdn_c(d[2 * i], vv[i], c4.x, c4.y);
        o[i] = gdn_o(c[i], c4.z, c4.x, d[2 * i + 1], scale);
      }
      if (j == 0) put(node, o);
      // a leaf's state is never read, so its update is skipped (the branch
      // is uniform over the CTA: every lane group visits the same node)
      if (hc) {
#pragma unroll
        for (int i = 0; i < RPG; i++) gdn_update(st[i], k, c4.x, c[i]);
      }
      e = en;
#pragma unroll
      for (int i = 0; i < kPairs; i++) {
        k[i] = kn[i];
        q[i] = qn[i];
      }
      c4 = c4n;
#pragma unroll
      for (int i = 0; i < RPG; i++) vv[i] = vn[i];
    }
    if (save) {
      float* sl = slot0 + static_cast<size_t>(save - 1) * R * DK;
#pragma unroll
      for (int i = 0; i < RPG; i++) store_row<LPR>(sl + i * DK, st[i], j);
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
  constexpr int DK = 2 * kPairs * LPR;
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
  f2_t st[kPairs];
  if (valid) {
    load_row<LPR>(st, Srow, j);
  } else {
#pragma unroll
    for (int e = 0; e < kPairs; e++) st[e] = 0ull;
  }
  f2_t kk[kPairs], qq[kPairs];
  load_row<LPR>(kk, kb, j);
  load_row<LPR>(qq, qb, j);
  const float kq = kq_group<LPR>(kk, qq);
  const size_t hi = static_cast<size_t>(s) * p.Hv + h;
  const float vv = valid ? to_f32(static_cast<const T*>(p.v)[hi * p.dv + row]) : 0.f;
  const float o = gdn_row_step<LPR, true>(st, kk, qq, kq, vv, p.alpha[hi], p.beta[hi], p.scale, true);
  if (valid) {
    store_row<LPR>(Srow, st, j);
    if (j == 0) static_cast<T*>(p.out)[hi * p.dv + row] = from_f32<T>(o);
  }
}

static bool gdn_shape_ok(const tv_gdn_layer* l) {
  return l && (l->dtype == TV_F32 || l->dtype == TV_BF16) && l->Hk >= 1 && l->Hv >= l->Hk && l->Hv % l->Hk == 0 &&
         (l->dk == 64 || l->dk == 128) && l->dv >= 1 && l->dv <= 256 && l->S;
}

template <typename T, int LPR, int WARPS, bool FRONT>
static void launch_verify_w(const GdnVerifyParams& p, int n_seq, cudaStream_t st, bool ov) {
  using Sh = GdnShape<LPR, kGdnRpg, WARPS>;
  constexpr int R = Sh::R;
  auto kern = gdn_verify_kernel<T, LPR, kGdnRpg, WARPS, FRONT>;
  static bool attrs = false;  // one-time, sized for the largest tree
  if (!attrs) {
    const int smem_max = static_cast<int>(gdn_verify_smem<T, Sh>(TV_MAX_NODES, slots_for(TV_MAX_NODES)));
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    attrs = true;
  }
  const dim3 grid(p.Hv * ((p.dv + R - 1) / R), n_seq);
  launch_k(ov, kern, grid, dim3(32 * WARPS), gdn_verify_smem<T, Sh>(p.n_max, p.n_slots), st, p);
}
template <typename T, int LPR, bool FRONT>
static void launch_verify(const GdnVerifyParams& p, int n_seq, cudaStream_t st, bool ov) {
  constexpr int R4 = GdnShape<LPR, kGdnRpg, 4>::R;
  const long long ctas4 = static_cast<long long>(p.Hv) * ((p.dv + R4 - 1) / R4) * n_seq;
  if (ctas4 <= 2LL * num_sms()) launch_verify_w<T, LPR, 8, FRONT>(p, n_seq, st, ov);
  else launch_verify_w<T, LPR, 4, FRONT>(p, n_seq, st, ov);
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
    constexpr int LPR = lanes_per_row<128>();
    if (bf) launch_decode<__nv_bfloat16, LPR>(p, n_seq, st); else launch_decode<float, LPR>(p, n_seq, st);
  } else {
    constexpr int LPR = lanes_per_row<64>();
    if (bf) launch_decode<__nv_bfloat16, LPR>(p, n_seq, st); else launch_decode<float, LPR>(p, n_seq, st);
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
    constexpr int LPR = lanes_per_row<128>();
    if (bf) launch_verify<__nv_bfloat16, LPR, false>(p, t->n_seq, st, ov); else launch_verify<float, LPR, false>(p, t->n_seq, st, ov);
  } else {
    constexpr int LPR = lanes_per_row<64>();
    if (bf) launch_verify<__nv_bfloat16, LPR, false>(p, t->n_seq, st, ov); else launch_verify<float, LPR, false>(p, t->n_seq, st, ov);
  }
  return launch_status();
}

// The fused form: the front end computed inside the verify kernel from the
// raw projections (no q, k, v, alpha or beta in memory), then the gated RMS
// norm of the outputs in place.  The norm needs all dv rows of a (node,
// value head), which two CTAs of the verify kernel share, so it is a second
// kernel over `out`.
extern "C" tv_status tv_gdn_tree_verify_fused(const tv_gdn_layer* l, const tv_gdn_front_layer* f, const tv_tree* t,
                                              const void* x, const float* a_raw, const float* b_raw, const void* z,
                                              const float* w_norm, void* out, float scale, tv_stream stream) {
  if (!tree_ok(t)) return TV_ERR_ARG;
  if (!l || !l->S || !f) return TV_ERR_ARG;
  if (l->dtype != TV_F32 && l->dtype != TV_BF16) return TV_ERR_DTYPE;
  if (!gdn_shape_ok(l) || !front_layer_ok(f)) return TV_ERR_SHAPE;
  if (f->dtype != l->dtype || f->Hk != l->Hk || f->Hv != l->Hv || f->dk != l->dk || f->dv != l->dv)
    return TV_ERR_SHAPE;
  if (!x || !a_raw || !b_raw || !z || !w_norm || !out) return TV_ERR_ARG;
  if (!aligned16(out)) return TV_ERR_ALIGN;
  GdnVerifyParams p{};
  for (int s = 0; s < t->n_seq; s++) {
    if (!l->S[s]) return TV_ERR_ARG;
    if (!aligned16(l->S[s])) return TV_ERR_ALIGN;
    if (f->width > 1 && !f->tail[s]) return TV_ERR_ARG;
    p.S[s] = l->S[s];
    p.tail[s] = f->tail[s];
  }
  p.out = out;
  p.meta = t->meta; p.status = t->status;
  p.n_total = t->n_total; p.n_max = t->n_max; p.n_slots = slots_for(t->n_max);
  p.Hk = l->Hk; p.Hv = l->Hv; p.dv = l->dv; p.scale = scale;
  p.x = x; p.a_raw = a_raw; p.b_raw = b_raw; p.wconv = f->wconv;
  p.C = 2 * l->Hk * l->dk + l->Hv * l->dv;
  p.W = f->width;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool bf = l->dtype == TV_BF16;
  const bool ov = tree_overlap(t);
  if (l->dk == 128) {
    constexpr int LPR = lanes_per_row<128>();
    if (bf) launch_verify<__nv_bfloat16, LPR, true>(p, t->n_seq, st, ov); else launch_verify<float, LPR, true>(p, t->n_seq, st, ov);
  } else {
    constexpr int LPR = lanes_per_row<64>();
    if (bf) launch_verify<__nv_bfloat16, LPR, true>(p, t->n_seq, st, ov); else launch_verify<float, LPR, true>(p, t->n_seq, st, ov);
  }
  const tv_status ls = launch_status();
  if (ls != TV_OK) return ls;
  return tv_gdn_out_norm(f, t->n_total, out, z, w_norm, out, stream);
}
