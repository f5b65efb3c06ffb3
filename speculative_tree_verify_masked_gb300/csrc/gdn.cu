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
//
// Fused form (tv_gdn_tree_verify_fused; "Adding a model", the Gated
// DeltaNet layer with its gated norm; "The model layer", the convolution
// tails).  The same kernel with the front end in its staging and the gated
// norm after its visits: each node's query, key, value and gates are formed
// from the raw projections in shared memory (front_gdn.cuh's operations in
// tv_gdn_front's order), and the CTAs that share a key head run as one
// thread-block cluster, splitting the key head's queries and keys by node
// and gathering each (node, value head)'s outputs through distributed shared
// memory for the norm.  The result is the three separate calls' bit for bit.
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
  int front_off;  // byte offset of the front-end staging in shared memory
  // gated norm inside the kernel (norm_in): the CTA's outputs staged at
  // obuf_off, each (node, value head)'s then gathered in the head's CTA that
  // normalizes it, out = norm(o) * w_norm * SiLU(z)
  const void* z;
  const float* w_norm;
  int norm_in, obuf_off;
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
constexpr size_t kGdnSmemMax = 232448;  // dynamic shared memory a CTA may opt into

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

// Front-end staging of the fused verify (bytes, each part 16-byte aligned):
// raw rows [W-1+n_max][CH] T (the tail rows, then the nodes'; channels: the
// key head's query and key, then the CTA's value rows) | convolution weights
// [CH][W] f32 | window rows [n_max][8] as byte offsets into the raw rows u32.
// It lies in the slots when they are large enough (nothing uses them before
// the first visit), else after the other tables.
struct FrontLayout {
  size_t xs, ws, win, bytes;
};
__host__ __device__ inline FrontLayout front_layout(int n_max, int W, int DK, int R, int tsize) {
  const size_t CH = 2 * static_cast<size_t>(DK) + R;
  auto a16 = [](size_t b) { return (b + 15) / 16 * 16; };
  FrontLayout f;
  f.xs = 0;
  f.ws = a16(static_cast<size_t>(W - 1 + n_max) * CH * tsize);
  f.win = f.ws + a16(CH * W * 4);
  f.bytes = f.win + a16(static_cast<size_t>(n_max) * 32);
  return f;
}

// Shared-memory accesses by 32-bit shared-window address.
__device__ __forceinline__ uint32_t sh_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float sh_f32(uint32_t a) { return __uint_as_float(sh_u32(a)); }
__device__ __forceinline__ uint4 sh_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ f2_t sh_f2(uint32_t a) {
  f2_t v;
  asm volatile("ld.shared.b64 %0, [%1];" : "=l"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sh_st_f2(uint32_t a, float x, float y) {
  asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(x), "f"(y) : "memory");
}

// Thread-block cluster: rank, size, barrier, peer shared-memory loads.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint4 peer_v4(uint32_t local_addr, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local_addr), "r"(rank));
  uint4 v;
  asm volatile("ld.shared::cluster.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a)
               : "memory");
  return v;
}

__device__ __forceinline__ void peer_st_v4(uint32_t local_addr, uint32_t rank, uint4 v) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local_addr), "r"(rank));
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
// One element of type T at a shared-window address of CTA `rank` of the
// cluster (this CTA's own when rank is its own), widened to fp32.
template <typename T>
__device__ __forceinline__ float cluster_ld(uint32_t local_addr, uint32_t rank, uint32_t self) {
  uint32_t a = local_addr, v;
  if (rank != self) asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local_addr), "r"(rank));
  if constexpr (sizeof(T) == 2) {
    unsigned short h;
    asm volatile("ld.shared::cluster.b16 %0, [%1];" : "=h"(h) : "r"(a) : "memory");
    v = static_cast<uint32_t>(h) << 16;
  } else {
    asm volatile("ld.shared::cluster.b32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  }
  return __uint_as_float(v);
}

// Values of the fused verify: convolution and SiLU of the staged value
// channels (pairs [DK, DK + vch / 2) of the staged row) for a window of WW
// taps at every node, rounded to T, into vb [n][R] f32.  Thread unit u takes
// channels ch, ch + 1 (packed pairs, the weights in registers) of nodes ph,
// ph + NS, ...; four nodes' chains at a time, their loads ahead of their
// stores.  Each value is formed as conv_silu forms it (front_gdn.cuh): taps
// in order from +0, then SiLU.  All addresses are shared-window offsets: xs
// raw rows [.][CH] T, ws weights [CH][WW], wof [n][8] byte offsets of each
// node's window rows within xs.
template <int WW, typename T, int DK, int R, int NT>
__device__ __forceinline__ void front_values(int tid, int vch, int count, uint32_t xs, uint32_t ws, uint32_t wof,
                                             uint32_t vb) {
  constexpr int NB = 4, TS = static_cast<int>(sizeof(T));
  const int np = vch / 2, NS = (count + NB - 1) / NB;
  for (int u = tid; u < np * NS; u += NT) {
    const int ch = 2 * (DK + u % np), ph = u / np;
    f2_t wr[WW];
#pragma unroll
    for (int jj = 0; jj < WW; jj++) wr[jj] = f2_pack(sh_f32(ws + (ch * WW + jj) * 4), sh_f32(ws + ((ch + 1) * WW + jj) * 4));
    const uint32_t xb = xs + ch * TS;
    const uint32_t db = vb + (ch - 2 * DK) * 4;
    {
      const int k0 = ph;
      // the window offsets of the four nodes, then all their taps' loads,
      // then the chains
      uint4 o[NB][WW > 4 ? 2 : 1];
#pragma unroll
      for (int b = 0; b < NB; b++) {
        const int node = min(k0 + b * NS, count - 1);  // past the end: a repeat, not stored
        o[b][0] = sh_v4(wof + node * 32);
        if constexpr (WW > 4) o[b][1] = sh_v4(wof + node * 32 + 16);
      }
      f2_t x2[NB][WW];
#pragma unroll
      for (int b = 0; b < NB; b++)
#pragma unroll
        for (int jj = 0; jj < WW; jj++) {
          const uint4 q4 = o[b][jj / 4];
          const uint32_t off = (jj & 3) == 0 ? q4.x : (jj & 3) == 1 ? q4.y : (jj & 3) == 2 ? q4.z : q4.w;
          if constexpr (TS == 2) {
            const uint32_t w2 = sh_u32(xb + off);
            x2[b][jj] = f2_pack(bf16_lo(w2), bf16_hi(w2));
          } else {
            x2[b][jj] = sh_f2(xb + off);
          }
        }
      f2_t acc[NB];
#pragma unroll
      for (int b = 0; b < NB; b++) {
        acc[b] = 0ull;
#pragma unroll
        for (int jj = 0; jj < WW; jj++) acc[b] = f2_fma(wr[jj], x2[b][jj], acc[b]);
      }
#pragma unroll
      for (int b = 0; b < NB; b++) {
        if (k0 + b * NS < count) {
          const int node = k0 + b * NS;
          float a0, a1;
          f2_unpack(acc[b], a0, a1);
          sh_st_f2(db + node * R * 4, to_f32(from_f32<T>(silu_f(a0))), to_f32(from_f32<T>(silu_f(a1))));
        }
      }
    }
  }
}

// Queries and keys of the fused verify's staged rows for a window of WW
// taps: a warp per (node, vector) of this CTA's share (nodes crank, crank +
// csize, ...; vector 0 the query, 1 the key), lane channels lane + 32e as
// tv_gdn_front holds them: convolution (taps in order), SiLU, division by
// the L2 norm (warp_l2_scale), rounding; the row then goes to every other
// CTA of the cluster at the same offset.  With an even warp count a warp
// keeps to one vector, so its weights stay in registers.
template <int WW, typename T, typename KQ, int DK, int R, int WARPS>
__device__ __forceinline__ void front_qk(int warp, int lane, uint32_t crank, uint32_t csize, int own, const T* xs,
                                        const float* ws, const uint32_t* wof, KQ* qb, KQ* kb) {
  constexpr int CPL = DK / 32, CPV = DK * static_cast<int>(sizeof(KQ)) / 16;
  static_assert(WARPS % 2 == 0, "a warp keeps to one vector");
  const int is_k = warp & 1;
  float wr[CPL][WW];
#pragma unroll
  for (int e = 0; e < CPL; e++)
#pragma unroll
    for (int jj = 0; jj < WW; jj++) wr[e][jj] = ws[(is_k * DK + lane + 32 * e) * WW + jj];
  for (int t = warp; t < 2 * own; t += WARPS) {
    const int node = static_cast<int>(crank + csize * (t >> 1));
    int off[WW];
#pragma unroll
    for (int jj = 0; jj < WW; jj++) off[jj] = static_cast<int>(wof[node * 8 + jj] / sizeof(T));
    float val[CPL];
#pragma unroll
    for (int e = 0; e < CPL; e++) {
      const int c = is_k * DK + lane + 32 * e;
      float acc = 0.f;
#pragma unroll
      for (int jj = 0; jj < WW; jj++) acc = __fmaf_rn(wr[e][jj], to_f32(xs[off[jj] + c]), acc);
      val[e] = silu_f(acc);
    }
    const float sc = warp_l2_scale<CPL>(val);
    KQ* dst = (is_k ? kb : qb) + static_cast<size_t>(node) * DK;
#pragma unroll
    for (int e = 0; e < CPL; e++) dst[lane + 32 * e] = from_f32<KQ>(__fmul_rn(val[e], sc));
    if (csize > 1) {
      __syncwarp();
      const uint32_t a0 = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
      for (int i = lane; i < CPV * static_cast<int>(csize - 1); i += 32) {
        const uint32_t a = a0 + (i % CPV) * 16;
        const uint32_t peer = (crank + 1 + static_cast<uint32_t>(i / CPV)) % csize;
        uint4 v;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
        peer_st_v4(a, peer, v);
      }
    }
  }
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
  extern __shared__ float4 smem4[];
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
  if constexpr (!FRONT) {
    // this CTA's node inputs into L2 while the previous kernel finishes (the
    // key head's key and query rows, the head's value rows of this CTA): the
    // node range comes from the tree tables, written at the start of the
    // round, and is clamped to the buffers, so a stale read only warms
    // other rows of the same inputs
    const SeqInfo si = meta_view(const_cast<void*>(p.meta), p.n_total).seq[s];
    const int n0 = min(max(si.n, 0), min(p.n_max, p.n_total)), off0 = min(max(si.off, 0), p.n_total - n0);
    const int g0 = h / (p.Hv / p.Hk);
    constexpr int KL = DK * static_cast<int>(sizeof(T)) / 128;  // 128-byte lines of a key row
    for (int idx = tid; idx < n0 * (2 * KL + 1); idx += 32 * WARPS) {
      const int node = off0 + idx / (2 * KL + 1), part = idx % (2 * KL + 1);
      const char* a;
      if (part < 2 * KL) {
        const T* base = static_cast<const T*>(part < KL ? p.k : p.q);
        a = reinterpret_cast<const char*>(base + (static_cast<size_t>(node) * p.Hk + g0) * DK) + (part % KL) * 128;
      } else {
        a = reinterpret_cast<const char*>(static_cast<const T*>(p.v) +
                                          (static_cast<size_t>(node) * p.Hv + h) * p.dv + rb * R);
      }
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
    }
  }
  if constexpr (FRONT) {
    // the convolution weights of the CTA's channels (constant: no earlier
    // kernel writes them) start on their way before the wait
    const int g0 = h / (p.Hv / p.Hk), vch0 = min(R, p.dv - rb * R);
    float* ws = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(smem4) + p.front_off +
                                         front_layout(p.n_max, p.W, DK, R, static_cast<int>(sizeof(T))).ws);
    const size_t v0 = static_cast<size_t>(2) * p.Hk * DK + static_cast<size_t>(h) * p.dv + rb * R;
    const int wq = DK * p.W / 4, wv = vch0 * p.W / 4;  // 16-byte chunks
    for (int idx = tid; idx < 2 * wq + wv; idx += 32 * WARPS) {
      const size_t src = idx < wq ? static_cast<size_t>(g0) * DK * p.W + idx * 4
                                  : (idx < 2 * wq ? static_cast<size_t>(p.Hk + g0) * DK * p.W + (idx - wq) * 4
                                                  : v0 * p.W + (idx - 2 * wq) * 4);
      cp_async16_g(ws + idx * 4, p.wconv + src);
    }
  }
  pdl_wait();  // tree tables, status and node inputs come from earlier kernels
  pdl_trigger();
  MetaView mv = meta_view(const_cast<void*>(p.meta), p.n_total);
  const SeqInfo info = mv.seq[s];
  // The fused form may run in clusters of the CTAs that share a key head
  // (they split its queries and keys by node, then exchange them, and gather
  // each head's outputs for the norm): a CTA that leaves early still takes
  // the cluster's barriers (the exchange's and, with the norm inside, the
  // gather's), so none waits on it.  The status word can change under the launch, so CTAs of one
  // cluster can take different paths here (each CTA decides as one: its
  // threads vote).
  uint32_t crank = 0, csize = 1;
  if constexpr (FRONT) {
    crank = cluster_rank();
    csize = cluster_size();
  }
  auto leave = [&]() {
    if (FRONT) asm volatile("cp.async.wait_all;" ::: "memory");  // the weights' copies land before the CTA leaves
    if (FRONT && csize > 1) {
      cluster_sync_all();                  // the exchange of queries and keys
      if (p.norm_in) cluster_sync_all();  // the outputs gathered
    }
  };
  if (FRONT ? __syncthreads_or(status_bad(p.status)) != 0 : status_bad(p.status)) {
    leave();
    return;
  }
  const int n = info.n, off = info.off, n_seg = info.n_seg;
  if (n <= 0 || n > p.n_max || n_seg < 1 || n_seg > n) {
    leave();
    return;
  }
  if (info.max_slot > p.n_slots) {
    if (tid == 0) set_status(p.status, TV_ERR_TREE);
    leave();
    return;
  }
  const int g = h / (p.Hv / p.Hk);

  float* slots = reinterpret_cast<float*>(smem4);  // [n_slots][R][DK]
  KQ* kb = reinterpret_cast<KQ*>(slots + static_cast<size_t>(p.n_slots) * R * DK);
  const size_t kq_bytes = (static_cast<size_t>(p.n_max) * DK * sizeof(KQ) + 15) / 16 * 16;
  KQ* qb = reinterpret_cast<KQ*>(reinterpret_cast<uint8_t*>(kb) + kq_bytes);
  float4* nc = reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(qb) + kq_bytes);  // [n_max]
  float* vb = reinterpret_cast<float*>(nc + p.n_max);                                // [n_max][R]
  int* sch = reinterpret_cast<int*>(vb + static_cast<size_t>(p.n_max) * R);          // [n_max] visits
  int* sgt = sch + p.n_max;                                                           // [n_max] segments

  if constexpr (FRONT) {
    // The front end, as tv_gdn_front forms it (front_gdn.cuh), in one memory
    // round trip: the raw rows this CTA reads (the sequence's tail and its
    // nodes, at the key head's query and key channels and the CTA's value
    // rows), the convolution weights of those channels (copied before the
    // wait), each node's window rows and, with the norm inside, z and w_norm
    // go to shared memory; then the values of the CTA's rows at every node
    // (convolution, SiLU, rounding), and the queries and keys of the CTA's
    // share of the nodes (convolution, SiLU, division by the L2 norm,
    // rounding), sent to the cluster's other CTAs.
    constexpr int CH = 2 * DK + R, EPC = 16 / static_cast<int>(sizeof(T));
    const int W = p.W, W1 = p.W - 1;
    const int vch = min(R, p.dv - rb * R);  // value channels this CTA holds
    const FrontLayout fl = front_layout(p.n_max, W, DK, R, static_cast<int>(sizeof(T)));
    uint8_t* fb = reinterpret_cast<uint8_t*>(smem4) + p.front_off;
    T* xs = reinterpret_cast<T*>(fb + fl.xs);
    float* ws = reinterpret_cast<float*>(fb + fl.ws);
    uint32_t* wof = reinterpret_cast<uint32_t*>(fb + fl.win);
    {
      // the loads of this thread's node (one node a thread: n <= 64 < NT)
      // go first, so their round trip overlaps the copies' issue
      static_assert(TV_MAX_NODES <= NT, "one node per thread");
      const bool has_node = tid < n;
      int depth = 0, e_s = 0, e_g = 0;
      ulonglong2 anc = make_ulonglong2(0ull, 0ull);  // the node's ancestors, one byte per depth
      float a_in = 0.f, b_in = 0.f;
      if (has_node) {
        const int row = off + tid;
        depth = mv.depth[row];
        anc = *reinterpret_cast<const ulonglong2*>(mv.anc_at + static_cast<size_t>(row) * TV_MAX_PATH);
        a_in = p.a_raw[static_cast<size_t>(row) * p.Hv + h];
        b_in = p.b_raw[static_cast<size_t>(row) * p.Hv + h];
        e_s = mv.sched[row];
        e_g = mv.seg[row];
      }
      const T* x = static_cast<const T*>(p.x);
      const T* tail = static_cast<const T*>(p.tail[s]);
      const int cq = DK / EPC, cpr = 2 * cq + vch / EPC;  // chunks of a row
      const size_t v0 = static_cast<size_t>(2) * p.Hk * DK + static_cast<size_t>(h) * p.dv + rb * R;
      // a warp a row, lanes over the row's chunks (each lane's source
      // channels fixed across rows)
      constexpr int CU = ((2 * DK + R) * static_cast<int>(sizeof(T)) / 16 + 31) / 32;
      const int lane0 = tid & 31, warp0 = tid >> 5;
      size_t chan[CU];
#pragma unroll
      for (int u = 0; u < CU; u++) {
        const int c = lane0 + 32 * u;
        chan[u] = c < cq ? static_cast<size_t>(g) * DK + c * EPC
                         : (c < 2 * cq ? static_cast<size_t>(p.Hk + g) * DK + (c - cq) * EPC : v0 + (c - 2 * cq) * EPC);
      }
      for (int r = warp0; r < W1 + n; r += WARPS) {
        const T* row = r < W1 ? tail + static_cast<size_t>(r) * p.C : x + static_cast<size_t>(off + r - W1) * p.C;
        T* dst = xs + static_cast<size_t>(r) * CH;
#pragma unroll
        for (int u = 0; u < CU; u++)
          if (lane0 + 32 * u < cpr) cp_async16_g(dst + (lane0 + 32 * u) * EPC, row + chan[u]);
      }
      if (p.norm_in) {
        // z of the nodes this CTA normalizes (rb, rb + rbph, ...) and w_norm
        T* zs = reinterpret_cast<T*>(reinterpret_cast<uint8_t*>(smem4) + p.obuf_off) +
                (static_cast<size_t>(p.n_max) * R + static_cast<size_t>((p.n_max + rb_per_head - 1) / rb_per_head) *
                                                        rb_per_head * R);
        float* wns = reinterpret_cast<float*>(zs + static_cast<size_t>((p.n_max + rb_per_head - 1) / rb_per_head) *
                                                       rb_per_head * R);
        const int nz = (n - rb + rb_per_head - 1) / rb_per_head, cz = p.dv / EPC;  // rows, chunks of a row
        const int dvp = rb_per_head * R;
        const T* z = static_cast<const T*>(p.z);
        for (int idx = tid; idx < nz * cz; idx += NT) {
          const int k = idx / cz, c = idx % cz;
          cp_async16_g(zs + static_cast<size_t>(k) * dvp + c * EPC,
                       z + (static_cast<size_t>(off + rb + k * rb_per_head) * p.Hv + h) * p.dv + c * EPC);
        }
        for (int idx = tid; idx < p.dv / 4; idx += NT) cp_async16_g(wns + idx * 4, p.w_norm + idx * 4);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      if (has_node) {
        const int idx = tid;
        for (int jj = 0; jj < W; jj++) {
          const int m = depth + jj - W1;  // window element jj: ancestor at depth m, or tail row m + W - 1
          const int am = static_cast<int8_t>(((m < 8 ? anc.x : anc.y) >> (8 * (m & 7))) & 0xFF);
          wof[idx * 8 + jj] = static_cast<uint32_t>((m < 0 ? m + W1 : W1 + am) * CH * static_cast<int>(sizeof(T)));
        }
        float a, b;
        front_gates(a_in, b_in, a, b);
        nc[idx] = make_float4(a, b, 0.f, 0.f);
        sch[idx] = e_s;
        sgt[idx] = e_g;
      }
      if (vch < R)
        for (int idx = tid; idx < n * R; idx += NT)
          if (idx % R >= vch) vb[idx] = 0.f;
      asm volatile("cp.async.wait_all;" ::: "memory");
      __syncthreads();
    }
    {
      const uint32_t xs_s = static_cast<uint32_t>(__cvta_generic_to_shared(xs));
      const uint32_t ws_s = static_cast<uint32_t>(__cvta_generic_to_shared(ws));
      const uint32_t wo_s = static_cast<uint32_t>(__cvta_generic_to_shared(wof));
      const uint32_t vb_s = static_cast<uint32_t>(__cvta_generic_to_shared(vb));
      // the values of this CTA's rows at every node (threads over channel
      // pairs), then this CTA's share of the queries and keys (warps over
      // nodes crank, crank + csize, ...), each row sent to the cluster
      const int own = (n - static_cast<int>(crank) + static_cast<int>(csize) - 1) / static_cast<int>(csize);
      const int warp = tid >> 5, lane = tid & 31;
#define TV_FRONT_CONV(WW)                                                                                   \
  front_values<WW, T, DK, R, NT>(tid, vch, n, xs_s, ws_s, wo_s, vb_s);                                      \
  front_qk<WW, T, KQ, DK, R, WARPS>(warp, lane, crank, csize, own, xs, ws, wof, qb, kb)
      switch (W) {
        case 1: TV_FRONT_CONV(1); break;
        case 2: TV_FRONT_CONV(2); break;
        case 3: TV_FRONT_CONV(3); break;
        case 4: TV_FRONT_CONV(4); break;
        case 5: TV_FRONT_CONV(5); break;
        case 6: TV_FRONT_CONV(6); break;
        case 7: TV_FRONT_CONV(7); break;
        default: TV_FRONT_CONV(8); break;
      }
#undef TV_FRONT_CONV
    }
    // every CTA's rows in place everywhere (the cluster's barrier), or this
    // CTA's own
    if (csize > 1) cluster_sync_all(); else __syncthreads();
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
  // fused form with the norm: this CTA's output rows of every node go to
  // stage [n_max][R] (shared memory), gathered after the visits
  const int dvp = rb_per_head * R;
  T* stage = FRONT ? reinterpret_cast<T*>(reinterpret_cast<uint8_t*>(smem4) + p.obuf_off) : nullptr;
  auto put = [&](int node, const float (&o)[RPG]) {
    if (FRONT && p.norm_in) {
#pragma unroll
      for (int i = 0; i < RPG; i++) stage[node * R + RPG * gi + i] = from_f32<T>(o[i]);
      return;
    }
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
#pragma unroll 4
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
  if constexpr (FRONT) {
    if (p.norm_in) {
      // gated norm of (node, head h) for this CTA's nodes rb, rb + rbph, ...,
      // two a warp at a time (z and w_norm staged with the front end)
      constexpr int CPL = DK / 32;  // the front end's dv = dk
      const int warp = tid >> 5, lane = tid & 31;
      T* o_out = static_cast<T*>(p.out);
      // gather: node k's rows go to the head's CTA k mod rb_per_head, which
      // holds the node's dv outputs at obuf[k / rb_per_head][.] (this CTA's
      // at rb R ..): 16-byte chunks, stored into peers directly
      const int stage_b = p.n_max * R * static_cast<int>(sizeof(T));
      const uint32_t st_s = static_cast<uint32_t>(__cvta_generic_to_shared(stage));
      const uint32_t ob_s = st_s + stage_b;
      const T* obuf = stage + p.n_max * R;
      {
        __syncthreads();
        constexpr int CPN = R * static_cast<int>(sizeof(T)) / 16;  // chunks of a node's rows
        for (int idx = tid; idx < n * CPN; idx += NT) {
          const int node = idx / CPN, c = idx % CPN, owner = node % rb_per_head;
          uint4 v;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                       : "r"(st_s + node * R * static_cast<int>(sizeof(T)) + c * 16));
          const uint32_t a = ob_s + ((node / rb_per_head) * dvp + rb * R) * static_cast<int>(sizeof(T)) + c * 16;
          if (owner == rb) {
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                         : "memory");
          } else {
            peer_st_v4(a, static_cast<uint32_t>(h * rb_per_head + owner) % csize, v);
          }
        }
      }
      auto row = [&](int k) { return (static_cast<size_t>(off + rb + k * rb_per_head) * p.Hv + h) * p.dv; };
      const int nrows = (p.n_max + rb_per_head - 1) / rb_per_head;
      const T* zs = obuf + static_cast<size_t>(nrows) * dvp;  // staged z rows, then w_norm
      const float* wns = reinterpret_cast<const float*>(zs + static_cast<size_t>(nrows) * dvp);
      float wn[CPL];
#pragma unroll
      for (int e = 0; e < CPL; e++) wn[e] = wns[lane + 32 * e];
      if (csize > 1) cluster_sync_all(); else __syncthreads();
      for (int k = warp; rb + k * rb_per_head < n; k += 2 * WARPS) {
        const int k2 = k + WARPS;
        const bool has2 = rb + k2 * rb_per_head < n;
        float oa[CPL], ob[CPL], za[CPL], zb[CPL];
#pragma unroll
        for (int e = 0; e < CPL; e++) {
          oa[e] = to_f32(obuf[k * dvp + lane + 32 * e]);
          za[e] = to_f32(zs[k * dvp + lane + 32 * e]);
          ob[e] = has2 ? to_f32(obuf[k2 * dvp + lane + 32 * e]) : 0.f;
          zb[e] = has2 ? to_f32(zs[k2 * dvp + lane + 32 * e]) : 0.f;
        }
        gated_norm_vals<T, CPL>(oa, za, wn, o_out + row(k), lane);
        if (has2) gated_norm_vals<T, CPL>(ob, zb, wn, o_out + row(k2), lane);
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

// Fused decode: tv_gdn_front (one token a sequence), the decode step of
// tv_decode_step and tv_gdn_out_norm in one kernel, one CTA of 256 threads
// per (value head, sequence) owning all dv rows (RPG = dv / (256 / LPR) rows
// a lane group, one after another), so the gated norm needs no other CTA.
// Every value is formed as the three calls form it: the front end with
// front_gdn.cuh's operations (queries and keys rounded to the layer type and
// widened, as the decode kernel stages them), each row's step with
// gdn_row_step, the norm with gated_norm_vals.
struct GdnDecodeFusedParams {
  float* S[TV_MAX_SEQ];
  const void* tail[TV_MAX_SEQ];
  const void* x;
  const float* a_raw;
  const float* b_raw;
  const float* wconv;
  const void* z;
  const float* w_norm;
  void* out;
  int32_t* status;
  int Hk, Hv, dv, C, W;
  float scale;
};

template <typename T, int LPR>
__global__ void __launch_bounds__(256) gdn_decode_fused_kernel(const GdnDecodeFusedParams p) {
  constexpr int DK = 2 * kPairs * LPR, NT = 256, NG = NT / LPR, CPL = DK / 32, RPG = DK / NG;
  const int h = blockIdx.x, s = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gi = tid / LPR, j = tid % LPR;
  if (__syncthreads_or(status_bad(p.status))) return;
  const int g = h / (p.Hv / p.Hk);
  // this lane group's state rows (gi, gi + NG, ...) first: their loads run
  // under the front end
  f2_t st[RPG][kPairs];
#pragma unroll
  for (int i = 0; i < RPG; i++)
    load_row<LPR>(st[i], p.S[s] + (static_cast<size_t>(h) * p.dv + gi + i * NG) * DK, j);
  __shared__ __align__(16) float kb[DK];
  __shared__ __align__(16) float qb[DK];
  __shared__ float vbuf[DK];  // dv = dk
  __shared__ T obuf[DK];
  __shared__ float gates[2];
  const T* x = static_cast<const T*>(p.x);
  const T* tail = static_cast<const T*>(p.tail[s]);
  int src[kMaxConvWidth];
  conv_window(src, p.W, 0, s, nullptr, s);  // a decoded token: the tail, then itself
  if (warp < 2) {
    // warp 0 the query, warp 1 the key: convolution, SiLU, L2 norm, rounding
    const int c0 = (warp == 0 ? g : p.Hk + g) * DK;
    float val[CPL];
#pragma unroll
    for (int e = 0; e < CPL; e++) val[e] = conv_silu(x, tail, p.wconv, p.C, p.W, src, c0 + lane + 32 * e);
    const float sc = warp_l2_scale<CPL>(val);
    float* dst = warp == 0 ? qb : kb;
#pragma unroll
    for (int e = 0; e < CPL; e++) dst[lane + 32 * e] = to_f32(from_f32<T>(__fmul_rn(val[e], sc)));
  }
  for (int c = tid; c < p.dv; c += NT)
    vbuf[c] = to_f32(from_f32<T>(conv_silu(x, tail, p.wconv, p.C, p.W, src, 2 * p.Hk * DK + h * p.dv + c)));
  if (tid == 0) front_gates(p.a_raw[static_cast<size_t>(s) * p.Hv + h], p.b_raw[static_cast<size_t>(s) * p.Hv + h],
                            gates[0], gates[1]);
  __syncthreads();
  f2_t kk[kPairs], qq[kPairs];
  load_row<LPR>(kk, kb, j);
  load_row<LPR>(qq, qb, j);
  const float kq = kq_group<LPR>(kk, qq);
  const float alpha = gates[0], beta = gates[1];
#pragma unroll
  for (int i = 0; i < RPG; i++) {
    const int row = gi + i * NG;
    const float o = gdn_row_step<LPR, true>(st[i], kk, qq, kq, vbuf[row], alpha, beta, p.scale, true);
    store_row<LPR>(p.S[s] + (static_cast<size_t>(h) * p.dv + row) * DK, st[i], j);
    if (j == 0) obuf[row] = from_f32<T>(o);
  }
  __syncthreads();
  if (warp == 0) {
    const size_t base = (static_cast<size_t>(s) * p.Hv + h) * p.dv;
    const T* z = static_cast<const T*>(p.z) + base;
    float ov[CPL], zv[CPL], wn[CPL];
#pragma unroll
    for (int e = 0; e < CPL; e++) {
      ov[e] = to_f32(obuf[lane + 32 * e]);
      zv[e] = to_f32(z[lane + 32 * e]);
      wn[e] = p.w_norm[lane + 32 * e];
    }
    gated_norm_vals<T, CPL>(ov, zv, wn, static_cast<T*>(p.out) + base, lane);
  }
}

static bool gdn_shape_ok(const tv_gdn_layer* l) {
  return l && (l->dtype == TV_F32 || l->dtype == TV_BF16) && l->Hk >= 1 && l->Hv >= l->Hk && l->Hv % l->Hk == 0 &&
         (l->dk == 64 || l->dk == 128) && l->dv >= 1 && l->dv <= 256 && l->S;
}

// Whether clusters of G CTAs of this kernel and shared memory can be placed
// at all (answers cached per kernel, size and shared memory).
static bool cluster_fits(const void* kern, int G, dim3 grid, dim3 block, size_t smem) {
  struct Entry {
    const void* k;
    int G;
    size_t smem;
    bool ok;
  };
  static Entry cache[64];
  static int n_cache = 0;
  for (int i = 0; i < n_cache; i++)
    if (cache[i].k == kern && cache[i].G == G && cache[i].smem == smem) return cache[i].ok;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = G;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n_clusters = 0;
  const bool ok = cudaOccupancyMaxActiveClusters(&n_clusters, kern, &cfg) == cudaSuccess && n_clusters > 0;
  cudaGetLastError();
  if (n_cache < 64) cache[n_cache++] = {kern, G, smem, ok};
  return ok;
}

// Shared memory of the fused verify (front-end staging inside the slots when
// it fits, else after the tables; the norm's output rows last) and the
// offsets it places.
template <typename T, typename Sh>
static size_t fused_smem(const GdnVerifyParams& p, bool norm_in, int* front_off, int* obuf_off) {
  size_t smem = gdn_verify_smem<T, Sh>(p.n_max, p.n_slots);
  *front_off = 0;
  const size_t fb = front_layout(p.n_max, p.W, Sh::DK, Sh::R, static_cast<int>(sizeof(T))).bytes;
  if (fb > static_cast<size_t>(p.n_slots) * Sh::R * Sh::DK * 4) {
    *front_off = static_cast<int>((smem + 15) / 16 * 16);
    smem = *front_off + fb;
  }
  *obuf_off = static_cast<int>((smem + 15) / 16 * 16);
  const int rbph = (p.dv + Sh::R - 1) / Sh::R;
  // stage [n_max][R], gathered outputs and staged z [ceil(n_max / rbph)][rbph R] each, w_norm [rbph R] f32
  if (norm_in)
    smem = *obuf_off +
           (static_cast<size_t>(p.n_max) + 2 * static_cast<size_t>((p.n_max + rbph - 1) / rbph) * rbph) * Sh::R *
               sizeof(T) +
           static_cast<size_t>(rbph) * Sh::R * 4;
  return smem;
}

// Launches the verify kernel; for the fused form, returns whether the gated
// norm ran inside it (else the caller runs tv_gdn_out_norm over out).
template <typename T, int LPR, int WARPS, bool FRONT>
static bool launch_verify_w(const GdnVerifyParams& p, int n_seq, cudaStream_t st, bool ov) {
  using Sh = GdnShape<LPR, kGdnRpg, WARPS>;
  constexpr int R = Sh::R;
  auto kern = gdn_verify_kernel<T, LPR, kGdnRpg, WARPS, FRONT>;
  static bool attrs = false;  // one-time, sized for the largest tree
  if (!attrs) {
    const size_t smem_max = FRONT ? kGdnSmemMax : gdn_verify_smem<T, Sh>(TV_MAX_NODES, slots_for(TV_MAX_NODES));
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_max));
    if (FRONT) cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    attrs = true;
  }
  const dim3 grid(p.Hv * ((p.dv + R - 1) / R), n_seq);
  if (!FRONT) {
    launch_k(ov, kern, grid, dim3(32 * WARPS), gdn_verify_smem<T, Sh>(p.n_max, p.n_slots), st, p);
    return false;
  }
  // clusters of the CTAs that share a key head (heads per key head x row
  // blocks per head, at most 16): they split its queries and keys by node,
  // and gather each head's outputs for the norm
  const int rbph = (p.dv + R - 1) / R;
  int G = (p.Hv / p.Hk) * rbph;
  if (G > 16) G = 1;
  GdnVerifyParams q = p;
  const bool norm_fits = fused_smem<T, Sh>(p, true, &q.front_off, &q.obuf_off) <= kGdnSmemMax;
  size_t smem = fused_smem<T, Sh>(p, norm_fits, &q.front_off, &q.obuf_off);
  if (G > 1 && !cluster_fits(reinterpret_cast<const void*>(kern), G, grid, dim3(32 * WARPS), smem)) G = 1;
  q.norm_in = norm_fits && (G > 1 || rbph == 1) ? 1 : 0;
  smem = fused_smem<T, Sh>(p, q.norm_in != 0, &q.front_off, &q.obuf_off);
  if (G > 1) launch_k_cluster(ov, G, kern, grid, dim3(32 * WARPS), smem, st, q);
  else launch_k(ov, kern, grid, dim3(32 * WARPS), smem, st, q);
  return q.norm_in != 0;
}
template <typename T, int LPR, bool FRONT>
static bool launch_verify(const GdnVerifyParams& p, int n_seq, cudaStream_t st, bool ov) {
  constexpr int R4 = GdnShape<LPR, kGdnRpg, 4>::R;
  const long long ctas4 = static_cast<long long>(p.Hv) * ((p.dv + R4 - 1) / R4) * n_seq;
  bool four = ctas4 > 2LL * num_sms();
  if (FRONT && four) {  // the fused form's tables must fit CTAs of four warps
    int fo, oo;
    four = fused_smem<T, GdnShape<LPR, kGdnRpg, 4>>(p, false, &fo, &oo) <= kGdnSmemMax;
  }
  return four ? launch_verify_w<T, LPR, 4, FRONT>(p, n_seq, st, ov) : launch_verify_w<T, LPR, 8, FRONT>(p, n_seq, st, ov);
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
// norm of the outputs.  The norm of a (node, value head) needs all dv rows,
// which the head's CTAs share: they run as one cluster (with the other heads
// of the key head) and gather the rows through distributed shared memory.
// Where no such cluster can be placed (more than 16 CTAs to a key head) the
// norm runs as a second kernel over `out`.
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
  if (!aligned16(out) || !aligned16(x) || !aligned16(f->wconv) || !aligned16(z) || !aligned16(w_norm))
    return TV_ERR_ALIGN;
  GdnVerifyParams p{};
  for (int s = 0; s < t->n_seq; s++) {
    if (!l->S[s]) return TV_ERR_ARG;
    if (!aligned16(l->S[s])) return TV_ERR_ALIGN;
    if (f->width > 1 && !f->tail[s]) return TV_ERR_ARG;
    if (f->width > 1 && !aligned16(f->tail[s])) return TV_ERR_ALIGN;
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
  p.z = z; p.w_norm = w_norm;
  const bool bf = l->dtype == TV_BF16;
  const bool ov = tree_overlap(t);
  bool norm_in;
  if (l->dk == 128) {
    constexpr int LPR = lanes_per_row<128>();
    norm_in = bf ? launch_verify<__nv_bfloat16, LPR, true>(p, t->n_seq, st, ov) : launch_verify<float, LPR, true>(p, t->n_seq, st, ov);
  } else {
    constexpr int LPR = lanes_per_row<64>();
    norm_in = bf ? launch_verify<__nv_bfloat16, LPR, true>(p, t->n_seq, st, ov) : launch_verify<float, LPR, true>(p, t->n_seq, st, ov);
  }
  const tv_status ls = launch_status();
  if (ls != TV_OK || norm_in) return ls;
  return tv_gdn_out_norm(f, t->n_total, out, z, w_norm, out, stream);
}

extern "C" tv_status tv_gdn_decode_fused(const tv_gdn_layer* l, const tv_gdn_front_layer* f, int32_t n_seq,
                                         const void* x, const float* a_raw, const float* b_raw, const void* z,
                                         const float* w_norm, void* out, float scale, int32_t* status,
                                         tv_stream stream) {
  if (!l || !l->S || !f) return TV_ERR_ARG;
  if (l->dtype != TV_F32 && l->dtype != TV_BF16) return TV_ERR_DTYPE;
  if (!gdn_shape_ok(l) || !front_layer_ok(f)) return TV_ERR_SHAPE;
  if (f->dtype != l->dtype || f->Hk != l->Hk || f->Hv != l->Hv || f->dk != l->dk || f->dv != l->dv)
    return TV_ERR_SHAPE;
  if (n_seq < 1 || n_seq > TV_MAX_SEQ || !x || !a_raw || !b_raw || !z || !w_norm || !out || !status)
    return TV_ERR_ARG;
  if (!aligned16(status)) return TV_ERR_ALIGN;
  GdnDecodeFusedParams p{};
  for (int s = 0; s < n_seq; s++) {
    if (!l->S[s]) return TV_ERR_ARG;
    if (!aligned16(l->S[s])) return TV_ERR_ALIGN;
    if (f->width > 1 && !f->tail[s]) return TV_ERR_ARG;
    p.S[s] = l->S[s];
    p.tail[s] = f->tail[s];
  }
  p.x = x; p.a_raw = a_raw; p.b_raw = b_raw; p.wconv = f->wconv; p.z = z; p.w_norm = w_norm; p.out = out;
  p.status = status;
  p.Hk = l->Hk; p.Hv = l->Hv; p.dv = l->dv; p.C = 2 * l->Hk * l->dk + l->Hv * l->dv; p.W = f->width;
  p.scale = scale;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const dim3 grid(l->Hv, n_seq);
  const bool bf = l->dtype == TV_BF16;
  if (l->dk == 128) {
    constexpr int LPR = lanes_per_row<128>();
    if (bf) gdn_decode_fused_kernel<__nv_bfloat16, LPR><<<grid, 256, 0, st>>>(p);
    else gdn_decode_fused_kernel<float, LPR><<<grid, 256, 0, st>>>(p);
  } else {
    constexpr int LPR = lanes_per_row<64>();
    if (bf) gdn_decode_fused_kernel<__nv_bfloat16, LPR><<<grid, 256, 0, st>>>(p);
    else gdn_decode_fused_kernel<float, LPR><<<grid, 256, 0, st>>>(p);
  }
  return launch_status();
}
