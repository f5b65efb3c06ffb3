// Commit of the accepted path ("One request, end to end" 2.6: the engine
// commits that path's KV rows and recurrent state; "Adding a model", step 4:
// commit_tree / rollback_to).  Verify never writes the caches or the states,
// so rolling back everything past the accepted path costs nothing; commit
// copies the path's K/V rows to rows L..L+a-1 of every attention layer,
// replays the path through every Gated DeltaNet layer's state with the same
// step function verify and decode use, and advances the lengths.
#include <climits>

#include "common.cuh"
#include "gdn_step.cuh"
#include "host.hpp"

namespace tv {

// Layers per launch.  The per-layer pointer blocks travel as kernel
// parameters (up to 32 KB of them on this toolkit and architecture): 64 GDN
// layers take 6.2 KB, so a 48-layer stack commits in one launch instead of
// two that each leave the GPU half busy at their end.
constexpr int kAttnCommitLayers = 16;
constexpr int kGdnCommitLayers = 64;

// Capacity and path-length checks for every sequence, before anything is written.
__global__ void commit_check_kernel(const int32_t* acc_len, const int32_t* len, int32_t* status, int n_seq,
                                    int min_cap) {
  pdl_wait();
  const int s = threadIdx.x;
  if (s >= n_seq || status_bad(status)) return;
  const int a = acc_len[s], L = len[s];
  if (a < 1 || a > TV_MAX_PATH || L < 0) set_status(status, TV_ERR_ARG);
  else if (static_cast<long long>(L) + a > min_cap) set_status(status, TV_ERR_CAPACITY);
}

struct AttnCommitLayer {
  void* K[TV_MAX_SEQ];
  void* V[TV_MAX_SEQ];
  const void* kt;
  const void* vt;
};
struct AttnCommitParams {
  AttnCommitLayer L[kAttnCommitLayers];
  const int32_t* path;
  const int32_t* acc_len;
  const int32_t* len;
  const void* meta;
  int32_t* status;
  int n_total, Hkv, cap, row_bytes;
};

__global__ void __launch_bounds__(128) attn_commit_kernel(const AttnCommitParams p) {
  pdl_wait();
  const int g = blockIdx.x, s = blockIdx.y, li = blockIdx.z;
  if (status_bad(p.status)) return;
  const int a = p.acc_len[s], L = p.len[s];
  const MetaView mv = meta_view(const_cast<void*>(p.meta), p.n_total);
  const int off = mv.seq[s].off;
  const AttnCommitLayer& lay = p.L[li];
  const int chunks = p.row_bytes / 16;
  for (int idx = threadIdx.x; idx < a * chunks; idx += blockDim.x) {
    const int j = idx / chunks, cc = idx % chunks;
    const size_t node = static_cast<size_t>(off + p.path[s * TV_MAX_PATH + j]);
    const size_t src = (node * p.Hkv + g) * p.row_bytes;
    const size_t dst = (static_cast<size_t>(g) * p.cap + L + j) * p.row_bytes;
    reinterpret_cast<uint4*>(static_cast<char*>(lay.K[s]) + dst)[cc] =
        reinterpret_cast<const uint4*>(static_cast<const char*>(lay.kt) + src)[cc];
    reinterpret_cast<uint4*>(static_cast<char*>(lay.V[s]) + dst)[cc] =
        reinterpret_cast<const uint4*>(static_cast<const char*>(lay.vt) + src)[cc];
  }
}

struct GdnCommitLayer {
  float* S[TV_MAX_SEQ];
  const void* k;
  const void* v;
  const float* alpha;
  const float* beta;
};
struct GdnCommitParams {
  GdnCommitLayer L[kGdnCommitLayers];
  const int32_t* path;
  const int32_t* acc_len;
  const void* meta;
  int32_t* status;
  int n_total, Hk, Hv, dv;
};

// Two state rows per lane group (the rows the GDN verify kernel pairs), so
// a CTA of 128 threads replays 2 * 128/LPR rows: half the CTAs of one row
// per group, and two independent replays to overlap.  The rows are loaded
// before the wait: no kernel of the round directly before a commit writes
// the recurrent states.
template <typename T, int LPR>
__global__ void __launch_bounds__(128) gdn_commit_kernel(const GdnCommitParams p) {
  constexpr int DK = 2 * kPairs * LPR;
  constexpr int R = 2 * (128 / LPR);
  const int s = blockIdx.y, li = blockIdx.z;
  const int rb_per_head = (p.dv + R - 1) / R;
  const int h = blockIdx.x / rb_per_head, rb = blockIdx.x % rb_per_head;
  const GdnCommitLayer& lay = p.L[li];
  const int gi = threadIdx.x / LPR, jl = threadIdx.x % LPR;
  const int row0 = rb * R + 2 * gi;
  const bool valid0 = row0 < p.dv, valid1 = row0 + 1 < p.dv;
  float* S0 = lay.S[s] + (static_cast<size_t>(h) * p.dv + (valid0 ? row0 : 0)) * DK;
  float* S1 = lay.S[s] + (static_cast<size_t>(h) * p.dv + (valid1 ? row0 + 1 : 0)) * DK;
  f2_t st0[kPairs], st1[kPairs];
  if (valid0) {
    load_row<LPR>(st0, S0, jl);
  } else {
#pragma unroll
    for (int e = 0; e < kPairs; e++) st0[e] = 0ull;
  }
  if (valid1) {
    load_row<LPR>(st1, S1, jl);
  } else {
#pragma unroll
    for (int e = 0; e < kPairs; e++) st1[e] = 0ull;
  }
  {
    // the keys and values of every node of the sequence into L2 while the
    // accept kernel finishes (the accepted path is only known after the
    // wait): node range from the tree tables, clamped to the buffers (a
    // cache hint)
    const SeqInfo si = meta_view(const_cast<void*>(p.meta), p.n_total).seq[s];
    const int n0 = min(max(si.n, 0), min(TV_MAX_NODES, p.n_total)), off0 = min(max(si.off, 0), p.n_total - n0);
    const int g0 = h / (p.Hv / p.Hk);
    constexpr int KL = DK * static_cast<int>(sizeof(T)) / 128;  // 128-byte lines of a key row
    for (int idx = threadIdx.x; idx < n0 * (KL + 1); idx += 128) {
      const int node = off0 + idx / (KL + 1), part = idx % (KL + 1);
      const char* ad = part < KL ? reinterpret_cast<const char*>(static_cast<const T*>(lay.k) +
                                                                 (static_cast<size_t>(node) * p.Hk + g0) * DK) +
                                       part * 128
                                 : reinterpret_cast<const char*>(static_cast<const T*>(lay.v) +
                                                                 (static_cast<size_t>(node) * p.Hv + h) * p.dv + rb * R);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(ad));
    }
  }
  pdl_wait();
  if (status_bad(p.status)) return;
  const int g = h / (p.Hv / p.Hk);
  const int a = p.acc_len[s];
  if (a < 1 || a > TV_MAX_PATH) return;
  const MetaView mv = meta_view(const_cast<void*>(p.meta), p.n_total);
  const int off = mv.seq[s].off;
  __shared__ __align__(16) float kb[TV_MAX_PATH][DK];
  __shared__ __align__(8) float vb[TV_MAX_PATH][R];
  __shared__ float ab[TV_MAX_PATH], bb[TV_MAX_PATH];
  const T* k = static_cast<const T*>(lay.k);
  const T* v = static_cast<const T*>(lay.v);
  // the path's keys, values, gates: every load issued before any store
  {
    constexpr int UK = TV_MAX_PATH * DK / 128, UV = TV_MAX_PATH * R / 128;
    float kv[UK], vv[UV];
#pragma unroll
    for (int u = 0; u < UK; u++) {
      const int idx = threadIdx.x + 128 * u, j = idx / DK, e = idx % DK;
      kv[u] = j < a ? to_f32(k[(static_cast<size_t>(off + p.path[s * TV_MAX_PATH + j]) * p.Hk + g) * DK + e]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < UV; u++) {
      const int idx = threadIdx.x + 128 * u, j = idx / R, r = idx % R, row = rb * R + r;
      vv[u] = j < a && row < p.dv
                  ? to_f32(v[(static_cast<size_t>(off + p.path[s * TV_MAX_PATH + j]) * p.Hv + h) * p.dv + row])
                  : 0.f;
    }
    float av = 0.f, bv = 0.f;
    if (threadIdx.x < a) {
      const size_t node = static_cast<size_t>(off + p.path[s * TV_MAX_PATH + threadIdx.x]);
      av = lay.alpha[node * p.Hv + h];
      bv = lay.beta[node * p.Hv + h];
    }
#pragma unroll
    for (int u = 0; u < UK; u++) {
      const int idx = threadIdx.x + 128 * u;
      kb[idx / DK][idx % DK] = kv[u];
    }
#pragma unroll
    for (int u = 0; u < UV; u++) {
      const int idx = threadIdx.x + 128 * u;
      vb[idx / R][idx % R] = vv[u];
    }
    if (threadIdx.x < a) {
      ab[threadIdx.x] = av;
      bb[threadIdx.x] = bv;
    }
  }
  __syncthreads();
  for (int j = 0; j < a; j++) {
    f2_t kk[kPairs];
    load_row<LPR>(kk, kb[j], jl);
    const float2 v2 = *reinterpret_cast<const float2*>(&vb[j][2 * gi]);
    gdn_row_step<LPR, false>(st0, kk, kk, 0.f, v2.x, ab[j], bb[j], 0.f, true);
    gdn_row_step<LPR, false>(st1, kk, kk, 0.f, v2.y, ab[j], bb[j], 0.f, true);
  }
  if (valid0) store_row<LPR>(S0, st0, jl);
  if (valid1) store_row<LPR>(S1, st1, jl);
}

__global__ void commit_len_kernel(int32_t* len, const int32_t* acc_len, const int32_t* status, int n_seq) {
  pdl_wait();
  const int s = threadIdx.x;
  if (s < n_seq && !status_bad(status)) len[s] += acc_len[s];
}

template <typename T, int LPR>
static void launch_gdn_commit(const GdnCommitParams& p, int n_seq, int nl, cudaStream_t st, bool ov) {
  constexpr int R = 2 * (128 / LPR);
  const dim3 grid(p.Hv * ((p.dv + R - 1) / R), n_seq, nl);
  launch_k(ov, gdn_commit_kernel<T, LPR>, grid, dim3(128), 0, st, p);
}

}  // namespace tv

using namespace tv;

extern "C" tv_status tv_commit_path(const tv_tree* t, const int32_t* path, const int32_t* acc_len, int32_t n_attn,
                                    const tv_attn_layer* attn, const void* const* k_t, const void* const* v_t,
                                    int32_t n_gdn, const tv_gdn_layer* gdn, const void* const* k,
                                    const void* const* v, const float* const* alpha, const float* const* beta,
                                    int32_t* len, tv_stream stream) {
  if (!tree_ok(t) || !path || !acc_len || !len || n_attn < 0 || n_gdn < 0) return TV_ERR_ARG;
  if (!aligned16(path) || !aligned16(acc_len) || !aligned16(len)) return TV_ERR_ALIGN;
  if (n_attn > 0 && (!attn || !k_t || !v_t)) return TV_ERR_ARG;
  if (n_gdn > 0 && (!gdn || !k || !v || !alpha || !beta)) return TV_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int n_seq = t->n_seq;
  int min_cap = INT_MAX;
  for (int i = 0; i < n_attn; i++) {
    const tv_attn_layer& l = attn[i];
    if (l.Hkv != attn[0].Hkv || l.D != attn[0].D || l.dtype != attn[0].dtype) return TV_ERR_SHAPE;
    if (l.cap < 1 || !l.K || !l.V || !k_t[i] || !v_t[i]) return TV_ERR_ARG;
    if (!aligned16(k_t[i]) || !aligned16(v_t[i])) return TV_ERR_ALIGN;
    for (int s = 0; s < n_seq; s++) {
      if (!l.K[s] || !l.V[s]) return TV_ERR_ARG;
      if (!aligned16(l.K[s]) || !aligned16(l.V[s])) return TV_ERR_ALIGN;
    }
    min_cap = l.cap < min_cap ? l.cap : min_cap;
  }
  for (int i = 0; i < n_gdn; i++) {
    const tv_gdn_layer& l = gdn[i];
    if (l.Hk != gdn[0].Hk || l.Hv != gdn[0].Hv || l.dk != gdn[0].dk || l.dv != gdn[0].dv ||
        l.dtype != gdn[0].dtype)
      return TV_ERR_SHAPE;
    if ((l.dk != 64 && l.dk != 128) || l.Hk < 1 || l.Hv % l.Hk || l.dv < 1 || l.dv > 256) return TV_ERR_SHAPE;
    if (!l.S || !k[i] || !v[i] || !alpha[i] || !beta[i]) return TV_ERR_ARG;
    if (!aligned16(k[i]) || !aligned16(v[i]) || !aligned16(alpha[i]) || !aligned16(beta[i])) return TV_ERR_ALIGN;
    for (int s = 0; s < n_seq; s++) {
      if (!l.S[s]) return TV_ERR_ARG;
      if (!aligned16(l.S[s])) return TV_ERR_ALIGN;
    }
  }
  const bool ov = tree_overlap(t);
  launch_k(ov, commit_check_kernel, dim3(1), dim3(32), 0, st, acc_len, static_cast<const int32_t*>(len), t->status,
           n_seq, min_cap);
  for (int base = 0; base < n_attn; base += kAttnCommitLayers) {
    const int nl = n_attn - base < kAttnCommitLayers ? n_attn - base : kAttnCommitLayers;
    AttnCommitParams p{};
    for (int i = 0; i < nl; i++) {
      for (int s = 0; s < n_seq; s++) {
        p.L[i].K[s] = attn[base + i].K[s];
        p.L[i].V[s] = attn[base + i].V[s];
      }
      p.L[i].kt = k_t[base + i];
      p.L[i].vt = v_t[base + i];
    }
    p.path = path;
    p.acc_len = acc_len;
    p.len = len;
    p.meta = t->meta;
    p.status = t->status;
    p.n_total = t->n_total;
    p.Hkv = attn[0].Hkv;
    p.cap = attn[0].cap;
    p.row_bytes = attn[0].D * (attn[0].dtype == TV_BF16 ? 2 : 4);
    bool same_cap = true;
    for (int i = 0; i < nl; i++) same_cap = same_cap && attn[base + i].cap == p.cap;
    if (!same_cap) return TV_ERR_SHAPE;
    launch_k(ov, attn_commit_kernel, dim3(p.Hkv, n_seq, nl), dim3(128), 0, st, p);
  }
  for (int base = 0; base < n_gdn; base += kGdnCommitLayers) {
    const int nl = n_gdn - base < kGdnCommitLayers ? n_gdn - base : kGdnCommitLayers;
    GdnCommitParams p{};
    for (int i = 0; i < nl; i++) {
      for (int s = 0; s < n_seq; s++) p.L[i].S[s] = gdn[base + i].S[s];
      p.L[i].k = k[base + i];
      p.L[i].v = v[base + i];
      p.L[i].alpha = alpha[base + i];
      p.L[i].beta = beta[base + i];
    }
    p.path = path;
    p.acc_len = acc_len;
    p.meta = t->meta;
    p.status = t->status;
    p.n_total = t->n_total;
    p.Hk = gdn[0].Hk;
    p.Hv = gdn[0].Hv;
    p.dv = gdn[0].dv;
    const bool bf = gdn[0].dtype == TV_BF16;
    if (gdn[0].dk == 128) {
      constexpr int LPR = lanes_per_row<128>();
      if (bf) launch_gdn_commit<__nv_bfloat16, LPR>(p, n_seq, nl, st, ov); else launch_gdn_commit<float, LPR>(p, n_seq, nl, st, ov);
    } else {
      constexpr int LPR = lanes_per_row<64>();
      if (bf) launch_gdn_commit<__nv_bfloat16, LPR>(p, n_seq, nl, st, ov); else launch_gdn_commit<float, LPR>(p, n_seq, nl, st, ov);
    }
  }
  launch_k(ov, commit_len_kernel, dim3(1), dim3(32), 0, st, len, acc_len, static_cast<const int32_t*>(t->status),
           n_seq);
  return launch_status();
}
