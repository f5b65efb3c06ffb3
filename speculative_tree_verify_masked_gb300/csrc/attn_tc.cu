// Tree-masked grouped-query attention for bf16 KV caches on the tcgen05 tensor
// cores ("One request, end to end" 2.6: one forward pass verifies the whole
// tree; "Adding a model" step 4: every verified row equals the decode row).
//
// Row function.  Row (node, query head) sees logical positions 0 .. P =
// L+d: the L cache rows, then its ancestors-or-self at L .. L+d.  Its
// positions split at 64R, R = max(floor(P/64) - 1, 0), a function of P alone.
// Below 64R: tiles of 64 positions in splits of plan.split positions, both
// aligned at absolute position 0.  Within a split the tiles run in order
// through one online softmax: S = Q K^T on the tensor core (fp32); the tile's
// 64 slots are handled as two halves of 32 that share the scaled tile max;
// p = 2^(s*c - m) rounded to bf16; each half keeps its own running sum of the
// rounded p; O = O * alpha + P V on the tensor core.  From 64R to P (65 to
// 128 positions once P >= 64: at most two cache tiles and the ancestors):
// the own segment, one softmax in fp32 on the CUDA cores.  The split states
// and the own state are merged in that order.  Every state is carried as
// exact fp32 and each piece runs the same code for the same positions, so
// the result depends only on the row's query and key sequence: a node
// verified in a tree and the same token decoded after its ancestors were
// committed produce the same bits.
//
// Kernels.
//  split kernel (persistent, one CTA per SM): the tiles that every node of a
//    sequence shares (below 64 * (floor((L + d_max)/64) - 1), all cache rows)
//    for up to 128 query rows (node x head of one KV head) at once.  Warps 0
//    and 10 stream K and V tiles with TMA (128B-swizzled boxes) through two
//    rings, prefetching into L2 the tile two ahead (and, before the wait for
//    the previous kernel, the first tiles);
//    warp 1 issues QK^T (Q in TMEM, K in
//    shared memory, S double-buffered in TMEM) and warp 11 issues PV (P in a
//    ring of shared-memory slots, V in shared memory, O in TMEM); warps 2-5
//    and 6-9 run the softmax, one TMEM lane (query row) and one half tile per
//    thread.  An S buffer is reused as soon as the softmax has read it, so
//    QK^T runs ahead of the softmax and the tensor pipe overlaps the narrow
//    QK^T steps with the wide PV steps.  When the largest tree spans two
//    128-row blocks, the two row blocks of a (sequence, KV head, split) run
//    on neighbouring CTAs that stream the same tiles side by side, so the
//    second read of a tile is served by L2; each of the two prefetches half
//    of every tile's boxes into L2.  Each split's state goes to the
//    workspace; the last split of a sequence whose rows start their own
//    segments at two different tiles also leaves its state one tile before
//    its end.
//  tail kernel (one CTA per node and KV head, no tensor memory): the node's
//    own segment for its G query rows, from K/V rows gathered into shared
//    memory with cp.async, computed while the split kernel's last CTAs run;
//    then, after the wait for the split kernel, the in-order merge and the
//    bf16 output (times the front end's sigmoid gate when one is given).
//  Decode runs the same two kernels with a one-node tree per sequence and
//  appends its own K/V row.
#include <cmath>
#include <cstring>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "host.hpp"
#include "launchers.hpp"
#include "ptx.cuh"

namespace tv {

constexpr int kTile = 64;       // KV positions per tile
constexpr int kHalf = 32;       // positions per softmax half
constexpr int kBox = 64 * 128;  // one [64 rows x 128 B] 128B-swizzled box
constexpr int kMaxGroup = 64;   // query heads per KV head on this path
// The K/V producers also prefetch into L2 the boxes of the tile this many
// tiles ahead: a CTA's rings hold at most 5 tiles (160 KiB), fewer bytes
// than HBM needs in flight per SM at ~2 us of loaded latency.  Prefetching
// much further ahead lets the prefetched lines be evicted before their loads.
constexpr int kL2Ahead = 2;

template <int D>
struct Tc {
  static constexpr int KB = D / 64;           // 64-column boxes per row
  static constexpr int TILE = kTile * D * 2;  // bytes of one K or V tile
  // K and V tiles stream through separate rings: a K slot frees as soon as
  // QK^T of its tile completes, a V slot after PV, so K loads run further ahead.
  static constexpr int NK = (D == 256) ? 3 : (D == 128 ? 4 : 6);
  static constexpr int NV = (D == 256) ? 2 : (D == 128 ? 4 : 6);
  // P tiles (bf16, 128 rows x 64 positions, the PV A operand) live in a ring
  // of shared-memory slots, so an S buffer in TMEM is free again as soon as
  // the softmax has read it.
  static constexpr int PTILE = 128 * kTile * 2;
  static constexpr int NP = 3;
  static constexpr int T_O = 0;              // TMEM columns: O [D]
  static constexpr int T_S = D;              //   S [2 x 64]
  static constexpr int T_Q = D + 2 * kTile;  //   Q [D/2] (bf16 pairs)
  static constexpr int COLS = (D + 2 * kTile + D / 2) <= 256 ? 256 : 512;
  static constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, kTile, false, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, false, true);
  static constexpr int RING = (NK + NV) * TILE + NP * PTILE;
  static constexpr int NBAR = 2 * (NK + NV) + 2 * NP + 15;
  static constexpr int SMEM_SPLIT = 1024 + RING + NBAR * 8 + 16;
};

struct TcParams {
  CUtensorMap tmK[TV_MAX_SEQ];
  CUtensorMap tmV[TV_MAX_SEQ];
  __nv_bfloat16* K[TV_MAX_SEQ];
  __nv_bfloat16* V[TV_MAX_SEQ];
  const __nv_bfloat16* q;
  const __nv_bfloat16* kt;
  const __nv_bfloat16* vt;
  __nv_bfloat16* out;
  const __nv_bfloat16* gate;  // output gate of the front end, or null
  const int32_t* len;
  const int32_t* node_off;
  const void* meta;
  int32_t* status;
  float* ws;
  int n_seq, n_total, Hq, Hkv, G, cap, max_len, split_tiles, max_splits, rows_max, decode;
  int ws_splits;    // records per (sequence, KV head, row): the splits, then the snapshot
  int tail_two;     // tail kernel: keys and values staged at once (else keys, then values)
  int tail_staged;  // tail kernel: the split records' weights and sums fit its shared memory
  int tail_a;       // tail kernel: offset of the own-segment buffers (and staged records) in shared memory
  int n_mstage;     // tail kernel: split records staged in shared memory
  int pair;      // split kernel: CTAs 2c, 2c+1 run row blocks 0, 1 of the same (sequence, KV head, split)
  float c;  // scale * log2(e)
};

// ---------------------------------------------------------------------------
// shared pieces of the row function
// ---------------------------------------------------------------------------
// K tile: QK^T operand B, K-major, step kk covers head-dim columns 16kk..16kk+15.
__device__ __forceinline__ uint64_t desc_k(uint32_t ktile, int kk) {
  return sdesc_sw128(ktile + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024);
}
// V tile: PV operand B, MN-major (head dim contiguous), step kk covers
// positions 16kk..16kk+15; the 64-column boxes are kBox apart.
__device__ __forceinline__ uint64_t desc_v(uint32_t vtile, int kk) {
  return sdesc_sw128(vtile + kk * 2048, kBox, 1024);
}

template <int D>
__device__ __forceinline__ void issue_qk(uint32_t tS, uint32_t tQ, uint32_t ktile) {
#pragma unroll
  for (int kk = 0; kk < D / 16; kk++) tc_mma_ts(tS, tQ + kk * 8, desc_k(ktile, kk), Tc<D>::IDESC_QK, kk > 0 ? 1u : 0u);
}
// One K=16 step of QK^T from the tile's step-0 descriptor (the start-address
// field is in 16-byte units; every offset stays inside the field).
template <int D>
__device__ __forceinline__ void issue_qk_step_from(uint32_t tS, uint32_t tQ, uint64_t kd0, int kk) {
  const uint64_t d = kd0 + static_cast<uint64_t>(((kk >> 2) * kBox + (kk & 3) * 32) >> 4);
  tc_mma_ts(tS, tQ + kk * 8, d, Tc<D>::IDESC_QK, kk > 0 ? 1u : 0u);
}
// P tile in shared memory, K-major with the 128-byte swizzle: row r (query
// row) is one 128-byte line of 64 bf16 probabilities; 16-byte chunk c sits at
// chunk position c ^ (r % 8) of its line, lines grouped in 1024-byte atoms.
__device__ __forceinline__ void store_p_half(uint32_t pslot, int row, int hf, const uint32_t (&P)[kHalf / 2]) {
  const uint32_t line = pslot + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
  for (int q = 0; q < 4; q++) {
    const uint32_t c = static_cast<uint32_t>(hf * 4 + q);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(line + ((c ^ (row & 7)) << 4)), "r"(P[4 * q]),
                 "r"(P[4 * q + 1]), "r"(P[4 * q + 2]), "r"(P[4 * q + 3])
                 : "memory");
  }
}
// O (+)= P V with P from a shared-memory slot (step kk: positions 16kk..16kk+15).
template <int D>
__device__ __forceinline__ void issue_pv_ss(uint32_t tO, uint32_t pslot, uint64_t vd0, bool acc) {
#pragma unroll
  for (int kk = 0; kk < kTile / 16; kk++)
    tc_mma_ss(tO, sdesc_sw128(pslot + kk * 32, 16, 1024), vd0 + static_cast<uint64_t>((kk * 2048) >> 4),
              Tc<D>::IDESC_PV, (acc || kk > 0) ? 1u : 0u);
}

// Max of the valid slots of one half tile (exact; any order gives the same).
__device__ __forceinline__ float half_max(const float (&s)[kHalf], int nvalid) {
  float v[kHalf];
#pragma unroll
  for (int j = 0; j < kHalf; j++) v[j] = j < nvalid ? s[j] : -INFINITY;
#pragma unroll
  for (int w = kHalf / 2; w >= 1; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; j++) v[j] = fmaxf(v[j], v[j + w]);
  return v[0];
}

// Probabilities of one half tile as packed bf16 pairs and the sum of the
// rounded values (fixed order).  m_new: the running max in the exp2 domain.
__device__ __forceinline__ float half_probs(const float (&s)[kHalf], int nvalid, float c, float m_new,
                                            uint32_t (&P)[kHalf / 2]) {
  const float neg = -m_new;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < kHalf; j += 2) {
    const float p0 = j < nvalid ? ex2_approx(__fmaf_rn(s[j], c, neg)) : 0.f;
    const float p1 = j + 1 < nvalid ? ex2_approx(__fmaf_rn(s[j + 1], c, neg)) : 0.f;
    const uint32_t w = pack_bf16x2(p0, p1);
    P[j / 2] = w;
    acc[(j / 2) & 3] = __fadd_rn(acc[(j / 2) & 3], __fadd_rn(bf16_lo(w), bf16_hi(w)));
  }
  return __fadd_rn(__fadd_rn(acc[0], acc[1]), __fadd_rn(acc[2], acc[3]));
}

// Reference max for the exponentials.  It moves only when the tile's scaled
// max exceeds it by more than kRescale (in log2 units), so most tiles keep it
// and skip rescaling O; probabilities then stay below 2^kRescale, well inside
// bf16 and fp32 range.  alpha is the factor for the running O and sums:
// exactly 1 when the reference is kept, 0 on the first tile.
constexpr float kRescale = 8.f;
__device__ __forceinline__ float next_max(float m, float mx_raw, float c, float& alpha) {
  const float mt = __fmul_rn(mx_raw, c);
  if (mt > __fadd_rn(m, kRescale) || m == -INFINITY) {
    alpha = ex2_approx(__fsub_rn(m, mt));
    return mt;
  }
  alpha = 1.f;
  return m;
}

__device__ __forceinline__ void tmem_ld32f(uint32_t taddr, float (&s)[kHalf]) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
#pragma unroll
  for (int i = 0; i < 32; i++) s[i] = __uint_as_float(r[i]);
}

// O columns [c0, c1) of this thread's lane times alpha.
__device__ __forceinline__ void rescale_o(uint32_t tO, int c0, int c1, float alpha) {
#pragma unroll 1
  for (int c = c0; c < c1; c += 32) {
    uint32_t r[32];
    tmem_ld32(tO + c, r);
#pragma unroll
    for (int i = 0; i < 32; i++) r[i] = __float_as_uint(__fmul_rn(__uint_as_float(r[i]), alpha));
    tmem_st32(tO + c, r);
  }
}

// Workspace record of (sequence, KV head, split, row).
// Record slot past the splits: the state of a sequence's last split one
// tile before its end.
__device__ __forceinline__ int snap_slot(const TcParams& p) { return p.max_splits; }
__device__ __forceinline__ float* ws_rec(const TcParams& p, int s, int g, int split, int row, int D) {
  return p.ws + ((((static_cast<size_t>(s) * p.Hkv + g) * p.ws_splits + split) * p.rows_max + row) *
                 static_cast<size_t>(D + 4));
}

// This half's O columns (TMEM) to the record; half 0 also writes m and l_A,
// half 1 writes l_B.
template <int D>
__device__ __forceinline__ void store_state(uint32_t tO, float* rec, int hf, float m, float lh) {
#pragma unroll 1
  for (int c0 = hf * (D / 2); c0 < (hf + 1) * (D / 2); c0 += 32) {
    uint32_t r[32];
    tmem_ld32(tO + c0, r);
    if (rec) {
      float4* d4 = reinterpret_cast<float4*>(rec + c0);
#pragma unroll
      for (int i = 0; i < 8; i++)
        d4[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]), __uint_as_float(r[4 * i + 2]),
                            __uint_as_float(r[4 * i + 3]));
    }
  }
  if (rec) {
    if (hf == 0) {
      rec[D] = m;
      rec[D + 1] = lh;
    } else {
      rec[D + 2] = lh;
    }
  }
}

// Queries of one row into TMEM (bf16 pairs, columns T_Q ..).  For D >= 128
// each half-tile thread moves its half of the row (D/4 columns from hf*D/4);
// for D = 64 the half-0 thread moves the whole row (32 columns).
template <int D>
struct QShare {
  static constexpr int N = D >= 128 ? D / 16 : D / 8;  // 16-byte pieces per thread
  static constexpr int COL0 = D >= 128 ? D / 4 : 0;    // first column of half 1
};
template <int D>
__device__ __forceinline__ void q_fetch(const __nv_bfloat16* qrow, int hf, uint4 (&qv)[QShare<D>::N]) {
  const bool act = qrow != nullptr && (D >= 128 || hf == 0);
  const uint4* q4 = act ? reinterpret_cast<const uint4*>(qrow) + hf * QShare<D>::N : nullptr;
#pragma unroll
  for (int i = 0; i < QShare<D>::N; i++) qv[i] = act ? q4[i] : make_uint4(0u, 0u, 0u, 0u);
}
template <int D>
__device__ __forceinline__ void q_store(uint32_t tq, int hf, const uint4 (&qv)[QShare<D>::N]) {
  if (D < 128 && hf != 0) return;
#pragma unroll
  for (int j = 0; j < QShare<D>::N / 8; j++) {
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 8; i++) {
      r[4 * i] = qv[8 * j + i].x;
      r[4 * i + 1] = qv[8 * j + i].y;
      r[4 * i + 2] = qv[8 * j + i].z;
      r[4 * i + 3] = qv[8 * j + i].w;
    }
    tmem_st32(tq + hf * QShare<D>::COL0 + 32 * j, r);
  }
}

// The split state of a warp's 32 rows (this half's O columns, then m and the
// half sums) to the workspace.  A thread holds one row after tcgen05.ld; the
// warp turns each 32-column block around through 4 KB of shared memory (rows
// of 128 bytes, 16-byte units at unit ^ (row % 8)) so that one store
// instruction writes 128 contiguous bytes of each of four rows instead of 16
// bytes of each of 32.  rec(r) is the record of warp row r or null.
template <int D, typename Rec>
__device__ __forceinline__ void store_state_warp(uint32_t tO, uint32_t xbuf, int hf, int lane, float m, float lh,
                                                 Rec rec) {
#pragma unroll 1
  for (int c0 = hf * (D / 2); c0 < (hf + 1) * (D / 2); c0 += 32) {
    uint32_t r[32];
    tmem_ld32(tO + c0, r);
#pragma unroll
    for (int u = 0; u < 8; u++)
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(xbuf + lane * 128 + ((u ^ (lane & 7)) << 4)),
                   "r"(r[4 * u]), "r"(r[4 * u + 1]), "r"(r[4 * u + 2]), "r"(r[4 * u + 3])
                   : "memory");
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const int rr = 4 * i + (lane >> 3), u = lane & 7;
      float4 v;
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                   : "r"(xbuf + rr * 128 + ((u ^ (rr & 7)) << 4))
                   : "memory");
      float* d = rec(rr);
      if (d) *reinterpret_cast<float4*>(d + c0 + 4 * u) = v;
    }
    __syncwarp();
  }
  float* own = rec(lane);
  if (own) {
    if (hf == 0) {
      own[D] = m;
      own[D + 1] = lh;
    } else {
      own[D + 2] = lh;
    }
  }
}

// ---------------------------------------------------------------------------
// rows and their segments
// ---------------------------------------------------------------------------
// First tile of the own segment of a row whose last position is P.  It
// depends on P alone, so a verified row and the decode row of the same token
// cut their positions in the same place; one tile back from P's tile, so
// that for every node of a tree (depth below 64) the tiles before it are
// cache tiles below floor(L/64), which the whole tree shares.
__device__ __forceinline__ int own_tile(int P) { return max((P >> 6) - 1, 0); }
// Tiles of a sequence that the split kernel runs: those below the own
// segment of its deepest possible row (depth below the tree's size and
// TV_MAX_PATH).  Every row of the sequence starts its own segment at this
// tile or one before it.
__device__ __forceinline__ int split_end(int L, int nodes, int decode) {
  const int dub = decode ? 0 : min(max(nodes - 1, 0), TV_MAX_PATH - 1);
  return own_tile(L + dub);
}

// The sequence, first node, context length, tree size and depth of a node
// (verify) or of a sequence's one row (decode).
struct RowInfo {
  int s, off, L, nodes, depth;
};
__device__ inline RowInfo row_info(const TcParams& p, int node_g) {
  RowInfo ri;
  if (p.decode) {
    ri.s = node_g;
    ri.off = node_g;
    ri.L = p.len[node_g];
    ri.nodes = 1;
    ri.depth = 0;
    return ri;
  }
  // every global load issued before any result is used
  int ends[TV_MAX_SEQ], lens[TV_MAX_SEQ];
#pragma unroll
  for (int i = 0; i < TV_MAX_SEQ; i++) {
    ends[i] = i < p.n_seq ? p.node_off[i + 1] : 0;
    lens[i] = i < p.n_seq ? p.len[i] : 0;
  }
  const int off0 = p.node_off[0];
  const MetaView mv = meta_view(const_cast<void*>(p.meta), p.n_total);
  const int depth = mv.depth[node_g];
  ri.depth = depth < 0 ? 0 : (depth >= TV_MAX_PATH ? TV_MAX_PATH - 1 : depth);
  ri.s = 0;
  ri.off = off0;
  ri.L = lens[0];
  int end = ends[0];
#pragma unroll
  for (int i = 0; i + 1 < TV_MAX_SEQ; i++) {
    if (i + 1 < p.n_seq && node_g >= ends[i]) {
      ri.s = i + 1;
      ri.off = ends[i];
      ri.L = lens[i + 1];
      end = ends[i + 1];
    }
  }
  ri.nodes = end - ri.off;
  return ri;
}
// A row unit the own-segment and merge kernels can run: a length within the
// host bound (and, for decode, a free cache row) and a node whose rows lie
// inside the workspace (a malformed tree is reported by tv_tree_prepare).
__device__ __forceinline__ bool row_ok(const TcParams& p, const RowInfo& ri, int local) {
  return ri.L >= 0 && ri.L <= p.max_len && !(p.decode && ri.L >= p.cap) && local >= 0 &&
         (local + 1) * p.G <= p.rows_max;
}

// ---------------------------------------------------------------------------
// split kernel
// ---------------------------------------------------------------------------
struct ItemSpace {
  int cum[TV_MAX_SEQ + 1];
  int tend[TV_MAX_SEQ];  // tiles of each sequence run here
  int snap[TV_MAX_SEQ];  // some row starts its own segment at tend - 1: the last split keeps a snapshot
  int nrb[TV_MAX_SEQ];   // 128-row blocks
  int rows[TV_MAX_SEQ];  // query rows = nodes * G
  int off[TV_MAX_SEQ];   // first node
};
struct Item {
  int s, g, rb, split, t0, t1;
};

__device__ inline void item_space(const TcParams& p, ItemSpace& is) {
  is.cum[0] = 0;
  for (int s = 0; s < p.n_seq; s++) {
    int L = p.len[s];
    if (L < 0 || L > p.max_len) L = 0;  // reported by the tail kernel
    // offsets and counts clamped to the node buffers: a malformed tree is
    // reported by tv_tree_prepare, and the query rows of the first item are
    // read before the status word is
    int off = p.decode ? s : p.node_off[s];
    off = off < 0 ? 0 : (off > p.n_total ? p.n_total : off);
    int nodes = p.decode ? 1 : p.node_off[s + 1] - off;
    nodes = nodes < 0 ? 0 : (nodes > TV_MAX_NODES ? TV_MAX_NODES : nodes);
    if (off + nodes > p.n_total) nodes = p.n_total - off;
    is.off[s] = off;
    is.rows[s] = nodes * p.G;
    is.nrb[s] = p.pair ? 1 : (is.rows[s] + 127) / 128;  // a pair covers row blocks 0 and 1
    is.tend[s] = split_end(L, nodes, p.decode);
    is.snap[s] = is.tend[s] > own_tile(L) ? 1 : 0;  // the root's row starts one tile earlier
    const int nsplit = (is.tend[s] + p.split_tiles - 1) / p.split_tiles;
    is.cum[s + 1] = is.cum[s] + nsplit * p.Hkv * is.nrb[s];
  }
}

__device__ inline Item item_at(const ItemSpace& is, const TcParams& p, int w, int rank) {
  int s = 0;
  while (s < p.n_seq - 1 && w >= is.cum[s + 1]) s++;
  int r = w - is.cum[s];
  Item it;
  it.s = s;
  it.rb = p.pair ? rank : r % is.nrb[s];
  r /= is.nrb[s];
  it.g = r % p.Hkv;
  it.split = r / p.Hkv;
  it.t0 = it.split * p.split_tiles;
  it.t1 = min(it.t0 + p.split_tiles, is.tend[s]);
  return it;
}

template <int D>
__global__ void __launch_bounds__(384, 1) attn_split_kernel(const __grid_constant__ TcParams p) {
  using C = Tc<D>;
  static_assert(C::NP * C::PTILE >= 8 * 4096, "the state store turns rows around in the P ring");
  extern __shared__ uint8_t smem_raw[];
  __shared__ ItemSpace is;
  __shared__ int skip;
  __shared__ float xmax[2][2][128];  // [tile parity][half][row]: half-tile maxima
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (sb - raw);
  const uint32_t bars = sb + C::RING;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + C::RING + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // ring barriers: KFULL[NK], KEMPTY[NK], VFULL[NV], VEMPTY[NV]
  const uint32_t KFULL0 = bars, KEMPTY0 = bars + 8u * C::NK;
  const uint32_t VFULL0 = bars + 16u * C::NK, VEMPTY0 = VFULL0 + 8u * C::NV;
  const int nb = 2 * (C::NK + C::NV);
  // S buffers (by tile parity): SFULL when QK^T has written S, SFREE when the
  // softmax has read it.  P slots (tile % NP): PFULL when the softmax has
  // written P, ODONE when PV has consumed it (and O holds that tile).
  const uint32_t SFULL0 = bars + 8u * nb, SFREE0 = SFULL0 + 16u;
  const uint32_t PFULL0 = SFREE0 + 16u, ODONE0 = PFULL0 + 8u * C::NP;
  const uint32_t QREADY = ODONE0 + 8u * C::NP;
  const uint32_t DRAIN = QREADY + 8u;  // [2] one per MMA warp
  const uint32_t XBAR0 = DRAIN + 16u;  // [2][4] half-max exchange, by tile parity and row quarter
  const uint32_t kring = sb, vring = sb + C::NK * C::TILE, pring = vring + C::NV * C::TILE;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Pair mode: CTAs 2c and 2c+1 run row blocks 0 and 1 of the same items,
  // loading the same tiles at nearly the same time, so one of the two reads
  // of a tile comes from L2.  Each prefetches only its half of the boxes.
  const bool pair = p.pair != 0;
  const int rank = pair ? static_cast<int>(blockIdx.x & 1u) : 0;
  const int cid = pair ? static_cast<int>(blockIdx.x) / 2 : static_cast<int>(blockIdx.x);
  const int ncl = pair ? static_cast<int>(gridDim.x) / 2 : static_cast<int>(gridDim.x);
  const int kb0 = pair ? rank * (C::KB / 2) : 0, kb1 = pair ? kb0 + C::KB / 2 : C::KB;  // L2 prefetch share

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NK; i++) {
      mbar_init(KFULL0 + 8u * i, 1);
      mbar_init(KEMPTY0 + 8u * i, 1);
    }
    for (int i = 0; i < C::NV; i++) {
      mbar_init(VFULL0 + 8u * i, 1);
      mbar_init(VEMPTY0 + 8u * i, 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(SFULL0 + 8u * b, 1);
      mbar_init(SFREE0 + 8u * b, 256);
      for (int q = 0; q < 4; q++) mbar_init(XBAR0 + 8u * (b * 4 + q), 64);  // the two warps of a row quarter
    }
    for (int i = 0; i < C::NP; i++) {
      mbar_init(PFULL0 + 8u * i, 256);
      mbar_init(ODONE0 + 8u * i, 1);
    }
    mbar_init(QREADY, 256);
    mbar_init(DRAIN, 1);
    mbar_init(DRAIN + 8u, 1);
    *abort_flag = 0;
    fence_mbar_init();
    item_space(p, is);  // lengths and node offsets: not written by the previous kernel of a round
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const int total = is.cum[p.n_seq];
  // L2 prefetch of the first item's first tiles and query rows while the
  // previous kernel finishes: a prefetch only warms L2 (the point of
  // coherence), so it is safe whatever the previous kernel writes, and the
  // ring's first loads and the first queries then hit L2.
  if ((warp == 0 || warp == 10) && lane == 0 && cid < total) {
    const Item I = item_at(is, p, cid, rank);
    const CUtensorMap* maps = warp == 0 ? p.tmK : p.tmV;
    const int nfirst = min(I.t1 - I.t0, (warp == 0 ? C::NK : C::NV) + kL2Ahead);
    for (int t = I.t0; t < I.t0 + nfirst; t++)
      for (int kb = kb0; kb < kb1; kb++) tma_prefetch_l2_2d(&maps[I.s], kb * 64, I.g * p.cap + t * kTile);
  }
  if (warp >= 2 && warp <= 9 && cid < total) {
    const Item I = item_at(is, p, cid, rank);
    const int row = I.rb * 128 + (warp & 3) * 32 + lane, hq = (warp - 2) >> 2;
    if (row < is.rows[I.s]) {
      const char* qr = reinterpret_cast<const char*>(
          p.q + (static_cast<size_t>(is.off[I.s] + row / p.G) * p.Hq + I.g * p.G + row % p.G) * D);
      for (int b = hq * (D * 2 / 2); b < (hq + 1) * (D * 2 / 2); b += 128) prefetch_l2(qr + b);
    }
  }
  pdl_wait();  // queries, status and the workspace (read by the previous tail) from here on
  pdl_trigger();
  if (threadIdx.x == 0) skip = status_bad(p.status) ? 1 : 0;
  // softmax threads: the first item's query row, in flight during the status read
  uint4 qv[QShare<D>::N];
  const bool softmax_warp = warp >= 2 && warp <= 9;
  const int hf = (warp - 2) >> 2;  // softmax half: 0: slots 0-31, 1: slots 32-63
  const int quad = warp & 3;
  const int lrow = quad * 32 + lane;
  auto q_row = [&](const Item& I) -> const __nv_bfloat16* {
    const int row = I.rb * 128 + lrow;
    if (row >= is.rows[I.s]) return nullptr;
    const int node = row / p.G, jh = row % p.G;
    return p.q + (static_cast<size_t>(is.off[I.s] + node) * p.Hq + I.g * p.G + jh) * D;
  };
  if (softmax_warp && cid < total) q_fetch<D>(q_row(item_at(is, p, cid, rank)), hf, qv);
  __syncthreads();

  if (!skip && (warp == 0 || warp == 10) && lane == 0) {
    // ---------------- TMA producers: warp 0 streams K tiles, warp 10 V tiles ----------------
    const bool is_k = warp == 0;
    const int nslot = is_k ? C::NK : C::NV;
    const uint32_t full0 = is_k ? KFULL0 : VFULL0, empty0 = is_k ? KEMPTY0 : VEMPTY0;
    const uint32_t ring = is_k ? kring : vring;
    const CUtensorMap* maps = is_k ? p.tmK : p.tmV;
    uint32_t it = 0;
    bool ok = true;
    for (int w = cid; w < total && ok; w += ncl) {
      const Item I = item_at(is, p, w, rank);
      const int ybase = I.g * p.cap;
      for (int t = I.t0; t < I.t1; t++) {
        const int st = it % nslot;
        if (!wait_role(empty0 + 8u * st, ((it / nslot) & 1) ^ 1, abort_flag, kWaitCycles)) {
          ok = false;
          break;
        }
        const uint32_t full = full0 + 8u * st;
        mbar_arrive_expect_tx(full, C::TILE);
        const uint32_t dst = ring + st * C::TILE;
        const int y = ybase + t * kTile;
        if (t + kL2Ahead < I.t1)
          for (int kb = kb0; kb < kb1; kb++) tma_prefetch_l2_2d(&maps[I.s], kb * 64, y + kL2Ahead * kTile);
#pragma unroll
        for (int kb = 0; kb < C::KB; kb++) tma_load_2d(dst + kb * kBox, &maps[I.s], full, kb * 64, y);
        it++;
      }
    }
    if (!ok) {
      set_status(p.status, TV_ERR_TIMEOUT);
      // let every issued copy land before the CTA's shared memory is released
      for (uint32_t i = it > (uint32_t)nslot ? it - nslot : 0; i < it; i++)
        mbar_wait(full0 + 8u * (i % nslot), (i / nslot) & 1, kWaitCycles);
    }
  } else if (!skip && (warp == 1 || warp == 11)) {
    // ---------------- MMA issuers, one warp each, whole-warp loops with one
    // elected lane issuing.  Warp 1 issues QK^T(t) as soon as K(t) has landed
    // and the softmax has read S(t-2) out of the same TMEM buffer; warp 11
    // issues PV(t) as soon as P(t) and V(t) are in shared memory.  The two
    // streams touch disjoint TMEM columns, and the tensor pipe overlaps the
    // narrow QK^T steps with the wide PV steps. ----------------
    const bool is_qk = warp == 1;
    uint32_t t = 0, q_ph = 0;  // CTA-wide tile counter
    bool ok = true;
    for (int w = cid; w < total && ok; w += ncl) {
      const Item I = item_at(is, p, w, rank);
      const int n = I.t1 - I.t0;
      if (is_qk) {
        if (!wait_warp(QREADY, q_ph, abort_flag, kWaitCycles)) {
          ok = false;
          break;
        }
        q_ph ^= 1;
      }
      for (int k = 0; k < n; k++, t++) {
        if (is_qk) {
          const int ks = t % C::NK, b = t & 1;
          if (!wait_warp(KFULL0 + 8u * ks, (t / C::NK) & 1, abort_flag, kWaitCycles) ||
              (t >= 2 && !wait_warp(SFREE0 + 8u * b, ((t - 2) >> 1) & 1, abort_flag, kWaitCycles))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tS = tbase + C::T_S + b * kTile, tQ = tbase + C::T_Q;
          const uint64_t kd = desc_k(kring + ks * C::TILE, 0);
          if (elect_one_sync()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++) issue_qk_step_from<D>(tS, tQ, kd, kk);
            tc_commit(SFULL0 + 8u * b);
            tc_commit(KEMPTY0 + 8u * ks);
          }
          __syncwarp();
        } else {
          const int ps = t % C::NP, vs = t % C::NV;
          if (!wait_warp(PFULL0 + 8u * ps, (t / C::NP) & 1, abort_flag, kWaitCycles) ||
              !wait_warp(VFULL0 + 8u * vs, (t / C::NV) & 1, abort_flag, kWaitCycles)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one_sync()) {
            issue_pv_ss<D>(tbase + C::T_O, pring + ps * C::PTILE, desc_v(vring + vs * C::TILE, 0), k > 0);
            tc_commit(VEMPTY0 + 8u * vs);
            tc_commit(ODONE0 + 8u * ps);
          }
          __syncwarp();
        }
      }
    }
    // every MMA issued by this warp completes before TMEM is released
    const uint32_t drain = DRAIN + (is_qk ? 0u : 8u);
    if (elect_one_sync()) tc_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, kWaitCycles);
    if (!ok && lane == 0) set_status(p.status, TV_ERR_TIMEOUT);
  } else if (!skip && warp >= 2 && warp <= 9) {
    // ---------------- softmax / epilogue: warps 2-9, two warpgroups, one half tile each ----------------
    // Their waits are warp-wide (every lane gets the same outcome), so a wait
    // that gives up takes the whole warp out of the loop and no tcgen05.ld or
    // .st below ever runs with part of a warp.
    const uint32_t tl = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    uint32_t t = 0;  // CTA-wide tile counter
    bool ok = true;
    for (int w = cid; w < total && ok; w += ncl) {
      const Item I = item_at(is, p, w, rank);
      const int n = I.t1 - I.t0;
      const int rbase = I.rb * 128 + quad * 32, nrows = is.rows[I.s];
      const bool snap_item = is.snap[I.s] && I.t1 == is.tend[I.s] && n >= 2;
      // this thread's Q share (bf16 pairs) into TMEM; every QK^T of the
      // previous item has completed (its S was read)
      if (w != cid) q_fetch<D>(q_row(I), hf, qv);
      q_store<D>(tl + C::T_Q, hf, qv);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(QREADY);
      float m = -INFINITY, lh = 0.f;
      for (int k = 0; k < n; k++) {
        const int b = t & 1;
        if (!wait_warp(SFULL0 + 8u * b, (t >> 1) & 1, abort_flag, kWaitCycles)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[kHalf];
        tmem_ld32f(tl + C::T_S + b * kTile + hf * kHalf, sv);
        tc_fence_before();
        mbar_arrive(SFREE0 + 8u * b);  // S(t) is in registers: QK^T(t+2) may overwrite the buffer
        if (snap_item && k == n - 1) {
          // The state one tile before the split's end, for the rows whose own
          // segment starts at this tile: O once PV of the previous tile is
          // complete, with m and the sums before this tile.  Every PV so far
          // is then complete, so the two P slots other than this tile's are
          // free (the next item's P waits for every softmax warp's queries):
          // warp (half, quarter) turns its rows around in 4 KB of them.
          const uint32_t tp = t - 1;
          if (!wait_warp(ODONE0 + 8u * (tp % C::NP), (tp / C::NP) & 1, abort_flag, kWaitCycles)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t xbuf = pring + ((t + 1 + hf) % C::NP) * C::PTILE + static_cast<uint32_t>(quad) * 4096u;
          store_state_warp<D>(tl + C::T_O, xbuf, hf, lane, m, lh,
                              [&](int r) -> float* {
                                return rbase + r < nrows ? ws_rec(p, I.s, I.g, snap_slot(p), rbase + r, D) : nullptr;
                              });
        }
        const float mh = half_max(sv, kHalf);
        xmax[b][hf][lrow] = mh;
        mbar_arrive(XBAR0 + 8u * (b * 4 + quad));
        if (!wait_warp(XBAR0 + 8u * (b * 4 + quad), (t >> 1) & 1, abort_flag, kWaitCycles)) {
          ok = false;
          break;
        }
        const float mo = xmax[b][hf ^ 1][lrow];
        float alpha;
        const float m_new = next_max(m, fmaxf(mh, mo), p.c, alpha);
        uint32_t P[kHalf / 2];
        const float rs = half_probs(sv, kHalf, p.c, m_new, P);
        lh = __fmaf_rn(lh, alpha, rs);
        m = m_new;
        const int ps = t % C::NP;
        if (t >= static_cast<uint32_t>(C::NP) &&
            !wait_warp(ODONE0 + 8u * ps, ((t - C::NP) / C::NP) & 1, abort_flag, kWaitCycles)) {  // slot's previous PV done
          ok = false;
          break;
        }
        store_p_half(pring + ps * C::PTILE, lrow, hf, P);
        if (k > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          const uint32_t tp = t - 1;  // PV of the previous tile must be complete
          if (!wait_warp(ODONE0 + 8u * (tp % C::NP), (tp / C::NP) & 1, abort_flag, kWaitCycles)) {
            ok = false;
            break;
          }
          tc_fence_after();
          rescale_o(tl + C::T_O, hf * (D / 2), (hf + 1) * (D / 2), alpha);
          tmem_st_wait();
        }
        fence_proxy_async_smem();  // P visible to the tensor core
        tc_fence_before();
        mbar_arrive(PFULL0 + 8u * ps);
        t++;
      }
      if (!ok) break;
      {
        const uint32_t tp = t - 1;  // the item's last PV
        if (!wait_warp(ODONE0 + 8u * (tp % C::NP), (tp / C::NP) & 1, abort_flag, kWaitCycles)) {
          ok = false;
          break;
        }
      }
      tc_fence_after();
      // the next item's first PV needs P of its first tile, which this
      // warpgroup writes only after this read of O.  Every PV of the item is
      // complete, so the P ring is free: warp k of the softmax turns its rows
      // around in the ring's k-th 4 KB.
      store_state_warp<D>(tl + C::T_O, pring + static_cast<uint32_t>(warp - 2) * 4096u, hf, lane, m, lh,
                          [&](int r) -> float* {
                            return rbase + r < nrows ? ws_rec(p, I.s, I.g, I.split, rbase + r, D) : nullptr;
                          });
    }
    if (!ok) set_status(p.status, TV_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, C::COLS);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// tail kernel: the row's own segment, then the merge
// ---------------------------------------------------------------------------
// Warp-level bf16 tensor-core tiles (m16n8k16, fp32 accumulate) for the own
// segment's two small products: its rows are one node's G query heads, far
// below the 64- or 128-row tiles of tcgen05, and these need no tensor memory,
// so several tail CTAs share an SM.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// d += a b for one 16 x 8 x 16 tile (a: 16 x 16 row-major, b: 16 x 8 column-major)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
               "{%0, %1, %2, %3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Byte offset of 16-byte chunk c of row r in a buffer of rows rb bytes long:
// chunk c sits at c ^ (r mod 8), so the 8 rows of an 8 x 8 matrix load fall
// on distinct banks.
__device__ __forceinline__ uint32_t swz(int r, int c, int rb) {
  return static_cast<uint32_t>(r * rb + ((c ^ (r & 7)) << 4));
}

template <int D>
struct Tail {
  static constexpr int NT = 512;          // threads
  static constexpr int NW = NT / 32;      // warps
  static constexpr int CH = D / 8;        // 16-byte chunks of a K/V/Q row
  static constexpr int NPOS = 2 * kTile;  // positions of an own segment, at most
  static constexpr int KV = NPOS * D * 2; // bytes of its keys (or values)
  static constexpr int PRB = NPOS * 2;    // bytes of a probability row
  static constexpr int MB = 8;            // unstaged split records in flight per merge thread
  static constexpr int REC = (D + 4) * 4; // bytes of one record row: O[D], m, l_A, l_B, pad
  // Shared memory: the own segment's O [G][D] fp32 and (when staged) the
  // merge's weights and sums come first; from offset tail_a the own
  // segment's buffers: keys [NPOS][D] bf16, values (their own buffer, or the
  // keys' after the scores), queries [16 MT][D] bf16, probabilities
  // [16 MT][NPOS] bf16 (MT = ceil(G/16) row tiles; K/V/Q/P rows
  // chunk-swizzled) and scores [G][NPOS] fp32.  Once the own segment is
  // done, the split records are staged from tail_a on, as many as fit.
  __host__ __device__ static constexpr int q_off(bool two) { return (two ? 2 : 1) * KV; }
  __host__ __device__ static constexpr int p_off(int G, bool two) { return q_off(two) + ((G + 15) / 16) * 16 * D * 2; }
  __host__ __device__ static constexpr int sc_off(int G, bool two) { return p_off(G, two) + ((G + 15) / 16) * 16 * PRB; }
  __host__ __device__ static constexpr int own_bytes(int G, bool two) { return sc_off(G, two) + G * NPOS * 4; }
  __host__ __device__ static constexpr int wbytes(int G, int max_splits) { return (2 * max_splits + 2) * G * 4; }
  __host__ __device__ static constexpr int a_off(int G, int wb) { return (G * D * 4 + wb + 1023) & ~1023; }
};

// One CTA per (node, KV head), or (sequence, KV head) for decode; the split
// kernel of the same call runs before it.
//  Own segment, before the wait for the split kernel (which writes none of
//  what it reads): the segment's K/V rows (cache rows below L, then the
//  node's ancestors-or-self at L .. L+d; zeros up to a multiple of 16) and
//  the node's G query rows come into shared memory with cp.async; with two
//  buffers the values load while the scores are computed, with one they
//  follow the keys into the same buffer.  S = Q K^T by 16 x 8 x 16 tensor-core
//  tiles, each output accumulated over the head dimension in order; m = the
//  segment's scaled maximum; p = 2^(s*c - m) rounded to bf16; l = the sum of
//  the rounded p over a warp's fixed lanes; O = P V by the same tiles,
//  accumulated over the positions in order.  Verify and decode place a
//  row's positions and heads in the same tile slots, so both run the same
//  arithmetic.
//  Merge, after the wait: the split records of the node's G rows (each
//  record's rows are contiguous) come into shared memory by bulk copies, as
//  many as fit, while the weights are formed from their m and l read
//  directly.  A row takes its split states, then its own state.  The last
//  split is the one the split kernel finished unless that split ran one
//  tile past the row's own segment start, in which case it is the snapshot
//  taken one tile before its end.  Weights 2^(m_i - max m), O = sum w_i O_i
//  and l = sum w_i (l_A + l_B) in record order; the output is O / l (times
//  the front end's sigmoid gate when one is given).  Decode then appends the
//  token's K/V at row L.
template <int D>
__global__ void __launch_bounds__(512, 2) attn_tail_kernel(const __grid_constant__ TcParams p) {
  using T = Tail<D>;
  extern __shared__ __align__(16) uint8_t tsm[];
  __shared__ int anc_s[TV_MAX_PATH];  // global node of the ancestor at each depth
  __shared__ int skip;
  __shared__ float mown[kMaxGroup], lown[kMaxGroup];
  __shared__ __align__(8) uint64_t mbar;  // staged split records
  const int G = p.G, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = static_cast<int>(blockIdx.x) % p.Hkv, node_g = static_cast<int>(blockIdx.x) / p.Hkv;
  const bool two = p.tail_two != 0;
  const int MT = (G + 15) / 16;
  const uint32_t MBAR = smem_u32(&mbar);
  if (tid == 0) {
    mbar_init(MBAR, 1);
    fence_mbar_init();
  }
  // Lengths, tree tables, queries, caches and the tree's K/V rows: none is
  // written by the split kernel before this one, and the split kernel lets
  // this kernel in only after its own wait, so all are complete.
  const RowInfo ri = row_info(p, node_g);
  const int local = node_g - ri.off;
  const bool rok = row_ok(p, ri, local);
  if (tid < TV_MAX_PATH) {
    int an = node_g;
    if (!p.decode) {
      const MetaView mv = meta_view(const_cast<void*>(p.meta), p.n_total);
      const int a = mv.anc_at[static_cast<size_t>(node_g) * TV_MAX_PATH + tid];
      an = tid > ri.depth ? node_g : ri.off + a;
    }
    // clamped to the node buffers: with a malformed tree (reported by
    // tv_tree_prepare) the tables may be stale
    anc_s[tid] = an < 0 ? 0 : (an >= p.n_total ? p.n_total - 1 : an);
  }
  __syncthreads();
  const int P = ri.L + ri.depth;
  const int tend = split_end(ri.L, ri.nodes, p.decode);
  const int R = min(own_tile(P), tend);
  const int p0 = R * kTile, n = min(P - p0 + 1, T::NPOS);
  const int n16 = (n + 15) & ~15;  // positions the tiles cover
  float* const oown = reinterpret_cast<float*>(tsm);  // [G][D]
  uint8_t* const ob = tsm + p.tail_a;                 // own-segment buffers, then staged records
  float* const sc = reinterpret_cast<float*>(ob + T::sc_off(G, two));  // [G][NPOS]
  if (rok) {
    const uint32_t kb = smem_u32(ob), vb = two ? kb + T::KV : kb;
    const uint32_t qb = kb + T::q_off(two), pb = kb + T::p_off(G, two);
    auto stage = [&](uint32_t dst, bool values) {
      const __nv_bfloat16* cache = values ? p.V[ri.s] : p.K[ri.s];
      const __nv_bfloat16* tree = values ? p.vt : p.kt;
      for (int idx = tid; idx < n16 * T::CH; idx += T::NT) {
        const int j = idx / T::CH, cc = idx % T::CH, pos = p0 + j;
        const __nv_bfloat16* src =
            j >= n ? tree
                   : (pos < ri.L ? cache + (static_cast<size_t>(g) * p.cap + pos) * D + cc * 8
                                 : tree + (static_cast<size_t>(anc_s[pos - ri.L]) * p.Hkv + g) * D + cc * 8);
        cp_async16(dst + swz(j, cc, D * 2), src, j < n);  // zeros past the segment
      }
    };
    stage(kb, false);
    {
      const __nv_bfloat16* qsrc = p.q + (static_cast<size_t>(node_g) * p.Hq + g * G) * D;
      for (int idx = tid; idx < MT * 16 * T::CH; idx += T::NT) {
        const int r = idx / T::CH, cc = idx % T::CH;
        cp_async16(qb + swz(r, cc, D * 2), r < G ? qsrc + r * D + cc * 8 : qsrc, r < G);
      }
    }
    cp_async_commit();
    if (two) stage(vb, true);
    cp_async_commit();
    // probability rows past the group stay zero
    for (int idx = tid; idx < (MT * 16 - G) * (T::PRB / 16); idx += T::NT) {
      const int r = G + idx / (T::PRB / 16), cc = idx % (T::PRB / 16);
      *reinterpret_cast<uint4*>(ob + T::p_off(G, two) + swz(r, cc, T::PRB)) = make_uint4(0u, 0u, 0u, 0u);
    }
    cp_async_wait_group<1>();  // keys and queries
    __syncthreads();
    // S = Q K^T: warp items (row tile, 8-position tile); two k-steps per pass
    {
      const int nt8 = (n + 7) >> 3, mi = lane >> 3, rr = lane & 7;
      for (int it = warp; it < MT * nt8; it += T::NW) {
        const int mt = it / nt8, nt = it % nt8;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const int qrow = mt * 16 + (mi & 1) * 8 + rr, krow = nt * 8 + rr;
#pragma unroll 4
        for (int ks = 0; ks < D / 16; ks += 2) {
          uint32_t a0[4], a1[4], b[4];
          ldsm_x4(qb + swz(qrow, 2 * ks + (mi >> 1), D * 2), a0);
          ldsm_x4(qb + swz(qrow, 2 * ks + 2 + (mi >> 1), D * 2), a1);
          ldsm_x4(kb + swz(krow, 2 * ks + mi, D * 2), b);  // chunks 2ks .. 2ks + 3 of the 8 key rows
          mma16816(acc, a0, b[0], b[1]);
          mma16816(acc, a1, b[2], b[3]);
        }
        const int r0 = mt * 16 + (lane >> 2), j0 = nt * 8 + 2 * (lane & 3);
#pragma unroll
        for (int h = 0; h < 2; h++) {
          const int r = r0 + 8 * h;
          if (r < G) {
            if (j0 < n) sc[r * T::NPOS + j0] = acc[2 * h];
            if (j0 + 1 < n) sc[r * T::NPOS + j0 + 1] = acc[2 * h + 1];
          }
        }
      }
    }
    __syncthreads();
    if (!two) {
      stage(kb, true);  // every read of the keys is done
      cp_async_commit();
    }
    // softmax: warp w takes rows w, w + 16, ...; lane takes positions lane + 32i
    {
#pragma unroll 1
      for (int r = warp; r < G; r += T::NW) {
        const float* row = sc + r * T::NPOS;
        float v[4], mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const int j = lane + 32 * i;
          v[i] = j < n ? row[j] : -INFINITY;
          mx = fmaxf(mx, v[i]);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m = __fmul_rn(mx, p.c);
        float e[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const int j = lane + 32 * i;
          const float pj = j < n ? ex2_approx(__fmaf_rn(v[i], p.c, -m)) : 0.f;
          const __nv_bfloat16 pb16 = __float2bfloat16_rn(pj);
          e[i] = __bfloat162float(pb16);
          *reinterpret_cast<__nv_bfloat16*>(ob + T::p_off(G, two) + swz(r, j >> 3, T::PRB) + (j & 7) * 2) = pb16;
        }
        float l = __fadd_rn(__fadd_rn(e[0], e[1]), __fadd_rn(e[2], e[3]));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) l = __fadd_rn(l, __shfl_xor_sync(0xffffffffu, l, o));
        if (lane == 0) {
          mown[r] = m;
          lown[r] = l;
        }
      }
    }
    cp_async_wait_group<0>();  // values
    __syncthreads();
    // O = P V: warp items (row tile, pair of 8-column tiles of the head dimension)
    {
      const int nk = n16 >> 4, mi = lane >> 3, rr = lane & 7;
      constexpr int NDT = D / 16;  // column-tile pairs
      for (int it = warp; it < MT * NDT; it += T::NW) {
        const int mt = it / NDT, dt = it % NDT;
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
        const int prow = mt * 16 + (mi & 1) * 8 + rr;
        // V^T fragments: matrices (rows 0-7, cols 2dt), (rows 8-15, 2dt), (0-7, 2dt+1), (8-15, 2dt+1)
        const int vrow_in = (mi & 1) * 8 + rr, vchunk = 2 * dt + (mi >> 1);
        for (int kt = 0; kt < nk; kt++) {
          uint32_t a[4], b[4];
          ldsm_x4(pb + swz(prow, 2 * kt + (mi >> 1), T::PRB), a);
          ldsm_x4_t(vb + swz(16 * kt + vrow_in, vchunk, D * 2), b);
          mma16816(acc0, a, b[0], b[1]);
          mma16816(acc1, a, b[2], b[3]);
        }
        const int r0 = mt * 16 + (lane >> 2), d0 = dt * 16 + 2 * (lane & 3);
#pragma unroll
        for (int h = 0; h < 2; h++) {
          const int r = r0 + 8 * h;
          if (r < G) {
            *reinterpret_cast<float2*>(oown + r * D + d0) = make_float2(acc0[2 * h], acc0[2 * h + 1]);
            *reinterpret_cast<float2*>(oown + r * D + d0 + 8) = make_float2(acc1[2 * h], acc1[2 * h + 1]);
          }
        }
      }
    }
  }
  // the split kernel before this one writes the workspace and may set the status
  pdl_wait();
  pdl_trigger();  // the next kernel may start on SMs this grid leaves free
  if (tid == 0) {
    int bad = status_bad(p.status) ? 1 : 0;
    if (!bad && (ri.L < 0 || ri.L > p.max_len)) {
      set_status(p.status, TV_ERR_LEN);
      bad = 1;
    }
    if (!bad && p.decode && ri.L >= p.cap) {
      set_status(p.status, TV_ERR_CAPACITY);
      bad = 1;
    }
    if (!bad && !rok) bad = 1;  // a malformed tree: reported by tv_tree_prepare
    skip = bad;
  }
  fence_proxy_async_smem();  // this thread's accesses to the own-segment buffers come before the bulk copies
  __syncthreads();  // also: the own segment's O, m and l are in shared memory
  if (skip) return;
  const int ST = p.split_tiles;
  const int n_reg = (R + ST - 1) / ST;
  const bool snap = n_reg > 0 && R != min(n_reg * ST, tend);
  // record i of the node's rows: split i, or the snapshot in place of the last split
  auto rec = [&](int i, int r) -> const float* {
    const int slot = (i == n_reg - 1 && snap) ? snap_slot(p) : i;
    return ws_rec(p, ri.s, g, slot, local * G + r, D);
  };
  const int nst = min(n_reg, p.n_mstage);  // records staged in shared memory
  const uint32_t rbytes = static_cast<uint32_t>(G * T::REC);
  if (warp == 0 && nst > 0) {
    // one lane sets the byte count first; the copies are spread over the warp
    if (lane == 0) mbar_arrive_expect_tx(MBAR, rbytes * nst);
    __syncwarp();
    for (int i = lane; i < nst; i += 32) bulk_g2s(smem_u32(ob) + i * rbytes, rec(i, 0), rbytes, MBAR);
  }
  auto weight = [](float m, float mm) { return m == mm ? 1.f : ex2_approx(__fsub_rn(m, mm)); };
  const bool staged = p.tail_staged != 0;
  float* const wgt = oown + G * D;                           // [n_reg][G]
  float* const lsm = wgt + static_cast<size_t>(n_reg) * G;   // [n_reg][G]
  float* const ltot = lsm + static_cast<size_t>(n_reg) * G;  // [G] max, then [G] sum
  float* const wown = ltot + G;                              // [G] own weight
  if (staged) {
    for (int idx = tid; idx < n_reg * G; idx += T::NT) {
      const float4 t4 = *reinterpret_cast<const float4*>(rec(idx / G, idx % G) + D);  // m, l_A, l_B, pad
      wgt[idx] = t4.x;
      lsm[idx] = __fadd_rn(t4.y, t4.z);
    }
    __syncthreads();
    for (int r = tid; r < G; r += T::NT) {
      float mm = mown[r];
      for (int i = 0; i < n_reg; i++) mm = fmaxf(mm, wgt[i * G + r]);
      ltot[r] = mm;
    }
    __syncthreads();
    for (int idx = tid; idx < n_reg * G; idx += T::NT) wgt[idx] = weight(wgt[idx], ltot[idx % G]);
    for (int r = tid; r < G; r += T::NT) wown[r] = weight(mown[r], ltot[r]);
    __syncthreads();
    for (int r = tid; r < G; r += T::NT) {
      float ls = 0.f;
      for (int i = 0; i < n_reg; i++) ls = __fmaf_rn(wgt[i * G + r], lsm[i * G + r], ls);
      ltot[r] = __fmaf_rn(wown[r], lown[r], ls);
    }
  }
  // the staged records have landed (every thread observes the barrier, and
  // no copy is in flight when the CTA leaves, whatever happened before)
  if (__syncthreads_or(nst > 0 && !mbar_wait(MBAR, 0, kWaitCycles))) {
    if (tid == 0) set_status(p.status, TV_ERR_TIMEOUT);
    return;
  }
  const float4* const st4 = reinterpret_cast<const float4*>(ob);
  for (int idx = tid; idx < G * (D / 4); idx += T::NT) {
    const int r = idx / (D / 4), c4 = idx % (D / 4);
    float mm = 0.f, ls = 0.f, wo = 0.f;
    if (!staged) {
      mm = mown[r];
      for (int i = 0; i < n_reg; i++) mm = fmaxf(mm, rec(i, r)[D]);
      for (int i = 0; i < n_reg; i++) {
        const float4 t4 = *reinterpret_cast<const float4*>(rec(i, r) + D);
        ls = __fmaf_rn(weight(t4.x, mm), __fadd_rn(t4.y, t4.z), ls);
      }
      wo = weight(mown[r], mm);
      ls = __fmaf_rn(wo, lown[r], ls);
    } else {
      ls = ltot[r];
      wo = wown[r];
    }
    auto wt = [&](int i) { return staged ? wgt[i * G + r] : weight(rec(i, r)[D], mm); };
    // records in order: the staged ones from shared memory (the first
    // unstaged ones already in flight), then the rest MB at a time, then
    // the own state
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 v[T::MB];
#pragma unroll
    for (int u = 0; u < T::MB; u++)
      if (nst + u < n_reg) v[u] = reinterpret_cast<const float4*>(rec(nst + u, r))[c4];
#pragma unroll 4
    for (int i = 0; i < nst; i++) {
      const float4 x = st4[(i * G + r) * (T::REC / 16) + c4];
      const float w = wt(i);
      o.x = __fmaf_rn(w, x.x, o.x);
      o.y = __fmaf_rn(w, x.y, o.y);
      o.z = __fmaf_rn(w, x.z, o.z);
      o.w = __fmaf_rn(w, x.w, o.w);
    }
    for (int i0 = nst; i0 < n_reg; i0 += T::MB) {
      if (i0 > nst) {
#pragma unroll
        for (int u = 0; u < T::MB; u++)
          if (i0 + u < n_reg) v[u] = reinterpret_cast<const float4*>(rec(i0 + u, r))[c4];
      }
#pragma unroll
      for (int u = 0; u < T::MB; u++) {
        if (i0 + u < n_reg) {
          const float w = wt(i0 + u);
          o.x = __fmaf_rn(w, v[u].x, o.x);
          o.y = __fmaf_rn(w, v[u].y, o.y);
          o.z = __fmaf_rn(w, v[u].z, o.z);
          o.w = __fmaf_rn(w, v[u].w, o.w);
        }
      }
    }
    {
      const float4 x = reinterpret_cast<const float4*>(oown + r * D)[c4];
      o.x = __fmaf_rn(wo, x.x, o.x);
      o.y = __fmaf_rn(wo, x.y, o.y);
      o.z = __fmaf_rn(wo, x.z, o.z);
      o.w = __fmaf_rn(wo, x.w, o.w);
    }
    const size_t oi = (static_cast<size_t>(node_g) * p.Hq + g * G + r) * D + 4 * c4;
    float4 y = make_float4(__fdiv_rn(o.x, ls), __fdiv_rn(o.y, ls), __fdiv_rn(o.z, ls), __fdiv_rn(o.w, ls));
    if (p.gate) {
      const uint2 gw = *reinterpret_cast<const uint2*>(p.gate + oi);
      y = make_float4(gate_mul(y.x, bf16_lo(gw.x)), gate_mul(y.y, bf16_hi(gw.x)), gate_mul(y.z, bf16_lo(gw.y)),
                      gate_mul(y.w, bf16_hi(gw.y)));
    }
    uint2 packed;
    packed.x = pack_bf16x2(y.x, y.y);
    packed.y = pack_bf16x2(y.z, y.w);
    *reinterpret_cast<uint2*>(p.out + oi) = packed;
  }
  if (p.decode) {
    // append the token's own key/value at row L
    const size_t dst = (static_cast<size_t>(g) * p.cap + ri.L) * D;
    const size_t src = (static_cast<size_t>(node_g) * p.Hkv + g) * D;
    for (int cc = tid; cc < D / 8; cc += T::NT) {
      reinterpret_cast<uint4*>(p.K[ri.s] + dst)[cc] = reinterpret_cast<const uint4*>(p.kt + src)[cc];
      reinterpret_cast<uint4*>(p.V[ri.s] + dst)[cc] = reinterpret_cast<const uint4*>(p.vt + src)[cc];
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// [Hkv * cap rows][D] bf16 cache as a 2-D tensor with 64 x 64 128B-swizzled boxes.
static bool encode_cache_map(CUtensorMap* m, void* base, int D, int rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int max_splits_for(int split_tiles, int max_len) {
  return (max_len + TV_MAX_PATH + split_tiles * kTile - 1) / (split_tiles * kTile) + 1;
}

// Workspace: per (sequence, KV head), max_splits split records and the
// snapshot record, each [rows][O[D], m, l_A, l_B, pad].
size_t attn_tc_ws_bytes(const tv_plan* plan, const tv_attn_layer* layer, int n_seq, int n_max, int max_len) {
  if (!plan || !layer || plan->split < kTile || plan->split % kTile) return 0;
  const int G = layer->Hq / (layer->Hkv > 0 ? layer->Hkv : 1);
  const size_t slots = static_cast<size_t>(max_splits_for(plan->split / kTile, max_len)) + 1;
  return static_cast<size_t>(n_seq) * layer->Hkv * slots * static_cast<size_t>(n_max) * G * (layer->D + 4) * 4;
}

// Dynamic shared memory the tail kernel may use (the per-block limit less
// its static arrays, with a margin), and the most that leaves room for two
// tail CTAs on an SM.
constexpr int kTailSmemMax = 232448 - 2048;
constexpr int kTailSmemTwoPerSm = 112 * 1024;

template <int D>
static tv_status launch_tc(TcParams& p, int n_items_bound, int n_units, cudaStream_t st, bool ov) {
  using C = Tc<D>;
  using T = Tail<D>;
  p.ws_splits = p.max_splits + 1;
  // weights and sums of every split record staged when they fit
  const int wb = T::wbytes(p.G, p.max_splits);
  p.tail_staged = T::a_off(p.G, wb) + T::own_bytes(p.G, false) <= kTailSmemMax ? 1 : 0;
  p.tail_a = T::a_off(p.G, p.tail_staged ? wb : 0);
  // keys and values staged at once while the tail CTAs fit one wave at one
  // CTA per SM; otherwise one buffer, so that two CTAs share an SM
  p.tail_two = (n_units <= num_sms() && p.tail_a + T::own_bytes(p.G, true) <= kTailSmemMax) ? 1 : 0;
  const int base = p.tail_a + T::own_bytes(p.G, p.tail_two != 0);
  if (base > kTailSmemMax) return TV_ERR_SHAPE;
  const int cap = p.tail_two || base > kTailSmemTwoPerSm ? kTailSmemMax : kTailSmemTwoPerSm;
  // split records staged for the merge: as many as the budget holds
  const int rbytes = p.G * T::REC;
  const int want = p.tail_a + p.max_splits * rbytes;
  const int smem_tail = want > base ? (want < cap ? want : cap) : base;
  p.n_mstage = (smem_tail - p.tail_a) / rbytes;
  // one-time attribute setup (never inside a stream capture after the first call)
  static bool attrs = false;
  if (!attrs) {
    if (cudaFuncSetAttribute(attn_split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_SPLIT) !=
            cudaSuccess ||
        cudaFuncSetAttribute(attn_tail_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTailSmemMax) !=
            cudaSuccess)
      return TV_ERR_CUDA;
    attrs = true;
  }
  if (n_items_bound > 0) {
    // pair mode: two CTAs per item (row blocks 0 and 1), at most one CTA per SM
    const int per = p.pair ? 2 : 1;
    const int units = n_items_bound < num_sms() / per ? n_items_bound : num_sms() / per;
    launch_k(ov, attn_split_kernel<D>, dim3(per * units), dim3(384), C::SMEM_SPLIT, st, p);
  }
  launch_k(ov, attn_tail_kernel<D>, dim3(n_units), dim3(T::NT), smem_tail, st, p);
  return launch_status();
}

tv_status attn_tc_launch(const tv_plan* plan, const AttnCall& a, void* ws, size_t ws_bytes, cudaStream_t st) {
  const tv_attn_layer* l = a.layer;
  if (!plan || plan->split < kTile || plan->split % kTile) return TV_ERR_ARG;
  const int G = l->Hq / l->Hkv;
  if (G > kMaxGroup) return TV_ERR_SHAPE;
  const int n_max = a.decode ? 1 : a.n_max;
  const size_t need = attn_tc_ws_bytes(plan, l, a.n_seq, n_max, a.max_len);
  if (!ws || ws_bytes < need) return TV_ERR_WORKSPACE;
  if (!aligned16(ws)) return TV_ERR_ALIGN;
  static_assert(alignof(TcParams) >= 64, "tensor maps need 64-byte alignment");
  TcParams p;
  memset(&p, 0, sizeof(p));
  for (int s = 0; s < a.n_seq; s++) {
    if (!l->K[s] || !l->V[s]) return TV_ERR_ARG;
    if (!aligned16(l->K[s]) || !aligned16(l->V[s])) return TV_ERR_ALIGN;
    p.K[s] = static_cast<__nv_bfloat16*>(l->K[s]);
    p.V[s] = static_cast<__nv_bfloat16*>(l->V[s]);
    if (!encode_cache_map(&p.tmK[s], l->K[s], l->D, l->Hkv * l->cap) ||
        !encode_cache_map(&p.tmV[s], l->V[s], l->D, l->Hkv * l->cap))
      return TV_ERR_CUDA;
  }
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.kt = static_cast<const __nv_bfloat16*>(a.kt);
  p.vt = static_cast<const __nv_bfloat16*>(a.vt);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.gate = static_cast<const __nv_bfloat16*>(a.gate);
  p.len = a.len;
  p.node_off = a.node_off;
  p.meta = a.meta;
  p.status = a.status;
  p.ws = static_cast<float*>(ws);
  p.n_seq = a.n_seq;
  p.n_total = a.n_total;
  p.Hq = l->Hq;
  p.Hkv = l->Hkv;
  p.G = G;
  p.cap = l->cap;
  p.max_len = a.max_len;
  p.split_tiles = plan->split / kTile;
  p.max_splits = max_splits_for(p.split_tiles, a.max_len);
  p.rows_max = n_max * G;
  p.decode = a.decode;
  p.c = a.scale * 1.4426950408889634f;
  // the split kernel runs at most floor(max_len / 64) tiles of a sequence
  const int tiles_bound = a.max_len / kTile;
  const int splits_bound = (tiles_bound + p.split_tiles - 1) / p.split_tiles;
  // pair mode when the largest tree spans exactly two 128-row blocks (and a
  // tile's boxes split evenly between the two CTAs)
  const int nrb_max = (n_max * G + 127) / 128;
  p.pair = (!a.decode && l->D >= 128 && nrb_max == 2) ? 1 : 0;
  const int items_bound = a.n_seq * l->Hkv * splits_bound * (p.pair ? 1 : nrb_max);
  const int n_units = (a.decode ? a.n_seq : a.n_total) * l->Hkv;
  switch (l->D) {
    case 64: return launch_tc<64>(p, items_bound, n_units, st, a.overlap);
    case 128: return launch_tc<128>(p, items_bound, n_units, st, a.overlap);
    case 256: return launch_tc<256>(p, items_bound, n_units, st, a.overlap);
    default: return TV_ERR_SHAPE;
  }
}

}  // namespace tv
