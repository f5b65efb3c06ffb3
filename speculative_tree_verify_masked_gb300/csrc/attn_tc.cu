// Tree-masked grouped-query attention for bf16 KV caches on the tcgen05 tensor
// cores ("One request, end to end" 2.6: one forward pass verifies the whole
// tree; "Adding a model" step 4: every verified row equals the decode row).
//
// Row function.  Row (node, query head) sees logical positions 0 .. L+d: the
// L cache rows, then its ancestors-or-self at L .. L+d.  Positions are cut
// into tiles of 64 and splits of plan.split positions, both aligned at
// absolute position 0.  Within a split the tiles run in order through one
// online softmax: S = Q K^T on the tensor core (fp32); the tile's 64 slots are
// handled as two halves of 32 that share the scaled tile max; p = 2^(s*c - m)
// rounded to bf16; each half keeps its own running sum of the rounded p;
// O = O * alpha + P V on the tensor core.  Splits are merged in split order.
// The running state (m, l_A, l_B, O) is carried between kernels as exact
// fp32 and every tile update runs the same code, so the result depends only
// on the row's query and key sequence: a node verified in a tree and the same
// token decoded after its ancestors were committed produce the same bits.
//
// Kernels.
//  split kernel (persistent, one CTA per SM): the tiles that every node of a
//    sequence shares (positions below 64*floor(L/64), all cache rows) for up to
//    128 query rows (node x head of one KV head) at once.  Warps 0 and 10
//    stream K and V tiles with TMA (128B-swizzled boxes) through two rings,
//    prefetching into L2 the tile two ahead (and, before the wait for the
//    previous kernel, the first tiles);
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
//    of every tile's boxes into L2.  Each split's state goes to the workspace.
//  tail kernel (one CTA per node and KV head): the node's own tiles (cache
//    rows past the last shared tile plus its ancestors at their logical
//    slots, gathered into shared memory with cp.async, the first one before
//    the wait for the split kernel), continuing the split state the split
//    kernel left, then the in-order merge of all splits and the bf16 output
//    (times the front end's sigmoid gate when one is given).
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
  static constexpr int NBAR = 2 * (NK + NV) + 2 * NP + 9;
  static constexpr int SMEM_SPLIT = 1024 + RING + NBAR * 8 + 16;
  // tail kernel: tiles, P, barriers, then (sized at launch) the staged
  // partial states of the splits the split kernel finished
  static constexpr int TAIL_FIXED = 1024 + 2 * TILE + PTILE + 1024;
  static constexpr int REC = D + 4;  // workspace record: O[D], m, l_A, l_B, pad
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
  int n_mstage;  // tail kernel: finished splits whose states are staged in shared memory
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
__device__ __forceinline__ float* ws_rec(const TcParams& p, int s, int g, int split, int row, int D) {
  return p.ws + ((((static_cast<size_t>(s) * p.Hkv + g) * p.max_splits + split) * p.rows_max + row) *
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
// split kernel
// ---------------------------------------------------------------------------
struct ItemSpace {
  int cum[TV_MAX_SEQ + 1];
  int tsh[TV_MAX_SEQ];   // shared tiles of each sequence
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
    is.tsh[s] = L / kTile;
    const int nsplit = (is.tsh[s] + p.split_tiles - 1) / p.split_tiles;
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
  it.t1 = min(it.t0 + p.split_tiles, is.tsh[s]);
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
  const uint32_t XBAR0 = DRAIN + 16u;  // [2] half-max exchange, by tile parity
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
      mbar_init(XBAR0 + 8u * b, 256);
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
  // L2 prefetch of the first item's first tiles while the previous kernel
  // finishes: a prefetch only warms L2 (the point of coherence), so it is
  // safe whatever the previous kernel writes, and the ring's first loads
  // then hit L2.
  if ((warp == 0 || warp == 10) && lane == 0 && cid < total) {
    const Item I = item_at(is, p, cid, rank);
    const CUtensorMap* maps = warp == 0 ? p.tmK : p.tmV;
    const int nfirst = min(I.t1 - I.t0, (warp == 0 ? C::NK : C::NV) + kL2Ahead);
    for (int t = I.t0; t < I.t0 + nfirst; t++)
      for (int kb = kb0; kb < kb1; kb++) tma_prefetch_l2_2d(&maps[I.s], kb * 64, I.g * p.cap + t * kTile);
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
        const float mh = half_max(sv, kHalf);
        xmax[b][hf][lrow] = mh;
        mbar_arrive(XBAR0 + 8u * b);
        if (!wait_warp(XBAR0 + 8u * b, (t >> 1) & 1, abort_flag, kWaitCycles)) {
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
      const int rbase = I.rb * 128 + quad * 32, nrows = is.rows[I.s];
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

// ---------------------------------------------------------------------------
// tail kernel: the node's own tiles, then the split merge
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <int D>
__global__ void __launch_bounds__(256, 1) attn_tail_kernel(const __grid_constant__ TcParams p) {
  using C = Tc<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int skip;
  __shared__ float xmax[2][128];
  __shared__ int anc_s[TV_MAX_PATH];  // global node of the ancestor at each depth
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (sb - raw);
  const uint32_t pbase = sb + 2 * C::TILE;  // P tile (the PV A operand)
  const uint32_t BAR = pbase + C::PTILE, DRAIN = BAR + 8, MBAR = BAR + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + 2 * C::TILE + C::PTILE + 16);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hf = warp >> 2;  // softmax half of this thread
  const int lrow = (warp & 3) * 32 + lane;
  const int item = blockIdx.x;
  const int g = item % p.Hkv;
  const int node_g = item / p.Hkv;  // global node (verify) or sequence (decode)
  // the node's sequence, offset, depth, ancestors and context length, with
  // every global load issued before any result is used
  int s = 0, off = 0, depth = 0, L = 0;
  if (p.decode) {
    s = node_g;
    off = node_g;
    L = p.len[s];
    if (threadIdx.x < TV_MAX_PATH) anc_s[threadIdx.x] = node_g;
  } else {
    int ends[TV_MAX_SEQ], lens[TV_MAX_SEQ];
#pragma unroll
    for (int i = 0; i < TV_MAX_SEQ; i++) {
      ends[i] = i < p.n_seq ? p.node_off[i + 1] : 0;
      lens[i] = i < p.n_seq ? p.len[i] : 0;
    }
    const int off0 = p.node_off[0];
    MetaView mv = meta_view(const_cast<void*>(p.meta), p.n_total);
    depth = mv.depth[node_g];
    depth = depth < 0 ? 0 : (depth >= TV_MAX_PATH ? TV_MAX_PATH - 1 : depth);
    const int a = threadIdx.x < TV_MAX_PATH ? mv.anc_at[static_cast<size_t>(node_g) * TV_MAX_PATH + threadIdx.x] : 0;
    off = off0;
    L = lens[0];
#pragma unroll
    for (int i = 0; i + 1 < TV_MAX_SEQ; i++) {
      if (i + 1 < p.n_seq && node_g >= ends[i]) {
        s = i + 1;
        off = ends[i];
        L = lens[i + 1];
      }
    }
    // clamped to the node buffers: with a malformed tree (reported by
    // tv_tree_prepare) the tables may be stale, and the first tile is
    // gathered before the status word is read
    const int an = threadIdx.x > depth ? node_g : off + a;
    if (threadIdx.x < TV_MAX_PATH) anc_s[threadIdx.x] = an < 0 ? 0 : (an >= p.n_total ? p.n_total - 1 : an);
  }
  const int local = node_g - off;
  const int G = p.G;
  // Set-up that needs nothing the split kernel writes: barriers, TMEM and,
  // when they fit in the P tile area, the node's query rows and its first
  // own tile (cache rows and tree rows), so that their loads overlap the
  // split kernel's last CTAs.  The carried split state waits for it.
  if (threadIdx.x == 0) {
    mbar_init(BAR, 1);
    mbar_init(DRAIN, 1);
    mbar_init(MBAR, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::COLS);
    tmem_relinquish();
  }
  const bool lok = L >= 0 && L <= p.max_len && !(p.decode && L >= p.cap);
  const uint32_t qbytes = static_cast<uint32_t>(G * D * 2 + 15) & ~15u;
  const bool early = lok && qbytes + static_cast<uint32_t>(G * C::REC * 4) <= static_cast<uint32_t>(C::PTILE);
  const uint32_t qstage = early ? pbase : sb + C::TILE, ostage = early ? pbase + qbytes : sb;
  const int P = L + depth + 1;
  const int tsh = lok ? L / kTile : 0;
  // the node's K/V tile t: cache rows below L, ancestors at L..L+d, zeros after
  auto gather = [&](int t) {
    for (int idx = threadIdx.x; idx < kTile * (D / 8); idx += blockDim.x) {
      const int j = idx / (D / 8), cc = idx % (D / 8), pos = t * kTile + j;
      const __nv_bfloat16* ksrc = p.kt;
      const __nv_bfloat16* vsrc = p.vt;
      bool have = false;
      if (pos < L) {
        const size_t r = (static_cast<size_t>(g) * p.cap + pos) * D + cc * 8;
        ksrc = p.K[s] + r;
        vsrc = p.V[s] + r;
        have = true;
      } else if (pos < P) {
        const size_t r = (static_cast<size_t>(anc_s[pos - L]) * p.Hkv + g) * D + cc * 8;
        ksrc = p.kt + r;
        vsrc = p.vt + r;
        have = true;
      }
      const int kb = cc >> 3, c = cc & 7;
      const uint32_t o = kb * kBox + (j >> 3) * 1024 + (j & 7) * 128 + ((c ^ (j & 7)) << 4);
      cp_async16(sb + o, ksrc, have);
      cp_async16(sb + C::TILE + o, vsrc, have);
    }
  };
  if (early) {
    __syncthreads();  // anc_s
    const __nv_bfloat16* qsrc = p.q + (static_cast<size_t>(node_g) * p.Hq + g * G) * D;
    for (int idx = threadIdx.x; idx < G * D / 8; idx += blockDim.x) cp_async16(qstage + idx * 16, qsrc + idx * 8, true);
    gather(tsh);
  }
  // the split kernel before this one writes the workspace and may set the status
  pdl_wait();
  if (threadIdx.x == 0) {
    int bad = status_bad(p.status) ? 1 : 0;
    if (!bad && (L < 0 || L > p.max_len)) {
      set_status(p.status, TV_ERR_LEN);
      bad = 1;
    }
    if (!bad && p.decode && L >= p.cap) {
      set_status(p.status, TV_ERR_CAPACITY);
      bad = 1;
    }
    skip = bad;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t tl = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);

  if (skip) cp_async_wait_all();  // copies issued before the wait land before the CTA leaves
  if (!skip) {
    const int tlast = (L + depth) / kTile;
    const int ST = p.split_tiles;
    const bool vrow = lrow < G;
    const int row_seq = local * G + lrow;
    int cur = tsh / ST;
    const bool cont = (tsh % ST) != 0;  // the split kernel started this split

    // The finished splits' states (the node's G rows of a split are one
    // contiguous block) come in by bulk copies issued first thing after the
    // wait, so their latency hides behind the carried state, the queries and
    // the node's own tiles; the node's final split state is kept in shared
    // memory too.  Shared layout: [nst][G][REC], then [G][REC].
    const uint32_t mst_s = sb + (C::TAIL_FIXED - 1024);
    const int nst = min(cur, p.n_mstage);
    const uint32_t mown_s = mst_s + static_cast<uint32_t>(nst * G * C::REC * 4);
    float* const mown = reinterpret_cast<float*>(gb + (C::TAIL_FIXED - 1024) + nst * G * C::REC * 4);
    if (warp == 0 && nst > 0) {
      // one lane sets the byte count first; the copies are spread over the warp
      const uint32_t bytes = static_cast<uint32_t>(G * C::REC * 4);
      if (lane == 0) mbar_arrive_expect_tx(MBAR, bytes * nst);
      __syncwarp();
      for (int sp = lane; sp < nst; sp += 32)
        bulk_g2s(mst_s + sp * bytes, ws_rec(p, s, g, sp, local * G, D), bytes, MBAR);
    }
    // stage this node's G query rows (unless staged early) and, when
    // continuing, the carried state records with cp.async
    const bool ostaged = early || G * C::REC * 4 <= C::TILE;
    {
      if (!early) {
        const __nv_bfloat16* qsrc = p.q + (static_cast<size_t>(node_g) * p.Hq + g * G) * D;
        for (int idx = threadIdx.x; idx < G * D / 8; idx += blockDim.x)
          cp_async16(qstage + idx * 16, qsrc + idx * 8, true);
      }
      if (cont && ostaged) {
        for (int idx = threadIdx.x; idx < G * C::REC / 4; idx += blockDim.x) {
          const int r = idx / (C::REC / 4), cc = idx % (C::REC / 4);
          cp_async16(ostage + idx * 16, ws_rec(p, s, g, cur, local * G + r, D) + cc * 4, true);
        }
      }
      cp_async_wait_all();
      __syncthreads();
    }
    // Q and the carried O into TMEM (each half its own columns)
    {
      const uint4* qs = reinterpret_cast<const uint4*>(gb + (qstage - sb)) + lrow * (D / 8);
#pragma unroll 1
      for (int c0 = hf * (D / 4); c0 < (hf + 1) * (D / 4); c0 += 32) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 8; i++) {
          const uint4 v = vrow ? qs[c0 / 4 + i] : make_uint4(0u, 0u, 0u, 0u);
          r[4 * i] = v.x;
          r[4 * i + 1] = v.y;
          r[4 * i + 2] = v.z;
          r[4 * i + 3] = v.w;
        }
        tmem_st32(tl + C::T_Q + c0, r);
      }
    }
    float m = -INFINITY, lh = 0.f;
    bool fresh = true;
    if (cont) {
      const float* rec = vrow ? (ostaged ? reinterpret_cast<const float*>(gb + (ostage - sb)) + lrow * C::REC
                                         : ws_rec(p, s, g, cur, row_seq, D))
                              : nullptr;
#pragma unroll 1
      for (int c0 = hf * (D / 2); c0 < (hf + 1) * (D / 2); c0 += 32) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 8; i++) {
          const uint4 v = rec ? reinterpret_cast<const uint4*>(rec + c0)[i] : make_uint4(0u, 0u, 0u, 0u);
          r[4 * i] = v.x;
          r[4 * i + 1] = v.y;
          r[4 * i + 2] = v.z;
          r[4 * i + 3] = v.w;
        }
        tmem_st32(tl + C::T_O + c0, r);
      }
      if (rec) {
        m = rec[D];
        lh = rec[D + 1 + hf];
      }
      fresh = false;
    }
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    uint32_t ph = 0;
    bool ok = true;
    for (int t = tsh; t <= tlast && ok; t++) {
      if (t / ST != cur) {
        store_state<D>(tl + C::T_O, vrow ? ws_rec(p, s, g, cur, row_seq, D) : nullptr, hf, m, lh);
        cur = t / ST;
        fresh = true;
        m = -INFINITY;
        lh = 0.f;
      }
      // the node's K/V tile (the first one may have been gathered before the wait)
      if (!(early && t == tsh)) gather(t);
      cp_async_wait_all();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (threadIdx.x == 0) {
        issue_qk<D>(tbase + C::T_S, tbase + C::T_Q, sb);
        tc_commit(BAR);
      }
      if (__syncthreads_or(!mbar_wait(BAR, ph, kWaitCycles))) {
        ok = false;
        break;
      }
      ph ^= 1;
      tc_fence_after();
      float sv[kHalf];
      tmem_ld32f(tl + C::T_S + hf * kHalf, sv);
      const int nvalid = min(kTile, P - t * kTile) - hf * kHalf;
      const float mh = half_max(sv, nvalid);
      xmax[hf][lrow] = mh;
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      const float mo = xmax[hf ^ 1][lrow];
      float alpha;
      const float m_new = next_max(m, fmaxf(mh, mo), p.c, alpha);
      uint32_t Pw[kHalf / 2];
      const float rs = half_probs(sv, nvalid, p.c, m_new, Pw);
      lh = __fmaf_rn(lh, alpha, rs);
      m = m_new;
      store_p_half(pbase, lrow, hf, Pw);
      if (!fresh && __any_sync(0xffffffffu, alpha != 1.f))
        rescale_o(tl + C::T_O, hf * (D / 2), (hf + 1) * (D / 2), alpha);
      tmem_st_wait();
      fence_proxy_async_smem();  // P visible to the tensor core
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (threadIdx.x == 0) {
        issue_pv_ss<D>(tbase + C::T_O, pbase, desc_v(sb + C::TILE, 0), !fresh);
        tc_commit(BAR);
      }
      if (__syncthreads_or(!mbar_wait(BAR, ph, kWaitCycles))) {
        ok = false;
        break;
      }
      ph ^= 1;
      tc_fence_after();
      fresh = false;
    }
    // the staged splits have landed (every thread observes the barrier, and
    // no copy is in flight when the CTA leaves, whatever happened before)
    if (__syncthreads_or(nst > 0 && !mbar_wait(MBAR, 0, kWaitCycles))) ok = false;
    if (!ok) {
      set_status(p.status, TV_ERR_TIMEOUT);
    } else {
      store_state<D>(tl + C::T_O, vrow ? mown + lrow * C::REC : nullptr, hf, m, lh);
      __syncthreads();
      // merge splits 0..cur in split order: weights 2^(m_s - max m), sums l_A + l_B
      const int ns = cur + 1;
      // O columns 4*c4 .. 4*c4+3 and (m, l_A, l_B) of split sp, row r
      auto rec4 = [&](int sp, int r, int c4) -> float4 {
        float4 v;
        if (sp < nst || sp == cur) {
          const uint32_t a = (sp < nst ? mst_s + static_cast<uint32_t>((sp * G + r) * C::REC * 4)
                                       : mown_s + static_cast<uint32_t>(r * C::REC * 4)) + 16u * c4;
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                       : "r"(a));
        } else {
          v = reinterpret_cast<const float4*>(ws_rec(p, s, g, sp, local * G + r, D))[c4];
        }
        return v;
      };
      float* wsm = reinterpret_cast<float*>(gb);                 // [ns][G] weights (tile area is free now)
      float* ltot = wsm + static_cast<size_t>(ns) * G;           // [G]
      const bool wstaged = (2 * static_cast<size_t>(ns) * G + 2 * G) * 4 <= 2 * C::TILE;
      if (wstaged) {
        // (m, l_A + l_B) of every (split, row), loaded in parallel
        float* lsm = ltot + G;  // [ns][G]
        for (int base = threadIdx.x; base < ns * G; base += 4 * blockDim.x) {
          float mv4[4], la[4], lb[4];
#pragma unroll
          for (int u = 0; u < 4; u++) {
            const int idx = base + u * blockDim.x;
            if (idx < ns * G) {
              const float4 t4 = rec4(idx / G, idx % G, D / 4);  // m, l_A, l_B, pad
              mv4[u] = t4.x;
              la[u] = t4.y;
              lb[u] = t4.z;
            }
          }
#pragma unroll
          for (int u = 0; u < 4; u++) {
            const int idx = base + u * blockDim.x;
            if (idx < ns * G) {
              wsm[idx] = mv4[u];
              lsm[idx] = __fadd_rn(la[u], lb[u]);
            }
          }
        }
        __syncthreads();
        // max reference per row, then every weight in parallel, then the sums in split order
        float* mref = lsm + static_cast<size_t>(ns) * G;  // [G]
        for (int r = threadIdx.x; r < G; r += blockDim.x) {
          float mm = -INFINITY;
#pragma unroll 8
          for (int sp = 0; sp < ns; sp++) mm = fmaxf(mm, wsm[sp * G + r]);
          mref[r] = mm;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < ns * G; idx += blockDim.x) {
          const float ms = wsm[idx], mm = mref[idx % G];
          wsm[idx] = (ms == mm) ? 1.f : ex2_approx(__fsub_rn(ms, mm));
        }
        __syncthreads();
        for (int r = threadIdx.x; r < G; r += blockDim.x) {
          float ls = 0.f;
#pragma unroll 8
          for (int sp = 0; sp < ns; sp++) ls = __fmaf_rn(wsm[sp * G + r], lsm[sp * G + r], ls);
          ltot[r] = ls;
        }
        __syncthreads();
      }
      for (int idx = threadIdx.x; idx < G * (D / 4); idx += blockDim.x) {
        const int r = idx / (D / 4), c4 = idx % (D / 4);
        float mm = 0.f, ls = 0.f;
        if (!wstaged) {
          mm = -INFINITY;
          for (int sp = 0; sp < ns; sp++) mm = fmaxf(mm, rec4(sp, r, D / 4).x);
        }
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        if (wstaged && nst == cur) {
          // every split's record is in shared memory (the common case): plain
          // shared loads the compiler can batch, accumulated in split order
          const float4* st4 = reinterpret_cast<const float4*>(gb + (C::TAIL_FIXED - 1024)) + r * (C::REC / 4) + c4;
#pragma unroll 4
          for (int sp = 0; sp < cur; sp++) {
            const float4 v = st4[static_cast<size_t>(sp) * G * (C::REC / 4)];
            const float wgt = wsm[sp * G + r];
            o.x = __fmaf_rn(wgt, v.x, o.x);
            o.y = __fmaf_rn(wgt, v.y, o.y);
            o.z = __fmaf_rn(wgt, v.z, o.z);
            o.w = __fmaf_rn(wgt, v.w, o.w);
          }
          {
            const float4 v = reinterpret_cast<const float4*>(mown + r * C::REC)[c4];
            const float wgt = wsm[cur * G + r];
            o.x = __fmaf_rn(wgt, v.x, o.x);
            o.y = __fmaf_rn(wgt, v.y, o.y);
            o.z = __fmaf_rn(wgt, v.z, o.z);
            o.w = __fmaf_rn(wgt, v.w, o.w);
          }
          ls = ltot[r];
        } else if (wstaged) {
          // up to 16 splits' partial rows in flight at a time, accumulated in split order
          for (int sp0 = 0; sp0 < ns; sp0 += 16) {
            float4 v[16];
#pragma unroll
            for (int u = 0; u < 16; u++)
              if (sp0 + u < ns) v[u] = rec4(sp0 + u, r, c4);
#pragma unroll
            for (int u = 0; u < 16; u++) {
              if (sp0 + u < ns) {
                const float wgt = wsm[(sp0 + u) * G + r];
                o.x = __fmaf_rn(wgt, v[u].x, o.x);
                o.y = __fmaf_rn(wgt, v[u].y, o.y);
                o.z = __fmaf_rn(wgt, v[u].z, o.z);
                o.w = __fmaf_rn(wgt, v[u].w, o.w);
              }
            }
          }
          ls = ltot[r];
        } else {
          for (int sp = 0; sp < ns; sp++) {
            const float4 t4 = rec4(sp, r, D / 4);
            const float ms = t4.x;
            const float wgt = (ms == mm) ? 1.f : ex2_approx(__fsub_rn(ms, mm));
            ls = __fmaf_rn(wgt, __fadd_rn(t4.y, t4.z), ls);
            const float4 v = rec4(sp, r, c4);
            o.x = __fmaf_rn(wgt, v.x, o.x);
            o.y = __fmaf_rn(wgt, v.y, o.y);
            o.z = __fmaf_rn(wgt, v.z, o.z);
            o.w = __fmaf_rn(wgt, v.w, o.w);
          }
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
        const size_t dst = (static_cast<size_t>(g) * p.cap + L) * D;
        const size_t src = (static_cast<size_t>(node_g) * p.Hkv + g) * D;
        for (int cc = threadIdx.x; cc < D / 8; cc += blockDim.x) {
          reinterpret_cast<uint4*>(p.K[s] + dst)[cc] = reinterpret_cast<const uint4*>(p.kt + src)[cc];
          reinterpret_cast<uint4*>(p.V[s] + dst)[cc] = reinterpret_cast<const uint4*>(p.vt + src)[cc];
        }
      }
    }
    if (threadIdx.x == 0) {
      tc_commit(DRAIN);
      mbar_wait(DRAIN, 0, kWaitCycles);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, C::COLS);
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

size_t attn_tc_ws_bytes(const tv_plan* plan, const tv_attn_layer* layer, int n_seq, int n_max, int max_len) {
  if (!plan || !layer || plan->split < kTile || plan->split % kTile) return 0;
  const int G = layer->Hq / (layer->Hkv > 0 ? layer->Hkv : 1);
  const size_t splits = static_cast<size_t>(max_splits_for(plan->split / kTile, max_len));
  return static_cast<size_t>(n_seq) * layer->Hkv * splits * static_cast<size_t>(n_max) * G * (layer->D + 4) * 4;
}

// Dynamic shared memory the tail kernel may use (the per-block limit less
// its static arrays, with a margin).
constexpr int kTailSmemMax = 232448 - 2048;

template <int D>
static tv_status launch_tc(TcParams& p, int n_items_bound, int n_tail, cudaStream_t st, bool ov) {
  using C = Tc<D>;
  // stage as many finished splits' states as fit next to the tail's tiles
  const int per_split = p.G * C::REC * 4;
  const int fit = (kTailSmemMax - C::TAIL_FIXED) / per_split - 1;  // less the node's own final split
  if (fit < 0) return TV_ERR_SHAPE;
  p.n_mstage = fit < p.max_splits ? fit : p.max_splits;
  const int smem_tail = C::TAIL_FIXED + (p.n_mstage + 1) * per_split;
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
  launch_k(ov, attn_tail_kernel<D>, dim3(n_tail), dim3(256), smem_tail, st, p);
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
  const int tiles_bound = a.max_len / kTile;
  const int splits_bound = (tiles_bound + p.split_tiles - 1) / p.split_tiles;
  // pair mode when the largest tree spans exactly two 128-row blocks (and a
  // tile's boxes split evenly between the two CTAs)
  const int nrb_max = (n_max * G + 127) / 128;
  p.pair = (!a.decode && l->D >= 128 && nrb_max == 2) ? 1 : 0;
  const int items_bound = a.n_seq * l->Hkv * splits_bound * (p.pair ? 1 : nrb_max);
  const int n_tail = (a.decode ? a.n_seq : a.n_total) * l->Hkv;
  switch (l->D) {
    case 64: return launch_tc<64>(p, items_bound, n_tail, st, a.overlap);
    case 128: return launch_tc<128>(p, items_bound, n_tail, st, a.overlap);
    case 256: return launch_tc<256>(p, items_bound, n_tail, st, a.overlap);
    default: return TV_ERR_SHAPE;
  }
}

}  // namespace tv
