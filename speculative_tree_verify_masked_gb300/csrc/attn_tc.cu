// Tree-masked grouped-query attention for bf16 KV caches on the tcgen05 tensor
// cores ("One request, end to end" 2.6: one forward pass verifies the whole
// tree; "Adding a model" step 4: every verified row equals the decode row).
//
// Row function.  Row (node, query head) sees logical positions 0 .. L+d: the
// L cache rows, then its ancestors-or-self at L .. L+d.  Positions are cut
// into tiles of 64 and splits of plan.split positions, both aligned at
// absolute position 0.  Within a split the tiles run in order through one
// online softmax: S = Q K^T on the tensor core (fp32), the scaled tile max,
// p = 2^(s*c - m) rounded to bf16, l += sum of the rounded p, O = O*alpha +
// P V on the tensor core.  Splits are merged in split order.  The running
// state (m, l, O) is carried between kernels as exact fp32, and every tile
// update runs the same code, so the result depends only on the row's query
// and key sequence: a node verified in a tree and the same token decoded
// after its ancestors were committed produce the same bits.
//
// Kernels.
//  split kernel (persistent, one CTA per SM): the tiles that every node of a
//    sequence shares (positions below 64*floor(L/64), all cache rows) for up to
//    128 query rows (node x head of one KV head) at once.  Warp 0 streams K/V
//    tiles with TMA (128B-swizzled boxes) through a ring of stages; warp 1
//    issues the tcgen05 MMAs (Q and P live in TMEM, K and V in shared memory,
//    S and O accumulate in TMEM); warps 2-5 run the softmax, one TMEM lane
//    (query row) per thread.  S is double-buffered so QK^T of tile t+1 runs on
//    the tensor core while the softmax of tile t runs.  Each split's (m, l, O)
//    goes to the workspace.
//  tail kernel (one CTA per node and KV head): the node's own tiles (cache
//    rows past the last shared tile plus its ancestors at their logical
//    slots, built in shared memory), continuing the split state left by the
//    split kernel, then the in-order merge of all splits and the bf16 output.
//  Decode runs the same two kernels with a one-node tree per sequence and
//  appends its own K/V row.
#include <cmath>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "host.hpp"
#include "launchers.hpp"
#include "ptx.cuh"

namespace tv {

constexpr int kTile = 64;         // KV positions per tile
constexpr int kBox = 64 * 128;    // one [64 rows x 128 B] 128B-swizzled box

template <int D>
struct Tc {
  static constexpr int KB = D / 64;                 // 64-column boxes per row
  static constexpr int TILE = kTile * D * 2;        // bytes of one K or V tile
  static constexpr int NS = (D == 256) ? 3 : 6;     // pipeline stages
  static constexpr int STAGE = 2 * TILE;
  static constexpr int T_O = 0;                     // TMEM columns: O [D]
  static constexpr int T_S = D;                     //   S/P [2 x 64]
  static constexpr int T_Q = D + 2 * kTile;         //   Q [D/2] (bf16 pairs)
  static constexpr int COLS = (D + 2 * kTile + D / 2) <= 256 ? 256 : 512;
  static constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, kTile, false, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, false, true);
  static constexpr int NBAR = 2 * NS + 7;
  static constexpr int SMEM_SPLIT = 1024 + NS * STAGE + NBAR * 8 + 16;
  static constexpr int SMEM_TAIL = 1024 + 2 * TILE + 16 + 16;
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
  const int32_t* len;
  const int32_t* node_off;
  const void* meta;
  int32_t* status;
  float* ws;
  int n_seq, n_total, Hq, Hkv, G, cap, max_len, split_tiles, max_splits, rows_max, decode;
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
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tO, uint32_t tP, uint32_t vtile, bool acc) {
#pragma unroll
  for (int kk = 0; kk < kTile / 16; kk++)
    tc_mma_ts(tO, tP + kk * 8, desc_v(vtile, kk), Tc<D>::IDESC_PV, (acc || kk > 0) ? 1u : 0u);
}

// Online-softmax update for one tile of one row.  s: raw scores of the tile's
// 64 slots, slots >= nvalid masked.  m is the running max in the exp2 domain
// (scaled by c), l the running sum of the bf16-rounded probabilities.
// Writes the tile's probabilities as packed bf16 pairs and the factor alpha
// that the running O must be multiplied by (exactly 1 when m is unchanged).
__device__ __forceinline__ void softmax_tile(const float (&s)[kTile], int nvalid, float c, float& m, float& l,
                                             uint32_t (&P)[kTile / 2], float& alpha) {
  float mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < kTile; j++) mx = fmaxf(mx, j < nvalid ? s[j] : -INFINITY);
  const float m_new = fmaxf(m, __fmul_rn(mx, c));
  alpha = (m_new == m) ? 1.f : ex2_approx(__fsub_rn(m, m_new));
  const float neg = -m_new;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < kTile; j += 2) {
    const float p0 = j < nvalid ? ex2_approx(__fmaf_rn(s[j], c, neg)) : 0.f;
    const float p1 = j + 1 < nvalid ? ex2_approx(__fmaf_rn(s[j + 1], c, neg)) : 0.f;
    const uint32_t w = pack_bf16x2(p0, p1);
    P[j / 2] = w;
    acc[(j / 2) & 3] = __fadd_rn(acc[(j / 2) & 3], __fadd_rn(bf16_lo(w), bf16_hi(w)));
  }
  const float rs = __fadd_rn(__fadd_rn(acc[0], acc[1]), __fadd_rn(acc[2], acc[3]));
  l = __fmaf_rn(l, alpha, rs);
  m = m_new;
}

__device__ __forceinline__ void tmem_ld64f(uint32_t taddr, float (&s)[kTile]) {
  uint32_t r0[32], r1[32];
  tmem_ld32(taddr, r0);
  tmem_ld32(taddr + 32, r1);
#pragma unroll
  for (int i = 0; i < 32; i++) {
    s[i] = __uint_as_float(r0[i]);
    s[32 + i] = __uint_as_float(r1[i]);
  }
}

template <int D>
__device__ __forceinline__ void rescale_o(uint32_t tO, float alpha) {
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t r[32];
    tmem_ld32(tO + c0, r);
#pragma unroll
    for (int i = 0; i < 32; i++) r[i] = __float_as_uint(__fmul_rn(__uint_as_float(r[i]), alpha));
    tmem_st32(tO + c0, r);
  }
}

// Q row (D bf16) into this thread's TMEM lane, zeros when q == nullptr.
template <int D>
__device__ __forceinline__ void load_q_tmem(uint32_t tQ, const __nv_bfloat16* q) {
#pragma unroll 1
  for (int c0 = 0; c0 < D / 2; c0 += 32) {
    uint32_t r[32];
    if (q) {
      const uint4* s4 = reinterpret_cast<const uint4*>(q) + c0 / 4;
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const uint4 v = s4[i];
        r[4 * i] = v.x;
        r[4 * i + 1] = v.y;
        r[4 * i + 2] = v.z;
        r[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; i++) r[i] = 0u;
    }
    tmem_st32(tQ + c0, r);
  }
}

// Workspace record of (split, row): O[D], m, l, 2 pad floats.
__device__ __forceinline__ float* ws_rec(const TcParams& p, int s, int g, int split, int row, int D) {
  return p.ws + ((((static_cast<size_t>(s) * p.Hkv + g) * p.max_splits + split) * p.rows_max + row) *
                 static_cast<size_t>(D + 4));
}

template <int D>
__device__ __forceinline__ void store_state(uint32_t tO, float* rec, float m, float l) {
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
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
    rec[D] = m;
    rec[D + 1] = l;
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
    int nodes = p.decode ? 1 : p.node_off[s + 1] - p.node_off[s];
    nodes = nodes < 0 ? 0 : (nodes > TV_MAX_NODES ? TV_MAX_NODES : nodes);
    is.off[s] = p.decode ? s : p.node_off[s];
    is.rows[s] = nodes * p.G;
    is.nrb[s] = (is.rows[s] + 127) / 128;
    is.tsh[s] = L / kTile;
    const int nsplit = (is.tsh[s] + p.split_tiles - 1) / p.split_tiles;
    is.cum[s + 1] = is.cum[s] + nsplit * p.Hkv * is.nrb[s];
  }
}

__device__ inline Item item_at(const ItemSpace& is, const TcParams& p, int w) {
  int s = 0;
  while (s < p.n_seq - 1 && w >= is.cum[s + 1]) s++;
  int r = w - is.cum[s];
  Item it;
  it.s = s;
  it.rb = r % is.nrb[s];
  r /= is.nrb[s];
  it.g = r % p.Hkv;
  it.split = r / p.Hkv;
  it.t0 = it.split * p.split_tiles;
  it.t1 = min(it.t0 + p.split_tiles, is.tsh[s]);
  return it;
}

// Bounded wait that also gives up as soon as another role has given up.
__device__ __forceinline__ bool wait_role(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      return false;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(192, 1) attn_split_kernel(const __grid_constant__ TcParams p) {
  using C = Tc<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ ItemSpace is;
  __shared__ int skip;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (sb - raw);
  const uint32_t bars = sb + C::NS * C::STAGE;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + C::NS * C::STAGE + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t SFULL0 = bars + 8u * (2 * C::NS), PFULL0 = bars + 8u * (2 * C::NS + 2);
  const uint32_t ODONE = bars + 8u * (2 * C::NS + 4), QREADY = bars + 8u * (2 * C::NS + 5);
  const uint32_t DRAIN = bars + 8u * (2 * C::NS + 6);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NS; i++) {
      mbar_init(bars + 8u * i, 1);
      mbar_init(bars + 8u * (C::NS + i), 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(SFULL0 + 8u * b, 1);
      mbar_init(PFULL0 + 8u * b, 128);
    }
    mbar_init(ODONE, 1);
    mbar_init(QREADY, 128);
    mbar_init(DRAIN, 1);
    *abort_flag = 0;
    fence_mbar_init();
    skip = status_bad(p.status) ? 1 : 0;
    item_space(p, is);
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

  if (!skip && warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    uint32_t it = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const Item I = item_at(is, p, w);
      for (int t = I.t0; t < I.t1; t++) {
        const int st = it % C::NS;
        if (!wait_role(bars + 8u * (C::NS + st), ((it / C::NS) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t full = bars + 8u * st;
        mbar_arrive_expect_tx(full, C::STAGE);
        const uint32_t kd = sb + st * C::STAGE, vd = kd + C::TILE;
        const int y = I.g * p.cap + t * kTile;
#pragma unroll
        for (int kb = 0; kb < C::KB; kb++) {
          tma_load_2d(kd + kb * kBox, &p.tmK[I.s], full, kb * 64, y);
          tma_load_2d(vd + kb * kBox, &p.tmV[I.s], full, kb * 64, y);
        }
        it++;
      }
    }
    if (!ok) {
      set_status(p.status, TV_ERR_TIMEOUT);
      // let every issued copy land before the CTA's shared memory is released
      for (uint32_t i = it > (uint32_t)C::NS ? it - C::NS : 0; i < it; i++)
        mbar_wait(bars + 8u * (i % C::NS), (i / C::NS) & 1, kWaitCycles);
    }
  } else if (!skip && warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    uint32_t it = 0, sbuf = 0, q_ph = 0, pf_ph[2] = {0u, 0u};
    bool ok = true;
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const Item I = item_at(is, p, w);
      const int n = I.t1 - I.t0;
      if (!wait_role(QREADY, q_ph, abort_flag)) {
        ok = false;
        break;
      }
      q_ph ^= 1;
      tc_fence_after();
      for (int k = 0; k < n; k++) {
        const int st = it % C::NS;
        if (!wait_role(bars + 8u * st, (it / C::NS) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int b = sbuf & 1;
        issue_qk<D>(tbase + C::T_S + b * kTile, tbase + C::T_Q, sb + st * C::STAGE);
        tc_commit(SFULL0 + 8u * b);
        if (k > 0) {
          const int pb = b ^ 1;
          if (!wait_role(PFULL0 + 8u * pb, pf_ph[pb], abort_flag)) {
            ok = false;
            break;
          }
          pf_ph[pb] ^= 1;
          tc_fence_after();
          const int pst = (it - 1) % C::NS;
          issue_pv<D>(tbase + C::T_O, tbase + C::T_S + pb * kTile, sb + pst * C::STAGE + C::TILE, k - 1 > 0);
          tc_commit(bars + 8u * (C::NS + pst));
          tc_commit(ODONE);
        }
        it++;
        sbuf++;
      }
      if (!ok) break;
      const int pb = (sbuf - 1) & 1;
      if (!wait_role(PFULL0 + 8u * pb, pf_ph[pb], abort_flag)) {
        ok = false;
        break;
      }
      pf_ph[pb] ^= 1;
      tc_fence_after();
      const int pst = (it - 1) % C::NS;
      issue_pv<D>(tbase + C::T_O, tbase + C::T_S + pb * kTile, sb + pst * C::STAGE + C::TILE, n - 1 > 0);
      tc_commit(bars + 8u * (C::NS + pst));
      tc_commit(ODONE);
    }
    // every MMA issued by this thread completes before TMEM is released
    tc_commit(DRAIN);
    mbar_wait(DRAIN, 0, kWaitCycles);
    if (!ok) set_status(p.status, TV_ERR_TIMEOUT);
  } else if (!skip && warp >= 2) {
    // ---------------- softmax / epilogue warpgroup ----------------
    const int quad = warp & 3;
    const int lrow = quad * 32 + lane;
    const uint32_t tl = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    uint32_t sbuf = 0, sf_ph[2] = {0u, 0u}, od_ph = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const Item I = item_at(is, p, w);
      const int n = I.t1 - I.t0;
      const int row = I.rb * 128 + lrow;
      const bool valid = row < is.rows[I.s];
      const __nv_bfloat16* qrow = nullptr;
      if (valid) {
        const int node = row / p.G, jh = row % p.G;
        qrow = p.q + (static_cast<size_t>(is.off[I.s] + node) * p.Hq + I.g * p.G + jh) * D;
      }
      load_q_tmem<D>(tl + C::T_Q, qrow);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(QREADY);
      float m = -INFINITY, l = 0.f;
      for (int k = 0; k < n; k++) {
        const int b = sbuf & 1;
        if (!wait_role(SFULL0 + 8u * b, sf_ph[b], abort_flag)) {
          ok = false;
          break;
        }
        sf_ph[b] ^= 1;
        tc_fence_after();
        float sv[kTile];
        tmem_ld64f(tl + C::T_S + b * kTile, sv);
        uint32_t P[kTile / 2];
        float alpha;
        softmax_tile(sv, kTile, p.c, m, l, P, alpha);
        tmem_st32(tl + C::T_S + b * kTile, P);
        if (k > 0) {
          if (!wait_role(ODONE, od_ph, abort_flag)) {
            ok = false;
            break;
          }
          od_ph ^= 1;
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.f)) rescale_o<D>(tl + C::T_O, alpha);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(PFULL0 + 8u * b);
        sbuf++;
      }
      if (!ok) break;
      if (!wait_role(ODONE, od_ph, abort_flag)) {
        ok = false;
        break;
      }
      od_ph ^= 1;
      tc_fence_after();
      store_state<D>(tl + C::T_O, valid ? ws_rec(p, I.s, I.g, I.split, row, D) : nullptr, m, l);
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
template <int D>
__global__ void __launch_bounds__(128, 1) attn_tail_kernel(const __grid_constant__ TcParams p) {
  using C = Tc<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int skip;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (sb - raw);
  const uint32_t BAR = sb + 2 * C::TILE, DRAIN = BAR + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + 2 * C::TILE + 16);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lrow = warp * 32 + lane;
  const int item = blockIdx.x;
  const int g = item % p.Hkv;
  const int node_g = item / p.Hkv;  // global node (verify) or sequence (decode)
  int s = 0, off = 0, depth = 0;
  const int8_t* anc = nullptr;
  if (p.decode) {
    s = node_g;
    off = node_g;
  } else {
    while (s < p.n_seq - 1 && node_g >= p.node_off[s + 1]) s++;
    off = p.node_off[s];
    MetaView mv = meta_view(const_cast<void*>(p.meta), p.n_total);
    depth = mv.depth[node_g];
    anc = mv.anc_at + static_cast<size_t>(node_g) * TV_MAX_PATH;
  }
  const int local = node_g - off;
  const int L = p.len[s];
  if (threadIdx.x == 0) {
    mbar_init(BAR, 1);
    mbar_init(DRAIN, 1);
    fence_mbar_init();
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
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t tl = tbase + (static_cast<uint32_t>(warp * 32) << 16);

  if (!skip) {
    const int P = L + depth + 1;
    const int tsh = L / kTile, tlast = (L + depth) / kTile;
    const int ST = p.split_tiles;
    const bool vrow = lrow < p.G;
    const int row_seq = local * p.G + lrow;
    const int qh = g * p.G + lrow;
    load_q_tmem<D>(tl + C::T_Q, vrow ? p.q + (static_cast<size_t>(node_g) * p.Hq + qh) * D : nullptr);
    float m = -INFINITY, l = 0.f;
    bool fresh = true;
    int cur = tsh / ST;
    if (tsh % ST != 0) {
      // continue the split the split kernel started for this row
      const float* rec = vrow ? ws_rec(p, s, g, cur, row_seq, D) : nullptr;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t r[32];
        if (rec) {
          const uint4* s4 = reinterpret_cast<const uint4*>(rec + c0);
#pragma unroll
          for (int i = 0; i < 8; i++) {
            const uint4 v = s4[i];
            r[4 * i] = v.x;
            r[4 * i + 1] = v.y;
            r[4 * i + 2] = v.z;
            r[4 * i + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; i++) r[i] = 0u;
        }
        tmem_st32(tl + C::T_O + c0, r);
      }
      if (rec) {
        m = rec[D];
        l = rec[D + 1];
      }
      fresh = false;
    }
    tmem_st_wait();
    uint32_t ph = 0;
    bool ok = true;
    for (int t = tsh; t <= tlast && ok; t++) {
      if (t / ST != cur) {
        store_state<D>(tl + C::T_O, vrow ? ws_rec(p, s, g, cur, row_seq, D) : nullptr, m, l);
        cur = t / ST;
        fresh = true;
        m = -INFINITY;
        l = 0.f;
      }
      // build the node's K/V tile: cache rows below L, ancestors at L..L+d, zeros after
      for (int idx = threadIdx.x; idx < kTile * (D / 8); idx += blockDim.x) {
        const int j = idx / (D / 8), cc = idx % (D / 8), pos = t * kTile + j;
        uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
        if (pos < L) {
          const size_t r = (static_cast<size_t>(g) * p.cap + pos) * D;
          kv = reinterpret_cast<const uint4*>(p.K[s] + r)[cc];
          vv = reinterpret_cast<const uint4*>(p.V[s] + r)[cc];
        } else if (pos < P) {
          const int tn = p.decode ? node_g : off + anc[pos - L];
          const size_t r = (static_cast<size_t>(tn) * p.Hkv + g) * D;
          kv = reinterpret_cast<const uint4*>(p.kt + r)[cc];
          vv = reinterpret_cast<const uint4*>(p.vt + r)[cc];
        }
        const int kb = cc >> 3, c = cc & 7;
        const uint32_t o = kb * kBox + (j >> 3) * 1024 + (j & 7) * 128 + ((c ^ (j & 7)) << 4);
        *reinterpret_cast<uint4*>(gb + o) = kv;
        *reinterpret_cast<uint4*>(gb + C::TILE + o) = vv;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (threadIdx.x == 0) {
        issue_qk<D>(tbase + C::T_S, tbase + C::T_Q, sb);
        tc_commit(BAR);
      }
      if (!mbar_wait(BAR, ph, kWaitCycles)) {
        ok = false;
        break;
      }
      ph ^= 1;
      tc_fence_after();
      float sv[kTile];
      tmem_ld64f(tl + C::T_S, sv);
      uint32_t Pw[kTile / 2];
      float alpha;
      softmax_tile(sv, min(kTile, P - t * kTile), p.c, m, l, Pw, alpha);
      tmem_st32(tl + C::T_S, Pw);
      if (!fresh && __any_sync(0xffffffffu, alpha != 1.f)) rescale_o<D>(tl + C::T_O, alpha);
      tmem_st_wait();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (threadIdx.x == 0) {
        issue_pv<D>(tbase + C::T_O, tbase + C::T_S, sb + C::TILE, !fresh);
        tc_commit(BAR);
      }
      if (!mbar_wait(BAR, ph, kWaitCycles)) {
        ok = false;
        break;
      }
      ph ^= 1;
      tc_fence_after();
      fresh = false;
      __syncthreads();
    }
    if (!ok) {
      set_status(p.status, TV_ERR_TIMEOUT);
    } else {
      store_state<D>(tl + C::T_O, vrow ? ws_rec(p, s, g, cur, row_seq, D) : nullptr, m, l);
      __syncthreads();
      // merge splits 0..cur in split order
      const int ns = cur + 1;
      const size_t sstride = static_cast<size_t>(p.rows_max) * (D + 4);
      for (int idx = threadIdx.x; idx < p.G * (D / 4); idx += blockDim.x) {
        const int r = idx / (D / 4), c4 = idx % (D / 4);
        const float* rec0 = ws_rec(p, s, g, 0, local * p.G + r, D);
        float mm = -INFINITY;
        for (int sp = 0; sp < ns; sp++) mm = fmaxf(mm, rec0[sp * sstride + D]);
        float ls = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 0; sp < ns; sp++) {
          const float* rec = rec0 + sp * sstride;
          const float ms = rec[D];
          const float wgt = (ms == mm) ? 1.f : ex2_approx(__fsub_rn(ms, mm));
          ls = __fmaf_rn(wgt, rec[D + 1], ls);
          const float4 v = reinterpret_cast<const float4*>(rec)[c4];
          o.x = __fmaf_rn(wgt, v.x, o.x);
          o.y = __fmaf_rn(wgt, v.y, o.y);
          o.z = __fmaf_rn(wgt, v.z, o.z);
          o.w = __fmaf_rn(wgt, v.w, o.w);
        }
        uint2 packed;
        packed.x = pack_bf16x2(__fdiv_rn(o.x, ls), __fdiv_rn(o.y, ls));
        packed.y = pack_bf16x2(__fdiv_rn(o.z, ls), __fdiv_rn(o.w, ls));
        *reinterpret_cast<uint2*>(p.out + (static_cast<size_t>(node_g) * p.Hq + g * p.G + r) * D + 4 * c4) = packed;
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

template <int D>
static tv_status launch_tc(const TcParams& p, int n_items_bound, int n_tail, cudaStream_t st) {
  using C = Tc<D>;
  // one-time attribute setup (never inside a stream capture after the first call)
  static bool attrs = false;
  if (!attrs) {
    if (cudaFuncSetAttribute(attn_split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_SPLIT) !=
            cudaSuccess ||
        cudaFuncSetAttribute(attn_tail_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_TAIL) !=
            cudaSuccess)
      return TV_ERR_CUDA;
    attrs = true;
  }
  if (n_items_bound > 0) {
    const int grid = n_items_bound < num_sms() ? n_items_bound : num_sms();
    attn_split_kernel<D><<<grid, 192, C::SMEM_SPLIT, st>>>(p);
  }
  attn_tail_kernel<D><<<n_tail, 128, C::SMEM_TAIL, st>>>(p);
  return launch_status();
}

tv_status attn_tc_launch(const tv_plan* plan, const AttnCall& a, void* ws, size_t ws_bytes, cudaStream_t st) {
  const tv_attn_layer* l = a.layer;
  if (!plan || plan->split < kTile || plan->split % kTile) return TV_ERR_ARG;
  const int G = l->Hq / l->Hkv;
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
  const int items_bound = a.n_seq * l->Hkv * splits_bound * ((n_max * G + 127) / 128);
  const int n_tail = (a.decode ? a.n_seq : a.n_total) * l->Hkv;
  switch (l->D) {
    case 64: return launch_tc<64>(p, items_bound, n_tail, st);
    case 128: return launch_tc<128>(p, items_bound, n_tail, st);
    case 256: return launch_tc<256>(p, items_bound, n_tail, st);
    default: return TV_ERR_SHAPE;
  }
}

}  // namespace tv
