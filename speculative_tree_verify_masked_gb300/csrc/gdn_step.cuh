// One token of the gated delta rule for one row of a Gated DeltaNet state,
// shared by tree verify, single-token decode and commit so that all three
// produce the same bits (the row-invariance rule of "Adding a model", step 4).
//
// State row r of value head h is s = S[h][r][:] (dk floats).  With
// x = s . k and y = s . q, one token is
//     c  = beta * (v_r - alpha * x)
//     s' = alpha * s + c * k          (= alpha s (I - beta k k^T) + beta v_r k^T)
//     o  = scale * (alpha * y + c * (k . q))   (= scale * s' . q)
// A row is spread over LPR lanes, 16 elements each, held as 8 packed fp32
// pairs: pair e of lane j covers columns ((e / 2) * LPR + j) * 4 + 2 (e % 2)
// and the next one, so a lane group reads whole 16-byte chunks of the row.
// The arithmetic uses the packed fp32x2 FMA / MUL instructions (two
// independent IEEE round-to-nearest operations each); every operation is
// explicit and in a fixed order.  A dot product is each lane's partial sum
// followed by a butterfly over the group's lanes, lane distance LPR/2 first,
// then halving; pairwise sums are commutative, so every lane of the group
// gets the same bits.  reduce_scatter forms the same sums for several values
// at once (each lane ends up with its share of the results) with one eighth
// of the shuffles, and gives the same bits as eight separate butterflies.
#pragma once
#include "common.cuh"

namespace tv {

typedef unsigned long long f2_t;  // two fp32 values in one 64-bit register

__device__ __forceinline__ f2_t f2_fma(f2_t a, f2_t b, f2_t c) {
  f2_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2_t f2_mul(f2_t a, f2_t b) {
  f2_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_dup(float x) {
  f2_t d;
  asm("mov.b64 %0, {%1, %1};" : "=l"(d) : "f"(x));
  return d;
}
__device__ __forceinline__ float f2_hsum(f2_t a) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a));
  return __fadd_rn(lo, hi);
}

template <int LPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int o = LPR / 2; o >= 1; o >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o, LPR));
  return x;
}

// Group sums of NV values v[0..NV) (each a per-lane partial), NV a power of
// two.  At lane distance o, while a lane still holds more than one value, the
// lanes with bit o set keep the upper half of their current values and the
// others the lower half, each adding its partner's partial of the kept
// values; once one value is left the step is a plain butterfly add.  Every
// sum is formed exactly as group_sum forms it.  Afterwards lane j holds
// rs_count<LPR, NV>() sums in v[0 ..): values j * (NV / LPR) + i when
// NV >= LPR, else value j >> log2(LPR / NV).
template <int LPR, int NV>
__device__ __forceinline__ void reduce_scatter(float (&v)[NV], int j) {
  int cnt = NV;
#pragma unroll
  for (int o = LPR / 2; o >= 1; o >>= 1) {
    if (cnt > 1) {
      const int half = cnt / 2;
      const bool up = (j & o) != 0;
#pragma unroll
      for (int m = 0; m < NV / 2; m++) {
        if (m < half) {
          const float send = up ? v[m] : v[m + half];
          const float keep = up ? v[m + half] : v[m];
          v[m] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, o, LPR));
        }
      }
      cnt = half;
    } else {
      v[0] = __fadd_rn(v[0], __shfl_xor_sync(0xffffffffu, v[0], o, LPR));
    }
  }
}
template <int LPR, int NV>
__device__ __forceinline__ constexpr int rs_count() {
  return NV >= LPR ? NV / LPR : 1;
}
// Lane (within the group) that holds value m after reduce_scatter, and the
// index of that value in its v[].
template <int LPR, int NV>
__device__ __forceinline__ int rs_lane(int m) {
  if constexpr (NV >= LPR) return m / (NV / LPR);
  else return m * (LPR / NV);
}
template <int LPR, int NV>
__device__ __forceinline__ int rs_index(int m) {
  if constexpr (NV >= LPR) return m % (NV / LPR);
  else return 0;
}
// Value held in v[i] by lane j after reduce_scatter, and whether lane j is
// the first of the lanes that hold it.
template <int LPR, int NV>
__device__ __forceinline__ int rs_value(int j, int i) {
  if constexpr (NV >= LPR) return j * (NV / LPR) + i;
  else return j / (LPR / NV);
}
template <int LPR, int NV>
__device__ __forceinline__ bool rs_first(int j) {
  if constexpr (NV >= LPR) return true;
  else return (j % (LPR / NV)) == 0;
}

// This lane's 8 pairs of a dk-long fp32 row (global or shared memory).
template <int LPR>
__device__ __forceinline__ void load_row8(f2_t (&d)[8], const float* src, int j) {
  const ulonglong2* p = reinterpret_cast<const ulonglong2*>(src);
#pragma unroll
  for (int c = 0; c < 4; c++) {
    const ulonglong2 v = p[c * LPR + j];
    d[2 * c] = v.x;
    d[2 * c + 1] = v.y;
  }
}
template <int LPR>
__device__ __forceinline__ void store_row8(float* dst, const f2_t (&s)[8], int j) {
  ulonglong2* p = reinterpret_cast<ulonglong2*>(dst);
#pragma unroll
  for (int c = 0; c < 4; c++) p[c * LPR + j] = make_ulonglong2(s[2 * c], s[2 * c + 1]);
}

// This lane's partial of s . w.
__device__ __forceinline__ float row_partial(const f2_t (&s)[8], const f2_t (&w)[8]) {
  f2_t acc = 0ull;  // (+0.0f, +0.0f)
#pragma unroll
  for (int e = 0; e < 8; e++) acc = f2_fma(s[e], w[e], acc);
  return f2_hsum(acc);
}

template <int LPR>
__device__ __forceinline__ float row_dot(const f2_t (&s)[8], const f2_t (&w)[8]) {
  return group_sum<LPR>(row_partial(s, w));
}

// The pieces of one step after the dot products, shared by every caller.
__device__ __forceinline__ float gdn_c(float x, float v, float alpha, float beta) {
  return __fmul_rn(beta, __fsub_rn(v, __fmul_rn(alpha, x)));
}
__device__ __forceinline__ float gdn_o(float c, float kq, float alpha, float y, float scale) {
  return __fmul_rn(scale, __fmaf_rn(c, kq, __fmul_rn(alpha, y)));
}
__device__ __forceinline__ void gdn_update(f2_t (&s)[8], const f2_t (&k)[8], float alpha, float c) {
  const f2_t a2 = f2_dup(alpha), c2 = f2_dup(c);
#pragma unroll
  for (int e = 0; e < 8; e++) s[e] = f2_fma(c2, k[e], f2_mul(a2, s[e]));
}

// Two bf16 (low half first) as a packed fp32 pair, exactly.
__device__ __forceinline__ f2_t f2_from_bf16x2(uint32_t w) {
  return (static_cast<f2_t>(w & 0xffff0000u) << 32) | static_cast<f2_t>(w << 16);
}
// This lane's 8 pairs of a dk-long row stored as bf16 (same columns as load_row8).
template <int LPR>
__device__ __forceinline__ void load_row8_bf16(f2_t (&d)[8], const __nv_bfloat16* src, int j) {
  const uint2* p = reinterpret_cast<const uint2*>(src);
#pragma unroll
  for (int c = 0; c < 4; c++) {
    const uint2 v = p[c * LPR + j];
    d[2 * c] = f2_from_bf16x2(v.x);
    d[2 * c + 1] = f2_from_bf16x2(v.y);
  }
}
template <int LPR>
__device__ __forceinline__ void load_row8_any(f2_t (&d)[8], const float* src, int j) {
  load_row8<LPR>(d, src, j);
}
template <int LPR>
__device__ __forceinline__ void load_row8_any(f2_t (&d)[8], const __nv_bfloat16* src, int j) {
  load_row8_bf16<LPR>(d, src, j);
}

// One token for one state row, with this lane's pairs of the token's key k
// and query q already in registers and kq = k . q (from kq_group).  Returns
// o when WITH_OUT; advances s when `update`.
template <int LPR, bool WITH_OUT>
__device__ __forceinline__ float gdn_row_step(f2_t (&s)[8], const f2_t (&k)[8], const f2_t (&q)[8], float kq, float v,
                                              float alpha, float beta, float scale, bool update) {
  const float x = row_dot<LPR>(s, k);
  float y = 0.f;
  if (WITH_OUT) y = row_dot<LPR>(s, q);
  const float c = gdn_c(x, v, alpha, beta);
  float o = 0.f;
  if (WITH_OUT) o = gdn_o(c, kq, alpha, y, scale);
  if (update) gdn_update(s, k, alpha, c);
  return o;
}

// k . q of one token, by one lane group with the row layout (the same
// reduction as a row dot), so every caller gets the same bits.
template <int LPR>
__device__ __forceinline__ float kq_group(const f2_t (&k)[8], const f2_t (&q)[8]) {
  return row_dot<LPR>(k, q);
}

}  // namespace tv
