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
// explicit and in a fixed order, and the lane reduction is a butterfly whose
// pairwise sums are commutative, so all lanes of a group hold the same bits.
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
  for (int o = 1; o < LPR; o <<= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o, LPR));
  return x;
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

template <int LPR>
__device__ __forceinline__ float row_dot(const f2_t (&s)[8], const f2_t (&w)[8]) {
  f2_t acc = 0ull;  // (+0.0f, +0.0f)
#pragma unroll
  for (int e = 0; e < 8; e++) acc = f2_fma(s[e], w[e], acc);
  return group_sum<LPR>(f2_hsum(acc));
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
  const float c = __fmul_rn(beta, __fsub_rn(v, __fmul_rn(alpha, x)));
  float o = 0.f;
  if (WITH_OUT) o = __fmul_rn(scale, __fmaf_rn(c, kq, __fmul_rn(alpha, y)));
  if (update) {
    const f2_t a2 = f2_dup(alpha), c2 = f2_dup(c);
#pragma unroll
    for (int e = 0; e < 8; e++) s[e] = f2_fma(c2, k[e], f2_mul(a2, s[e]));
  }
  return o;
}

// k . q of one token, by one lane group with the row layout (the same
// reduction as a row dot), so every caller gets the same bits.
template <int LPR>
__device__ __forceinline__ float kq_group(const f2_t (&k)[8], const f2_t (&q)[8]) {
  return row_dot<LPR>(k, q);
}

}  // namespace tv
