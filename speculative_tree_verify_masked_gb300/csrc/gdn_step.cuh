// One token of the gated delta rule for one row of a Gated DeltaNet state,
// shared by tree verify, single-token decode and commit so that all three
// produce the same bits (the row-invariance rule of "Adding a model", step 4).
//
// State row r of value head h is s = S[h][r][:] (dk floats).  With
// x = s . k and y = s . q, one token is
//     c  = beta * (v_r - alpha * x)
//     s' = alpha * s + c * k          (= alpha s (I - beta k k^T) + beta v_r k^T)
//     o  = scale * (alpha * y + c * (k . q))   (= scale * s' . q)
// A row is spread over LPR = dk / 16 lanes (a lane group), 16 elements each,
// held as kPairs = 8 packed fp32 pairs: chunk c (pairs 4c .. 4c+3) of lane j
// covers columns (c * LPR + j) * 8 .. +7, so a lane group reads LPR * 32
// contiguous bytes of an fp32 row per chunk, and one 16-byte load brings a
// lane a whole chunk of a bf16 key or query.
//
// The arithmetic uses the packed fp32x2 FMA / MUL / ADD instructions (two
// independent IEEE round-to-nearest operations each); every operation is
// explicit and in a fixed order.  A lane's partial dot product runs four
// accumulators over its pairs (pair e into accumulator e % 4), adds them as
// (a0 + a1) + (a2 + a3) and then the two halves of the pair; the group sum
// is a butterfly over the group's lanes, lane distance LPR/2 first, then
// halving.  Pairwise sums are commutative, so every lane of the group gets
// the same bits.
#pragma once
#include "common.cuh"

namespace tv {

constexpr int kPairs = 8;            // packed pairs of a row per lane (16 elements)
constexpr int kChunks = kPairs / 4;  // chunks of 8 columns of a row per lane

template <int LPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int o = LPR / 2; o >= 1; o >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o, LPR));
  return x;
}

// This lane's pairs of a dk-long fp32 row (global or shared memory).
template <int LPR>
__device__ __forceinline__ void load_row(f2_t (&d)[kPairs], const float* src, int j) {
#pragma unroll
  for (int c = 0; c < kChunks; c++) {
    const ulonglong2* p = reinterpret_cast<const ulonglong2*>(src + (c * LPR + j) * 8);
    const ulonglong2 v0 = p[0], v1 = p[1];
    d[4 * c] = v0.x;
    d[4 * c + 1] = v0.y;
    d[4 * c + 2] = v1.x;
    d[4 * c + 3] = v1.y;
  }
}
template <int LPR>
__device__ __forceinline__ void store_row(float* dst, const f2_t (&s)[kPairs], int j) {
#pragma unroll
  for (int c = 0; c < kChunks; c++) {
    ulonglong2* p = reinterpret_cast<ulonglong2*>(dst + (c * LPR + j) * 8);
    p[0] = make_ulonglong2(s[4 * c], s[4 * c + 1]);
    p[1] = make_ulonglong2(s[4 * c + 2], s[4 * c + 3]);
  }
}

// Two bf16 (low half first) as a packed fp32 pair, exactly.
__device__ __forceinline__ f2_t f2_from_bf16x2(uint32_t w) {
  return (static_cast<f2_t>(w & 0xffff0000u) << 32) | static_cast<f2_t>(w << 16);
}
// This lane's pairs of a dk-long row stored as bf16 (same columns as load_row).
template <int LPR>
__device__ __forceinline__ void load_row_bf16(f2_t (&d)[kPairs], const __nv_bfloat16* src, int j) {
#pragma unroll
  for (int c = 0; c < kChunks; c++) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + (c * LPR + j) * 8);
    d[4 * c] = f2_from_bf16x2(v.x);
    d[4 * c + 1] = f2_from_bf16x2(v.y);
    d[4 * c + 2] = f2_from_bf16x2(v.z);
    d[4 * c + 3] = f2_from_bf16x2(v.w);
  }
}
template <int LPR>
__device__ __forceinline__ void load_row_any(f2_t (&d)[kPairs], const float* src, int j) {
  load_row<LPR>(d, src, j);
}
template <int LPR>
__device__ __forceinline__ void load_row_any(f2_t (&d)[kPairs], const __nv_bfloat16* src, int j) {
  load_row_bf16<LPR>(d, src, j);
}

// This lane's partial of s . w.
__device__ __forceinline__ float row_partial(const f2_t (&s)[kPairs], const f2_t (&w)[kPairs]) {
  f2_t a0 = 0ull, a1 = 0ull, a2 = 0ull, a3 = 0ull;  // (+0.0f, +0.0f)
#pragma unroll
  for (int e = 0; e < kPairs; e += 4) {
    a0 = f2_fma(s[e], w[e], a0);
    a1 = f2_fma(s[e + 1], w[e + 1], a1);
    a2 = f2_fma(s[e + 2], w[e + 2], a2);
    a3 = f2_fma(s[e + 3], w[e + 3], a3);
  }
  return f2_hsum(f2_add(f2_add(a0, a1), f2_add(a2, a3)));
}

template <int LPR>
__device__ __forceinline__ float row_dot(const f2_t (&s)[kPairs], const f2_t (&w)[kPairs]) {
  return group_sum<LPR>(row_partial(s, w));
}

// The pieces of one step after the dot products, shared by every caller.
__device__ __forceinline__ float gdn_c(float x, float v, float alpha, float beta) {
  return __fmul_rn(beta, __fsub_rn(v, __fmul_rn(alpha, x)));
}
__device__ __forceinline__ float gdn_o(float c, float kq, float alpha, float y, float scale) {
  return __fmul_rn(scale, __fmaf_rn(c, kq, __fmul_rn(alpha, y)));
}
__device__ __forceinline__ void gdn_update(f2_t (&s)[kPairs], const f2_t (&k)[kPairs], float alpha, float c) {
  const f2_t a2 = f2_dup(alpha), c2 = f2_dup(c);
#pragma unroll
  for (int e = 0; e < kPairs; e++) s[e] = f2_fma(c2, k[e], f2_mul(a2, s[e]));
}

// Group sums of N values, their butterflies interleaved level by level
// (each sum formed exactly as group_sum forms it).
template <int LPR, int N>
__device__ __forceinline__ void group_sum_n(float (&x)[N]) {
#pragma unroll
  for (int o = LPR / 2; o >= 1; o >>= 1) {
    float t[N];
#pragma unroll
    for (int i = 0; i < N; i++) t[i] = __shfl_xor_sync(0xffffffffu, x[i], o, LPR);
#pragma unroll
    for (int i = 0; i < N; i++) x[i] = __fadd_rn(x[i], t[i]);
  }
}

// One token for one state row, with this lane's pairs of the token's key k
// and query q already in registers and kq = k . q (from kq_group).  Returns
// o when WITH_OUT; advances s when `update`.  Both dot products are formed
// before either butterfly.
template <int LPR, bool WITH_OUT>
__device__ __forceinline__ float gdn_row_step(f2_t (&s)[kPairs], const f2_t (&k)[kPairs], const f2_t (&q)[kPairs],
                                              float kq, float v, float alpha, float beta, float scale, bool update) {
  float x = row_partial(s, k);
  float y = 0.f;
  if (WITH_OUT) {
    float xy[2] = {x, row_partial(s, q)};
    group_sum_n<LPR, 2>(xy);
    x = xy[0];
    y = xy[1];
  } else {
    x = group_sum<LPR>(x);
  }
  const float c = gdn_c(x, v, alpha, beta);
  float o = 0.f;
  if (WITH_OUT) o = gdn_o(c, kq, alpha, y, scale);
  if (update) gdn_update(s, k, alpha, c);
  return o;
}

// k . q of one token, by one lane group with the row layout (the same
// reduction as a row dot), so every caller gets the same bits.
template <int LPR>
__device__ __forceinline__ float kq_group(const f2_t (&k)[kPairs], const f2_t (&q)[kPairs]) {
  return row_dot<LPR>(k, q);
}

// Lanes per row for a key dimension (dk = 64 or 128): 4 or 8.
template <int DK>
__host__ __device__ constexpr int lanes_per_row() {
  return DK / (2 * kPairs);
}

}  // namespace tv
