// One token of the gated delta rule for one row of a Gated DeltaNet state,
// shared by tree verify, single-token decode and commit so that all three
// produce the same bits (the row-invariance rule of "Adding a model", step 4).
//
// State row r of value head h is s = S[h][r][:] (dk floats).  With
// x = s . k and y = s . q, one token is
//     c  = beta * (v_r - alpha * x)
//     s' = alpha * s + c * k          (= alpha s (I - beta k k^T) + beta v_r k^T)
//     o  = scale * (alpha * y + c * (k . q))   (= scale * s' . q)
// A row is spread over LPR lanes, 16 elements each: element e of lane j is
// column ((e / 4) * LPR + j) * 4 + (e % 4), so a lane group reads whole
// 16-byte chunks of the row.  Every operation is an explicit IEEE op in a
// fixed order (no contraction left to the compiler), and the lane reduction
// is a butterfly whose pairwise sums are commutative, so all lanes of a group
// hold the same bits.
#pragma once
#include "common.cuh"

namespace tv {

template <int LPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int o = 1; o < LPR; o <<= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o, LPR));
  return x;
}

template <int LPR>
__device__ __forceinline__ void load_row16(float (&d)[16], const float* src, int j) {
  const float4* p = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int c = 0; c < 4; c++) {
    const float4 v = p[c * LPR + j];
    d[4 * c + 0] = v.x;
    d[4 * c + 1] = v.y;
    d[4 * c + 2] = v.z;
    d[4 * c + 3] = v.w;
  }
}

template <int LPR>
__device__ __forceinline__ void store_row16(float* dst, const float (&s)[16], int j) {
  float4* p = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int c = 0; c < 4; c++) p[c * LPR + j] = make_float4(s[4 * c], s[4 * c + 1], s[4 * c + 2], s[4 * c + 3]);
}

// k . q for one token, sequential fused multiply-adds from zero.
__device__ __forceinline__ float dot_seq(const float* a, const float* b, int n) {
  float acc = 0.f;
  for (int i = 0; i < n; i++) acc = __fmaf_rn(a[i], b[i], acc);
  return acc;
}

template <int LPR>
__device__ __forceinline__ float row_dot(const float (&s)[16], const float (&w)[16]) {
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int e = 0; e < 8; e++) a0 = __fmaf_rn(s[e], w[e], a0);
#pragma unroll
  for (int e = 8; e < 16; e++) a1 = __fmaf_rn(s[e], w[e], a1);
  return group_sum<LPR>(__fadd_rn(a0, a1));
}

// kv, qv: the token's key and query (fp32, dk values) in shared memory.
// Returns o when WITH_OUT; advances s when `update`.
template <int LPR, bool WITH_OUT>
__device__ __forceinline__ float gdn_row_step(float (&s)[16], const float* kv, const float* qv, int j, float kq,
                                              float v, float alpha, float beta, float scale, bool update) {
  float k[16];
  load_row16<LPR>(k, kv, j);
  const float x = row_dot<LPR>(s, k);
  float y = 0.f;
  if (WITH_OUT) {
    float q[16];
    load_row16<LPR>(q, qv, j);
    y = row_dot<LPR>(s, q);
  }
  const float c = __fmul_rn(beta, __fsub_rn(v, __fmul_rn(alpha, x)));
  float o = 0.f;
  if (WITH_OUT) o = __fmul_rn(scale, __fmaf_rn(c, kq, __fmul_rn(alpha, y)));
  if (update) {
#pragma unroll
    for (int e = 0; e < 16; e++) s[e] = __fmaf_rn(c, k[e], __fmul_rn(alpha, s[e]));
  }
  return o;
}

}  // namespace tv
