// Per-channel pieces of the Gated DeltaNet front end ("Adding a model", "What
// is still specific to Qwen3.8": the Gated DeltaNet layer with its gated
// norm; "The model layer": the per-sequence convolution tails), shared by
// tv_gdn_front and the front-end stage of the fused tree verify, so both form
// every value with the same operations in the same order.
#pragma once
#include "common.cuh"

namespace tv {

constexpr float kNormEps = 1e-6f;
constexpr int kMaxConvWidth = 8;

// SiLU as x / (1 + e^-x) with CUDA's fast exponential and divide (__expf,
// __fdividef: a few ulp, far below the bf16 rounding that follows); every
// path of the library forms it with this one function.  For x below -88 the
// exponential is infinite and the quotient 0, SiLU's limit.
__device__ __forceinline__ float silu_f(float x) { return __fdividef(x, __fadd_rn(1.f, __expf(-x))); }

// Gates from the raw values: alpha = exp(-softplus(a)), beta = sigmoid(b).
__device__ __forceinline__ void front_gates(float a, float b, float& alpha, float& beta) {
  const float sp = a > 20.f ? a : log1pf(expf(a));
  alpha = expf(-sp);
  beta = __fdiv_rn(1.f, __fadd_rn(1.f, expf(-b)));
}

// The rows of the convolution window of a token at `depth` on its root path:
// window element j reads the ancestor at depth depth + j - (W-1) (global
// row off + anc[m]; a decoded token, anc null, is its own row `self`), or
// tail row depth + j while that depth is negative (encoded -1 - r).
__device__ __forceinline__ void conv_window(int (&src)[kMaxConvWidth], int W, int depth, int off, const int8_t* anc,
                                            int self) {
#pragma unroll
  for (int j = 0; j < kMaxConvWidth; j++) {
    if (j < W) {
      const int m = depth + j - (W - 1);
      src[j] = m >= 0 ? (anc ? off + anc[m] : self) : -1 - (depth + j);
    }
  }
}

// Short convolution of channel c over the window (taps in order), then SiLU.
template <typename T>
__device__ __forceinline__ float conv_silu(const T* x, const T* tail, const float* wconv, int C, int W,
                                           const int (&src)[kMaxConvWidth], int c) {
  float acc = 0.f;
  for (int j = 0; j < W; j++) {
    const float xin = src[j] >= 0 ? to_f32(x[static_cast<size_t>(src[j]) * C + c])
                                  : to_f32(tail[static_cast<size_t>(-1 - src[j]) * C + c]);
    acc = __fmaf_rn(wconv[static_cast<size_t>(c) * W + j], xin, acc);
  }
  return silu_f(acc);
}

// 1 / sqrt(sum of squares + eps) of NH heads held by one warp, CPL
// channels a lane (lane + 32e): each lane's sum in e order, then a
// butterfly; the heads' chains interleave, each formed exactly as alone.
template <int CPL, int NH>
__device__ __forceinline__ void warp_l2_scales(const float (&val)[NH][CPL], float (&sc)[NH]) {
  float ss[NH];
#pragma unroll
  for (int i = 0; i < NH; i++) {
    ss[i] = 0.f;
#pragma unroll
    for (int e = 0; e < CPL; e++) ss[i] = __fmaf_rn(val[i][e], val[i][e], ss[i]);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
    for (int i = 0; i < NH; i++) ss[i] = __fadd_rn(ss[i], __shfl_xor_sync(0xffffffffu, ss[i], o));
#pragma unroll
  for (int i = 0; i < NH; i++) sc[i] = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(ss[i], kNormEps)));
}
template <int CPL>
__device__ __forceinline__ float warp_l2_scale(const float (&val)[CPL]) {
  float sc[1];
  warp_l2_scales<CPL, 1>(reinterpret_cast<const float(&)[1][CPL]>(val), sc);
  return sc[0];
}

// Gated RMS norm of one (row, value head) of DV = 32 CPL channels held by a
// warp (lane + 32e; o already rounded to the layer type, z widened from it):
// out = o / sqrt(mean(o^2) + eps) * w_norm * SiLU(z); the sum of squares per
// lane in e order, then a butterfly.  tv_gdn_out_norm and the fused verify
// both form it here.
template <typename T, int CPL>
__device__ __forceinline__ void gated_norm_vals(const float (&ov)[CPL], const float (&zv)[CPL],
                                                const float (&wn)[CPL], T* out, int lane) {
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < CPL; e++) ss = __fmaf_rn(ov[e], ov[e], ss);
#pragma unroll
  for (int sh = 16; sh >= 1; sh >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, sh));
  const float inv = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(32 * CPL)), kNormEps)));
#pragma unroll
  for (int e = 0; e < CPL; e++) {
    const float y = __fmul_rn(__fmul_rn(__fmul_rn(ov[e], inv), wn[e]), silu_f(zv[e]));
    out[lane + 32 * e] = from_f32<T>(y);
  }
}

}  // namespace tv
