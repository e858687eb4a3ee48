// frontend.cuh -- the single-precision arithmetic of the layer's front end.
//
// With bf16 activations the short convolution and the L2 norm end in a
// rounding to bf16, i.e. in a decision: a value near a bf16 rounding boundary
// goes one way or the other depending on the last bits of the fp32 result.
// Every kernel therefore evaluates the front end in one fixed order, each
// step rounded once:
//   conv:  y = w0 x_{t-3}, then y = fma(w_j, x_j, y) for the later taps
//          x_{t-2}, x_{t-1}, x_t (exact product and sum, one rounding)
//   norm:  s = sum of y_i^2 over the row by pairwise summation (the row split
//          in halves, recursively: adjacent pairs first), every square and
//          sum rounded on its own, r = 1 / sqrt(s + 1e-6), each element
//          scaled by r
// so that the same inputs give the same bf16 activations in every kernel:
// prefill, decode and speculative decode agree bit for bit on them.  A
// product that must round before a sum is never left for the compiler to
// fuse: sums after products are scalar __fadd_rn.  The two-lane forms
// (mul / add / fma on fp32 pairs) are used for the conv, whose sums are
// explicit fused multiply-adds, and for products not followed by a sum; a
// two-lane product followed by a two-lane sum was fused into one rounding
// even when written with the _rn intrinsics, which moved about one activation
// in 30,000 by a bf16 step.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace glinattn {
namespace fe {

// one output of the width-4 causal convolution, oldest tap first, every later
// tap added by one fused multiply-add
__device__ __forceinline__ float conv4(float w0, float w1, float w2, float w3, float x0, float x1, float x2,
                                       float x3) {
  float acc = __fmul_rn(w0, x0);
  acc = __fmaf_rn(w1, x1, acc);
  acc = __fmaf_rn(w2, x2, acc);
  return __fmaf_rn(w3, x3, acc);
}

// sum over the 32 lanes, adjacent lanes first (xor 1, 2, 4, 8, 16): the
// pairwise sum of 32 consecutive elements held one per lane; every lane gets it
__device__ __forceinline__ float warp_pairwise_sum(float x) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// pairwise sum of n (a power of two) consecutive partial sums
template <int N>
__device__ __forceinline__ float pairwise_sum(const float *s) {
  if constexpr (N == 1) {
    return s[0];
  } else {
    return __fadd_rn(pairwise_sum<N / 2>(s), pairwise_sum<N / 2>(s + N / 2));
  }
}

// the inverse norm of a row whose sum of squares is s
__device__ __forceinline__ float inv_norm(float s) { return __frcp_rn(__fsqrt_rn(__fadd_rn(s, 1e-6f))); }

// ---- two channels at once: the conv of a pair of channels
__device__ __forceinline__ float2 conv4x2(float2 w0, float2 w1, float2 w2, float2 w3, float2 x0, float2 x1, float2 x2,
                                          float2 x3) {
  float2 acc = __fmul2_rn(w0, x0);
  acc = __ffma2_rn(w1, x1, acc);
  acc = __ffma2_rn(w2, x2, acc);
  return __ffma2_rn(w3, x3, acc);
}
// two bf16x2 words a, b as fp32 pairs: their low halves (a.lo, b.lo) and their
// high halves (a.hi, b.hi)
__device__ __forceinline__ float2 bf16_lows(uint32_t a, uint32_t b) {
  return make_float2(__uint_as_float(a << 16), __uint_as_float(b << 16));
}
__device__ __forceinline__ float2 bf16_highs(uint32_t a, uint32_t b) {
  return make_float2(__uint_as_float(a & 0xffff0000u), __uint_as_float(b & 0xffff0000u));
}

// Pairwise row sums of 8 rows at once: s[r] is this lane's partial of row r;
// the lanes reduce as warp_pairwise_sum does (xor 1, 2, 4, 8, 16, the same
// additions in the same tree) but halve the rows they carry at each of the
// first three levels.  Returns the full sum of row 4 (l & 1) + 2 ((l >> 1) & 1)
// + ((l >> 2) & 1) in lane l; row_lane(r) names a lane holding row r.
__device__ __forceinline__ float warp_pairwise_sum8(const float (&s)[8], int lane) {
  const bool b0 = lane & 1, b1 = lane & 2, b2 = lane & 4;
  float t1[4], t2[2];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float keep = b0 ? s[k + 4] : s[k], send = b0 ? s[k] : s[k + 4];
    t1[k] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 1));
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float keep = b1 ? t1[k + 2] : t1[k], send = b1 ? t1[k] : t1[k + 2];
    t2[k] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  }
  const float keep = b2 ? t2[1] : t2[0], send = b2 ? t2[0] : t2[1];
  float t = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, 8));
  return __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, 16));
}
__device__ __forceinline__ constexpr int row_lane(int r) { return ((r >> 2) & 1) | (((r >> 1) & 1) << 1) | ((r & 1) << 2); }

}  // namespace fe
}  // namespace glinattn
