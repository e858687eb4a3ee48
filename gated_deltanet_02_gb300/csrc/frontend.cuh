// frontend.cuh -- the single-precision arithmetic of the layer's front end.
//
// With bf16 activations the short convolution and the L2 norm end in a
// rounding to bf16, i.e. in a decision: a value near a bf16 rounding boundary
// goes one way or the other depending on the last bits of the fp32 result.
// Every kernel therefore evaluates the front end in one fixed order, with
// every product and sum rounded on its own (no fused multiply-add):
//   conv:  y = ((w0 x_{t-3} + w1 x_{t-2}) + w2 x_{t-1}) + w3 x_t
//   norm:  s = sum of y_i^2 over the row by pairwise summation (the row split
//          in halves, recursively: adjacent pairs first), r = 1 / sqrt(s + 1e-6),
//          each element scaled by r
// so that the same inputs give the same bf16 activations in every kernel:
// prefill, decode and speculative decode agree bit for bit on them.
#pragma once

#include <cuda_runtime.h>

namespace glinattn {
namespace fe {

// one output of the width-4 causal convolution, oldest tap first
__device__ __forceinline__ float conv4(float w0, float w1, float w2, float w3, float x0, float x1, float x2,
                                       float x3) {
  float acc = __fadd_rn(__fmul_rn(w0, x0), __fmul_rn(w1, x1));
  acc = __fadd_rn(acc, __fmul_rn(w2, x2));
  return __fadd_rn(acc, __fmul_rn(w3, x3));
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

}  // namespace fe
}  // namespace glinattn
