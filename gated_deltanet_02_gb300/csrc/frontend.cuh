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
#include <stdint.h>

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

// ---- two channels at once: the packed fp32 pair instructions round each half
// on its own, exactly as the scalar operations above do
using f2 = unsigned long long;  // (low half, high half)

__device__ __forceinline__ f2 f2_pack(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(f2 v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
  f2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
  f2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// conv4 on a pair of channels
__device__ __forceinline__ f2 conv4x2(f2 w0, f2 w1, f2 w2, f2 w3, f2 x0, f2 x1, f2 x2, f2 x3) {
  return f2_add(f2_add(f2_add(f2_mul(w0, x0), f2_mul(w1, x1)), f2_mul(w2, x2)), f2_mul(w3, x3));
}
// two bf16x2 words a, b as fp32 pairs: their low halves (a.lo, b.lo) and their
// high halves (a.hi, b.hi)
__device__ __forceinline__ f2 bf16_lows(uint32_t a, uint32_t b) { return f2_pack(__uint_as_float(a << 16), __uint_as_float(b << 16)); }
__device__ __forceinline__ f2 bf16_highs(uint32_t a, uint32_t b) {
  return f2_pack(__uint_as_float(a & 0xffff0000u), __uint_as_float(b & 0xffff0000u));
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
