// tc_common.cuh -- device helpers shared by the tensor-core prefill kernels.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>
#include <string.h>

#include "sm100.cuh"

namespace glinattn {
namespace tc {

using namespace sm100;

// Bounded wait that also gives up as soon as another role has aborted.
template <bool kHint = true>
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort) {
  if (mbar_try_wait<kHint>(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait<kHint>(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      return false;
    }
  }
}

// Whether any of a unit's T gates (alpha at a[t * stride]) is outside (0, 1]:
// this thread's share, eight independent loads in flight per round.
__device__ __forceinline__ int gates_bad(const float *a, int T, size_t stride, int tid, int nthreads) {
  int bad = 0;
  for (int t0 = tid; t0 < T; t0 += 8 * nthreads) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t = t0 + j * nthreads;
      v[j] = t < T ? a[(size_t)t * stride] : 1.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) bad |= !(v[j] > 0.f && v[j] <= 1.f);
  }
  return bad;
}

// Warp-uniform version for warps that go on to warp-collective tcgen05.ld.
template <bool kHint = true>
__device__ __forceinline__ bool wait_bar_warp(uint64_t *bar, uint32_t parity, volatile int *abort) {
  const bool ok = wait_bar<kHint>(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk16) {
  return row * 128u + ((chunk16 ^ (row & 7u)) << 4);
}

// 8 fp32 -> bf16 high parts and bf16 remainders, packed as 16 bytes each.
// hi keeps the top 16 bits of x (bf16 by truncation), x - hi is exact in
// fp32, and its top 16 bits are the remainder; hi + lo matches x to 2^-14
// relative, using only integer / fp32 ops (no format conversions).
__device__ __forceinline__ uint32_t bits(__nv_bfloat162 v) {
  uint32_t u;
  memcpy(&u, &v, 4);
  return u;
}

__device__ __forceinline__ void split8(const float *x, uint4 &hi, uint4 &lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t u0 = __float_as_uint(x[2 * k]), u1 = __float_as_uint(x[2 * k + 1]);
    const float r0 = x[2 * k] - __uint_as_float(u0 & 0xffff0000u);
    const float r1 = x[2 * k + 1] - __uint_as_float(u1 & 0xffff0000u);
    h[k] = __byte_perm(u0, u1, 0x7632);
    l[k] = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void unpack8(const uint4 &u, float *x) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = __uint_as_float(w[k] << 16);
    x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
  }
}

// bf16 high parts (top 16 bits) and remainders of a pair, packed as 32 bits
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const uint32_t u0 = __float_as_uint(x0), u1 = __float_as_uint(x1);
  const float r0 = x0 - __uint_as_float(u0 & 0xffff0000u);
  const float r1 = x1 - __uint_as_float(u1 & 0xffff0000u);
  hi = __byte_perm(u0, u1, 0x7632);
  lo = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
}

// Arrive once per warp, after the warp's own work: __syncwarp orders the
// lanes' shared-memory and TMEM accesses before lane 0's arrival.
__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// log2 of the smallest per-row output scale c_i of the chunked kernels: the
// outputs are c_i (Q S + P'' V) with P''_ij = (Q K^T)_ij 2^(g_i - g_j) / c_i
// and c_i = 2^max(g_i, -100), so no factor of P'' exceeds 2^100
constexpr float kRowScaleFloor = -100.f;

}  // namespace tc
}  // namespace glinattn
