// nla_tc.cu -- chunked prefill of normalised kernelised linear attention.
//
// "Long context, fast inference, smart decoding, and life beyond attention",
// section "Linear attention: removing softmax entirely": with phi = elu + 1,
//   S_t = S_{t-1} + phi(k_t)^T v_t,   z_t = z_{t-1} + phi(k_t),
//   o_t = phi(q_t) S_t / (phi(q_t) . z_t + 1e-6).
// The numerator is gated linear attention with every gate equal to 1 on the
// features phi(q), phi(k), so it runs on the chunked tensor-core kernel; the
// denominator is a prefix sum of phi(k) dotted with phi(q).  Three launches:
//
//   1. nla_feature_kernel, one CTA per (chunk, q / k head, sequence): phi(q)
//      and phi(k) rounded to bf16 (the tensor-core operands) into the
//      workspace, and the chunk's column sums of phi(k); the chunk-0 CTAs
//      also copy the start normaliser, so that z_T may overwrite it;
//   2. gla_prefill_kernel without gates: phi(q) S_t, written in fp32 (into o
//      itself when o is fp32, else into the workspace);
//   3. nla_zscan_kernel, one thread per (sequence, q / k head, channel): the
//      exclusive prefix of the chunk sums, i.e. z at every chunk start;
//   4. nla_normalize_kernel, one CTA per (chunk, head, sequence): the 64
//      denominators of the chunk from z at its start (a warp per 16 tokens),
//      the division, and z_T from the last chunk.
//
// The denominators use the same bf16 feature values as the numerator.
#include <cuda_bf16.h>

#include "common.cuh"
#include "prefill_tc.cuh"

namespace glinattn {
namespace {

constexpr int kC = 64;    // chunk length (the tensor-core kernel's)
constexpr int kDK = 128;  // key head size

// exp of a non-positive argument through the fast exponential: its relative
// error (a few units of 2^-22) vanishes in the bf16 rounding that follows
__device__ __forceinline__ float feature_map(float x) { return x > 0.f ? x + 1.f : __expf(x); }

struct FeatureParams {
  const __nv_bfloat16 *q, *k;
  __nv_bfloat16 *fq, *fk;
  float *dz;        // [B, Hq, nchunks, dk]
  const float *z0;  // [B, H, dk] or NULL
  float *z0w;       // its copy (zeros for NULL)
  int T, H, Hq, nchunks;
};

constexpr int kFeatThreads = 256;  // 16 token rows x 16 groups of 8 channels

__device__ __forceinline__ uint4 features8(uint4 raw, float *rounded) {
  const __nv_bfloat162 *x = reinterpret_cast<const __nv_bfloat162 *>(&raw);
  uint4 out;
  uint32_t *o = reinterpret_cast<uint32_t *>(&out);
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const float2 f = __bfloat1622float2(x[m]);
    const __nv_bfloat162 y = __floats2bfloat162_rn(feature_map(f.x), feature_map(f.y));
    o[m] = *reinterpret_cast<const uint32_t *>(&y);
    if (rounded) {
      const float2 r = __bfloat1622float2(y);
      rounded[2 * m] = r.x;
      rounded[2 * m + 1] = r.y;
    }
  }
  return out;
}

// phi(q), phi(k) of one chunk of one q / k head, 16-byte accesses; the
// chunk's column sums of phi(k) are reduced across token rows in shared memory.
__global__ void __launch_bounds__(kFeatThreads, 4) nla_feature_kernel(const FeatureParams p) {
  __shared__ float red[16][kDK];
  const int c = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, cg = tid & 15, rg = tid >> 4;
  const int t0 = c * kC;
  uint4 qv[4], kv[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {  // every load issued before any store
    const int t = t0 + rg + 16 * j;
    if (t < p.T) {
      const size_t e = (((size_t)b * p.T + t) * p.Hq + hq) * kDK + 8 * cg;
      qv[j] = *reinterpret_cast<const uint4 *>(p.q + e);
      kv[j] = *reinterpret_cast<const uint4 *>(p.k + e);
    }
  }
  float zs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int t = t0 + rg + 16 * j;
    if (t < p.T) {
      const size_t e = (((size_t)b * p.T + t) * p.Hq + hq) * kDK + 8 * cg;
      float r[8];
      *reinterpret_cast<uint4 *>(p.fq + e) = features8(qv[j], nullptr);
      *reinterpret_cast<uint4 *>(p.fk + e) = features8(kv[j], r);
#pragma unroll
      for (int m = 0; m < 8; ++m) zs[m] += r[m];
    }
  }
#pragma unroll
  for (int m = 0; m < 8; ++m) red[rg][8 * cg + m] = zs[m];
  __syncthreads();
  if (tid < kDK) {
    float z = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r) z += red[r][tid];
    p.dz[(((size_t)b * p.Hq + hq) * p.nchunks + c) * kDK + tid] = z;
    if (c == 0) {
      const int rep = p.H / p.Hq;
      for (int h = hq * rep; h < (hq + 1) * rep; ++h) {
        const size_t e = ((size_t)b * p.H + h) * kDK + tid;
        p.z0w[e] = p.z0 ? p.z0[e] : 0.f;
      }
    }
  }
}

// z at every chunk start (without the start normaliser): zstart[c] = sum of
// the chunk sums before c.  The loads are independent; 8 are in flight.
__global__ void __launch_bounds__(kDK) nla_zscan_kernel(const float *__restrict__ dz, float *__restrict__ zstart,
                                                        int nchunks) {
  const size_t base = (size_t)blockIdx.x * nchunks * kDK + threadIdx.x;  // blockIdx.x = b * Hq + hq
  float z = 0.f;
  for (int c0 = 0; c0 < nchunks; c0 += 8) {
    float v[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) v[m] = c0 + m < nchunks ? dz[base + (size_t)(c0 + m) * kDK] : 0.f;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      if (c0 + m < nchunks) zstart[base + (size_t)(c0 + m) * kDK] = z;
      z += v[m];
    }
  }
}

struct NormParams {
  const __nv_bfloat16 *fq, *fk;
  const float *zstart, *z0;  // z0: the copy taken by the feature kernel
  float *z_T;
  const float *num;  // [B, T, H, dv] fp32 numerators
  void *o;           // [B, T, H, dv] out_dtype (may be num itself when fp32)
  int T, H, Hq, dv, nchunks, out_bf16;
};

// Warp w owns tokens 16w .. 16w+15 of the chunk and lane l the channels
// l + 32m: the lane first adds up phi(k) of the tokens before the warp's
// range, then for each of its tokens extends z and reduces phi(q) . z across
// the warp.  No shared-memory matrix, so many CTAs fit on an SM.
__global__ void __launch_bounds__(kDK) nla_normalize_kernel(const NormParams p) {
  __shared__ float inv_den[kC];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int hq = h / (p.H / p.Hq);
  const int t0 = c * kC, n = min(kC, p.T - t0);
  float zl[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int d = lane + 32 * m;
    zl[m] = p.z0[((size_t)b * p.H + h) * kDK + d] + p.zstart[(((size_t)b * p.Hq + hq) * p.nchunks + c) * kDK + d];
  }
  auto row = [&](int i) { return (((size_t)b * p.T + t0 + i) * p.Hq + hq) * kDK + lane; };
  const int first = 16 * warp;
  // phi(k) of the tokens before this warp's range, 8 rows of loads in flight
  for (int j0 = 0; j0 < min(first, n); j0 += 8) {
    float v[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int m = 0; m < 4; ++m) v[j][m] = j0 + j < n ? __bfloat162float(p.fk[row(j0 + j) + 32 * m]) : 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int m = 0; m < 4; ++m) zl[m] += v[j][m];
  }
  // this warp's tokens, 8 at a time
#pragma unroll
  for (int j0 = 0; j0 < 16; j0 += 8) {
    float fq[8][4], fk[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool in = first + j0 + j < n;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        fq[j][m] = in ? __bfloat162float(p.fq[row(first + j0 + j) + 32 * m]) : 0.f;
        fk[j][m] = in ? __bfloat162float(p.fk[row(first + j0 + j) + 32 * m]) : 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float s = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        zl[m] += fk[j][m];
        s += fq[j][m] * zl[m];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) inv_den[first + j0 + j] = 1.f / (s + 1e-6f);
    }
  }
  // the last warp's z covers every token of the chunk
  if (warp == 3 && c == p.nchunks - 1 && p.z_T)
#pragma unroll
    for (int m = 0; m < 4; ++m) p.z_T[((size_t)b * p.H + h) * kDK + lane + 32 * m] = zl[m];
  __syncthreads();
  const int d = tid;
  const int nv4 = p.dv / 4;
  const int total = n * nv4;
  for (int e0 = 0; e0 < total; e0 += 8 * kDK) {
    float4 x[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {  // all loads first: num may be o itself
      const int e = e0 + m * kDK + d;
      if (e < total) {
        const int i = e / nv4, j = 4 * (e - i * nv4);
        x[m] = *reinterpret_cast<const float4 *>(p.num + (((size_t)b * p.T + t0 + i) * p.H + h) * p.dv + j);
      }
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int e = e0 + m * kDK + d;
      if (e < total) {
        const int i = e / nv4, j = 4 * (e - i * nv4);
        const size_t off = (((size_t)b * p.T + t0 + i) * p.H + h) * p.dv + j;
        const float r = inv_den[i];
        const float4 y = make_float4(x[m].x * r, x[m].y * r, x[m].z * r, x[m].w * r);
        if (p.out_bf16) {
          const __nv_bfloat162 lo = __floats2bfloat162_rn(y.x, y.y), hi = __floats2bfloat162_rn(y.z, y.w);
          uint2 pk;
          pk.x = *reinterpret_cast<const uint32_t *>(&lo);
          pk.y = *reinterpret_cast<const uint32_t *>(&hi);
          *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.o) + off) = pk;
        } else {
          *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.o) + off) = y;
        }
      }
    }
  }
}

struct Carve {
  __nv_bfloat16 *fq, *fk;
  float *dz, *zstart, *z0w, *num;
  size_t bytes;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

Carve carve(void *base, const glinattn_prefill_args &a) {
  const int Hq = a.qk_heads > 0 ? a.qk_heads : a.heads;
  const int nchunks = (a.seqlen + kC - 1) / kC;
  const size_t feat = align256((size_t)a.batch * a.seqlen * Hq * kDK * 2);
  const size_t dz = align256((size_t)a.batch * Hq * nchunks * kDK * 4);
  const size_t zw = align256((size_t)a.batch * a.heads * kDK * 4);
  const size_t num = a.out_dtype == GLINATTN_BF16 ? align256((size_t)a.batch * a.seqlen * a.heads * a.dv * 4) : 0;
  uint8_t *p = static_cast<uint8_t *>(base);
  Carve c;
  c.fq = reinterpret_cast<__nv_bfloat16 *>(p);
  c.fk = reinterpret_cast<__nv_bfloat16 *>(p + feat);
  c.dz = reinterpret_cast<float *>(p + 2 * feat);
  c.zstart = reinterpret_cast<float *>(p + 2 * feat + dz);
  c.z0w = reinterpret_cast<float *>(p + 2 * feat + 2 * dz);
  c.num = num ? reinterpret_cast<float *>(p + 2 * feat + 2 * dz + zw) : nullptr;
  c.bytes = 2 * feat + 2 * dz + zw + num;
  return c;
}

}  // namespace

bool nla_tc_supports(const glinattn_prefill_args &a) {
  return a.variant == GLINATTN_NLA && a.in_dtype == GLINATTN_BF16 && a.dk == kDK && (a.dv == 128 || a.dv == 64) &&
         a.conv_w == nullptr && !a.qk_l2norm && a.state_every == 0 && a.seqlen > 0 && a.batch <= 65535 &&
         a.heads <= 65535;
}

size_t nla_tc_workspace_bytes(const glinattn_prefill_args &a) { return carve(nullptr, a).bytes; }

glinattn_status launch_nla_tc(const glinattn_prefill_args &a, cudaStream_t stream) {
  const int B = a.batch, T = a.seqlen, H = a.heads;
  const int Hq = a.qk_heads > 0 ? a.qk_heads : H;
  const int nchunks = (T + kC - 1) / kC;
  const Carve w = carve(a.workspace, a);

  FeatureParams fp;
  fp.q = static_cast<const __nv_bfloat16 *>(a.q);
  fp.k = static_cast<const __nv_bfloat16 *>(a.k);
  fp.fq = w.fq;
  fp.fk = w.fk;
  fp.dz = w.dz;
  fp.z0 = a.z0;
  fp.z0w = w.z0w;
  fp.T = T;
  fp.H = H;
  fp.Hq = Hq;
  fp.nchunks = nchunks;
  nla_feature_kernel<<<dim3((unsigned)nchunks, (unsigned)Hq, (unsigned)B), kFeatThreads, 0, stream>>>(fp);
  if (cudaGetLastError() != cudaSuccess) return GLINATTN_ERR_CUDA;

  // the numerator: gated linear attention with every gate 1, in fp32
  float *num = a.out_dtype == GLINATTN_BF16 ? w.num : static_cast<float *>(a.o);
  glinattn_prefill_args g = a;
  g.variant = GLINATTN_GLA;
  g.q = w.fq;
  g.k = w.fk;
  g.alpha = nullptr;
  g.beta = nullptr;
  g.o = num;
  g.out_dtype = GLINATTN_F32;
  g.state_every = 0;
  const glinattn_status st = launch_prefill_tc(g, stream);
  if (st != GLINATTN_OK) return st;

  nla_zscan_kernel<<<(unsigned)(B * Hq), kDK, 0, stream>>>(w.dz, w.zstart, nchunks);
  if (cudaGetLastError() != cudaSuccess) return GLINATTN_ERR_CUDA;

  NormParams np;
  np.fq = w.fq;
  np.fk = w.fk;
  np.zstart = w.zstart;
  np.z0 = w.z0w;
  np.z_T = a.z_T;
  np.num = num;
  np.o = a.o;
  np.T = T;
  np.H = H;
  np.Hq = Hq;
  np.dv = a.dv;
  np.nchunks = nchunks;
  np.out_bf16 = a.out_dtype == GLINATTN_BF16;
  nla_normalize_kernel<<<dim3((unsigned)nchunks, (unsigned)H, (unsigned)B), kDK, 0, stream>>>(np);
  return cudaGetLastError() == cudaSuccess ? GLINATTN_OK : GLINATTN_ERR_CUDA;
}

}  // namespace glinattn
