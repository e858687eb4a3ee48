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
//   3. nla_normalize_kernel, one CTA per (chunk, head, sequence): z at the
//      chunk start from the earlier chunks' sums, the 64 denominators of the
//      chunk, the division, and z_T from the last chunk.
//
// The denominators use the same bf16 feature values as the numerator.
#include <cuda_bf16.h>

#include "common.cuh"
#include "prefill_tc.cuh"

namespace glinattn {
namespace {

constexpr int kC = 64;    // chunk length (the tensor-core kernel's)
constexpr int kDK = 128;  // key head size

__device__ __forceinline__ float feature_map(float x) { return x > 0.f ? x + 1.f : expf(x); }

struct FeatureParams {
  const __nv_bfloat16 *q, *k;
  __nv_bfloat16 *fq, *fk;
  float *dz;        // [B, Hq, nchunks, dk]
  const float *z0;  // [B, H, dk] or NULL
  float *z0w;       // its copy (zeros for NULL)
  int T, H, Hq, nchunks;
};

__global__ void __launch_bounds__(kDK) nla_feature_kernel(const FeatureParams p) {
  const int c = blockIdx.x, hq = blockIdx.y, b = blockIdx.z, d = threadIdx.x;
  const int t0 = c * kC, n = min(kC, p.T - t0);
  float zsum = 0.f;
  for (int i = 0; i < n; ++i) {
    const size_t e = (((size_t)b * p.T + t0 + i) * p.Hq + hq) * kDK + d;
    p.fq[e] = __float2bfloat16_rn(feature_map(__bfloat162float(p.q[e])));
    const __nv_bfloat16 fk = __float2bfloat16_rn(feature_map(__bfloat162float(p.k[e])));
    p.fk[e] = fk;
    zsum += __bfloat162float(fk);
  }
  p.dz[(((size_t)b * p.Hq + hq) * p.nchunks + c) * kDK + d] = zsum;
  if (c == 0) {
    const int rep = p.H / p.Hq;
    for (int h = hq * rep; h < (hq + 1) * rep; ++h) {
      const size_t e = ((size_t)b * p.H + h) * kDK + d;
      p.z0w[e] = p.z0 ? p.z0[e] : 0.f;
    }
  }
}

struct NormParams {
  const __nv_bfloat16 *fq, *fk;
  const float *dz, *z0;  // z0: the copy taken by the feature kernel
  float *z_T;
  const float *num;  // [B, T, H, dv] fp32 numerators
  void *o;           // [B, T, H, dv] out_dtype (may be num itself when fp32)
  int T, H, Hq, dv, nchunks, out_bf16;
};

__global__ void __launch_bounds__(kDK) nla_normalize_kernel(const NormParams p) {
  __shared__ float red[kC][kDK + 1];  // padded: row i, column j in bank (i + j) % 32
  __shared__ float inv_den[kC];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, d = threadIdx.x;
  const int hq = h / (p.H / p.Hq);
  const int t0 = c * kC, n = min(kC, p.T - t0);
  // z at the start of the chunk: the start normaliser and the earlier chunks' sums
  float z = p.z0[((size_t)b * p.H + h) * kDK + d];
  for (int cc = 0; cc < c; ++cc) z += p.dz[(((size_t)b * p.Hq + hq) * p.nchunks + cc) * kDK + d];
  for (int i = 0; i < n; ++i) {
    const size_t e = (((size_t)b * p.T + t0 + i) * p.Hq + hq) * kDK + d;
    z += __bfloat162float(p.fk[e]);
    red[i][d] = __bfloat162float(p.fq[e]) * z;
  }
  if (c == p.nchunks - 1 && p.z_T) p.z_T[((size_t)b * p.H + h) * kDK + d] = z;
  __syncthreads();
  if (d < n) {
    float s = 0.f;
    for (int j = 0; j < kDK; ++j) s += red[d][j];
    inv_den[d] = 1.f / (s + 1e-6f);
  }
  __syncthreads();
  const int nv4 = p.dv / 4;
  for (int e = d; e < n * nv4; e += kDK) {
    const int i = e / nv4, j = 4 * (e - i * nv4);
    const size_t off = (((size_t)b * p.T + t0 + i) * p.H + h) * p.dv + j;
    float4 x = *reinterpret_cast<const float4 *>(p.num + off);
    const float r = inv_den[i];
    x.x *= r; x.y *= r; x.z *= r; x.w *= r;
    if (p.out_bf16) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y), hi = __floats2bfloat162_rn(x.z, x.w);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t *>(&lo);
      pk.y = *reinterpret_cast<const uint32_t *>(&hi);
      *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.o) + off) = pk;
    } else {
      *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.o) + off) = x;
    }
  }
}

struct Carve {
  __nv_bfloat16 *fq, *fk;
  float *dz, *z0w, *num;
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
  c.z0w = reinterpret_cast<float *>(p + 2 * feat + dz);
  c.num = num ? reinterpret_cast<float *>(p + 2 * feat + dz + zw) : nullptr;
  c.bytes = 2 * feat + dz + zw + num;
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
  nla_feature_kernel<<<dim3((unsigned)nchunks, (unsigned)Hq, (unsigned)B), kDK, 0, stream>>>(fp);
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

  NormParams np;
  np.fq = w.fq;
  np.fk = w.fk;
  np.dz = w.dz;
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
