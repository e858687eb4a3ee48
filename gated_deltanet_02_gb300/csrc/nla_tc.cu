// nla_tc.cu -- chunked prefill of normalised kernelised linear attention.
//
// "Long context, fast inference, smart decoding, and life beyond attention",
// section "Linear attention: removing softmax entirely": with phi = elu + 1,
//   S_t = S_{t-1} + phi(k_t)^T v_t,   z_t = z_{t-1} + phi(k_t),
//   o_t = phi(q_t) S_t / (phi(q_t) . z_t + 1e-6).
// The numerator is gated linear attention with every gate equal to 1 on the
// features phi(q), phi(k), so it runs on the chunked tensor-core kernel.
// Inside a chunk the denominator splits the same way as the numerator:
// phi(q_t) . z_t = phi(q_t) . z_start + sum over s <= t of phi(q_t) . phi(k_s),
// and the second term is the row sum of the masked phi(Q) phi(K)^T tile that
// the kernel already forms.  Two launches:
//
//   1. nla_feature_kernel, one CTA per (chunk, q / k head, sequence): phi(q)
//      and phi(k) rounded to bf16 (the tensor-core operands) into the
//      workspace, and the chunk's column sums of phi(k); the chunk-0 CTAs
//      also copy the start normaliser, so that z_T may overwrite it;
//   2. gla_prefill_kernel, normalised instance: no gates; z is the state of a
//      value column that is 1 in every token, so warpgroup A carries it from
//      chunk to chunk (the start normaliser plus each chunk's column sums,
//      which travel with the chunk's tiles) and forms each token's
//      denominator from z at its chunk start and the row sum; the outputs
//      are divided by it in the epilogue and written in the output dtype,
//      and z_T is written at the end.
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

struct Carve {
  __nv_bfloat16 *fq, *fk;
  float *dz, *z0w;
  size_t bytes;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

Carve carve(void *base, const glinattn_prefill_args &a) {
  const int Hq = a.qk_heads > 0 ? a.qk_heads : a.heads;
  const int nchunks = (a.seqlen + kC - 1) / kC;
  const size_t feat = align256((size_t)a.batch * a.seqlen * Hq * kDK * 2);
  const size_t dz = align256((size_t)a.batch * Hq * nchunks * kDK * 4);
  const size_t zw = align256((size_t)a.batch * a.heads * kDK * 4);
  uint8_t *p = static_cast<uint8_t *>(base);
  Carve c;
  c.fq = reinterpret_cast<__nv_bfloat16 *>(p);
  c.fk = reinterpret_cast<__nv_bfloat16 *>(p + feat);
  c.dz = reinterpret_cast<float *>(p + 2 * feat);
  c.z0w = reinterpret_cast<float *>(p + 2 * feat + dz);
  c.bytes = 2 * feat + dz + zw;
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

  // gated linear attention with every gate 1 on the features, normalised in
  // its epilogue
  glinattn_prefill_args g = a;
  g.variant = GLINATTN_GLA;
  g.q = w.fq;
  g.k = w.fk;
  g.alpha = nullptr;
  g.beta = nullptr;
  g.state_every = 0;
  return launch_prefill_tc_nla(g, stream, nullptr, w.dz, w.z0w, a.z_T);
}

}  // namespace glinattn
