// selective_scan.cu -- Mamba's selective state-space scan: chunked prefill and
// a slot-indexed decode step.
//
// "Long context, fast inference, smart decoding, and life beyond attention",
// chapter "05 · State-space models: the architectural alternative": with
// dt = softplus(delta) per channel d and a fixed A [D, N],
//   h_t[d, n] = exp(dt_t[d] A[d, n]) h_{t-1}[d, n] + dt_t[d] B_t[n] x_t[d],
//   y_t[d]    = sum_n h_t[d, n] C_t[n].
// Every (d, n) pair is an independent scalar recurrence, so the work is
// elementwise; what limits it is the serial dependence along t.  The section
// on Mamba's engineering replaces the loop by a parallel scan; here the scan is
// split into chunks of 64 tokens:
//
//   1. ssm_chunk_kernel: every (sequence, chunk, channel) runs its chunk from a
//      zero state and keeps the end state and sum(dt) (the chunk's decay is
//      exp(A sum(dt)), since A is fixed);
//   2. ssm_carry_kernel: per (sequence, channel, n), the chunk start states,
//      serially over chunks (one multiply-add each), and the final state;
//   3. ssm_chunk_kernel again (OUT = true): every chunk from its true start
//      state, writing y.
//
// A thread owns one channel and its N states in registers; the chunk's B and C
// rows (shared by all channels) are staged in shared memory, and x, delta are
// read 16 tokens ahead in one batch so their loads overlap.  The work is
// bound by the special-function unit (one exp per token, channel and state),
// so this file is compiled with fast math and the decays are exp2 of A log2(e)
// pre-scaled once per thread: one hardware exp2 per state element.  The
// arguments are non-positive, where its relative error (a few units of 2^-22)
// is far inside the fp32 tolerance of the scan; results below the normal
// range flush to zero, i.e. a state element that has decayed below 1e-38 is
// dropped.
#include <cuda_bf16.h>

#include "common.cuh"

namespace glinattn {
namespace {

constexpr int kL = 64;      // chunk length
constexpr int kCT = 128;    // channels per CTA
constexpr int kBatchT = 16; // tokens whose x, delta loads are in flight together

__device__ __forceinline__ float act_ld(const void *base, size_t i, int bf16) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[i]);
  return reinterpret_cast<const float *>(base)[i];
}

__device__ __forceinline__ void act_st(void *base, size_t i, float v, int bf16) {
  if (bf16)
    reinterpret_cast<__nv_bfloat16 *>(base)[i] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float *>(base)[i] = v;
}

// softplus(x) = log(1 + e^x) = max(x, 0) + log(1 + e^-|x|).  With e = e^-|x|
// in (0, 1]: below 1e-3 the series e - e^2/2 (truncation e^3/3, relative
// < 4e-7) avoids the cancellation of log(1 + e); above it the fast log of
// 1 + e in [1.001, 2] is accurate to about 1e-7 absolute.
__device__ __forceinline__ float softplus(float x) {
  const float e = __expf(-fabsf(x));
  const float l = e < 1e-3f ? e * (1.f - 0.5f * e) : __logf(1.f + e);
  return fmaxf(x, 0.f) + l;
}

struct ScanParams {
  const void *x, *delta, *Bm, *Cm;
  const float *A, *h0;
  float *h_T;
  void *y;
  float *h_end, *sdt, *h_start;  // workspace: [B, nc, D, N], [B, nc, D], [B, nc, D, N]
  int B, T, D, nc, in_bf16, out_bf16;
};

template <int N>
__device__ __forceinline__ void stage_bc(const ScanParams &p, int b, int t0, int n, float (*sB)[N], float (*sC)[N],
                                         bool withC) {
  for (int e = threadIdx.x; e < kL * N; e += kCT) {
    const int i = e / N, j = e - i * N;
    const bool in = i < n;
    const size_t g = ((size_t)b * p.T + t0 + i) * N + j;
    sB[i][j] = in ? act_ld(p.Bm, g, p.in_bf16) : 0.f;
    if (withC) sC[i][j] = in ? act_ld(p.Cm, g, p.in_bf16) : 0.f;
  }
}

// Passes 1 and 3 share this body: OUT = false keeps the chunk's end state and
// sum(dt); OUT = true starts from the carried state and writes y.
template <int N, bool OUT>
__global__ void __launch_bounds__(kCT) ssm_chunk_kernel(const ScanParams p) {
  __shared__ float sB[kL][N], sC[kL][N];
  const int c = blockIdx.y, b = blockIdx.z;
  const int d = blockIdx.x * kCT + threadIdx.x;
  const int t0 = c * kL, n = min(kL, p.T - t0);
  stage_bc<N>(p, b, t0, n, sB, sC, OUT);
  const bool active = d < p.D;
  float Ad[N], h[N];
#pragma unroll
  for (int j = 0; j < N; ++j) {
    Ad[j] = active ? p.A[(size_t)d * N + j] * 1.4426950408889634f : 0.f;  // A log2(e)
    h[j] = 0.f;
  }
  if (OUT && active) {
    const float4 *src = reinterpret_cast<const float4 *>(p.h_start + (((size_t)b * p.nc + c) * p.D + d) * N);
#pragma unroll
    for (int j = 0; j < N / 4; ++j) {
      const float4 v = src[j];
      h[4 * j] = v.x; h[4 * j + 1] = v.y; h[4 * j + 2] = v.z; h[4 * j + 3] = v.w;
    }
  }
  __syncthreads();
  float sdt = 0.f;
  for (int i0 = 0; i0 < n; i0 += kBatchT) {
    float xs[kBatchT], ds[kBatchT];
#pragma unroll
    for (int i = 0; i < kBatchT; ++i) {
      const bool in = active && i0 + i < n;
      const size_t g = ((size_t)b * p.T + t0 + i0 + i) * p.D + d;
      xs[i] = in ? act_ld(p.x, g, p.in_bf16) : 0.f;
      ds[i] = in ? act_ld(p.delta, g, p.in_bf16) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kBatchT; ++i) {
      if (i0 + i >= n) break;
      const float dt = softplus(ds[i]);
      const float dtx = dt * xs[i];
      float yv = 0.f;
#pragma unroll
      for (int j = 0; j < N; ++j) {
        h[j] = exp2f(dt * Ad[j]) * h[j] + dtx * sB[i0 + i][j];
        if (OUT) yv += h[j] * sC[i0 + i][j];
      }
      if (OUT) {
        if (active) act_st(p.y, ((size_t)b * p.T + t0 + i0 + i) * p.D + d, yv, p.out_bf16);
      } else {
        sdt += dt;
      }
    }
  }
  if (!OUT && active) {
    float4 *dst = reinterpret_cast<float4 *>(p.h_end + (((size_t)b * p.nc + c) * p.D + d) * N);
#pragma unroll
    for (int j = 0; j < N / 4; ++j) dst[j] = make_float4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
    p.sdt[((size_t)b * p.nc + c) * p.D + d] = sdt;
  }
}

// Chunk start states: h_start[c] = exp(A sum(dt)_{c-1}) h_start[c-1] + h_end[c-1].
template <int N>
__global__ void __launch_bounds__(256) ssm_carry_kernel(const ScanParams p) {
  const size_t e = (size_t)blockIdx.x * 256 + threadIdx.x;  // (b, d, n)
  const size_t per = (size_t)p.D * N;
  if (e >= (size_t)p.B * per) return;
  const int b = (int)(e / per);
  const size_t dn = e - (size_t)b * per;
  const int d = (int)(dn / N);
  const float A = p.A[dn];
  float h = p.h0 ? p.h0[(size_t)b * per + dn] : 0.f;
  // the end states and step sums of 8 chunks are loaded together
  for (int c0 = 0; c0 < p.nc; c0 += 8) {
    float he[8], sd[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int c = c0 + m;
      he[m] = c < p.nc ? p.h_end[((size_t)b * p.nc + c) * per + dn] : 0.f;
      sd[m] = c < p.nc ? p.sdt[((size_t)b * p.nc + c) * p.D + d] : 0.f;
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int c = c0 + m;
      if (c < p.nc) {
        p.h_start[((size_t)b * p.nc + c) * per + dn] = h;
        h = __expf(A * sd[m]) * h + he[m];
      }
    }
  }
  p.h_T[(size_t)b * per + dn] = h;
}

struct ScanDecodeParams {
  const void *x, *delta, *Bm, *Cm;
  const float *A;
  float *pool;
  const int32_t *slot_ids;
  void *y;
  uint32_t *dev_status;
  int R, D, P, in_bf16, out_bf16;
};

// One step per (request, channel): N / 4 consecutive threads share a channel,
// each moving one float4 of its states, so a warp reads and writes whole
// contiguous state rows; y is reduced across the channel's threads.
template <int N>
__global__ void __launch_bounds__(256) ssm_decode_kernel(const ScanDecodeParams p) {
  constexpr int kQ = N / 4;           // threads per channel
  constexpr int kCh = 256 / kQ;       // channels per CTA
  const int r = blockIdx.y;
  const int q = threadIdx.x % kQ;
  const int d = blockIdx.x * kCh + threadIdx.x / kQ;
  const bool valid = d < p.D;
  const int slot = p.slot_ids[r];
  if (slot < 0 || slot >= p.P) {  // uniform over the CTA
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_BAD_SLOT);
    return;
  }
  float4 *hp = reinterpret_cast<float4 *>(p.pool + ((size_t)slot * p.D + d) * N) + q;
  const float4 h4 = valid ? *hp : make_float4(0.f, 0.f, 0.f, 0.f);
  const float4 a4 = valid ? reinterpret_cast<const float4 *>(p.A + (size_t)d * N)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
  const size_t g = (size_t)r * p.D + (valid ? d : 0);
  const float dt = softplus(act_ld(p.delta, g, p.in_bf16));
  const float dtx = dt * act_ld(p.x, g, p.in_bf16);
  float h[4] = {h4.x, h4.y, h4.z, h4.w};
  const float av[4] = {a4.x, a4.y, a4.z, a4.w};
  float yv = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int n = 4 * q + j;
    h[j] = __expf(dt * av[j]) * h[j] + dtx * act_ld(p.Bm, (size_t)r * N + n, p.in_bf16);
    yv += h[j] * act_ld(p.Cm, (size_t)r * N + n, p.in_bf16);
  }
#pragma unroll
  for (int o = kQ / 2; o > 0; o >>= 1) yv += __shfl_xor_sync(0xffffffffu, yv, o);
  if (valid) {
    *hp = make_float4(h[0], h[1], h[2], h[3]);
    if (q == 0) act_st(p.y, g, yv, p.out_bf16);
  }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool state_ok(int n) { return n == 8 || n == 16 || n == 32; }

template <int N>
cudaError_t launch_scan(const ScanParams &p, cudaStream_t s) {
  const dim3 g13((unsigned)((p.D + kCT - 1) / kCT), (unsigned)p.nc, (unsigned)p.B);
  ssm_chunk_kernel<N, false><<<g13, kCT, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t total = (size_t)p.B * p.D * N;
  ssm_carry_kernel<N><<<(unsigned)((total + 255) / 256), 256, 0, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ssm_chunk_kernel<N, true><<<g13, kCT, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace
}  // namespace glinattn

using glinattn::align256;

namespace {

size_t scan_workspace(const glinattn_scan_args *a, size_t *off_sdt, size_t *off_hs) {
  const int nc = (a->seqlen + glinattn::kL - 1) / glinattn::kL;
  const size_t hb = align256((size_t)a->batch * nc * a->channels * a->state * 4);
  const size_t sb = align256((size_t)a->batch * nc * a->channels * 4);
  if (off_sdt) *off_sdt = hb;
  if (off_hs) *off_hs = hb + sb;
  return 2 * hb + sb;
}

glinattn_status check_scan(const glinattn_scan_args *a) {
  if (!a) return GLINATTN_ERR_INVALID_ARG;
  if ((a->in_dtype != GLINATTN_F32 && a->in_dtype != GLINATTN_BF16) ||
      (a->out_dtype != GLINATTN_F32 && a->out_dtype != GLINATTN_BF16))
    return GLINATTN_ERR_INVALID_ARG;
  if (a->batch < 0 || a->seqlen < 0 || a->channels <= 0 || a->state <= 0) return GLINATTN_ERR_INVALID_ARG;
  if (!glinattn::state_ok(a->state)) return GLINATTN_ERR_UNSUPPORTED;
  if ((long long)a->batch * a->channels * a->state > (1ll << 31) || a->batch > 65535 ||
      (long long)a->seqlen > (1ll << 30) || (a->seqlen + glinattn::kL - 1) / glinattn::kL > 65535)
    return GLINATTN_ERR_UNSUPPORTED;
  return GLINATTN_OK;
}

}  // namespace

extern "C" size_t glinattn_selective_scan_workspace_size(const glinattn_scan_args *a) {
  if (check_scan(a) != GLINATTN_OK || a->batch == 0 || a->seqlen == 0) return 0;
  return scan_workspace(a, nullptr, nullptr);
}

extern "C" glinattn_status glinattn_selective_scan(const glinattn_scan_args *a, glinattn_stream_t stream) {
  glinattn_status st = check_scan(a);
  if (st != GLINATTN_OK) return st;
  if (a->batch == 0) return GLINATTN_OK;
  if (!a->A || !a->h_T) return GLINATTN_ERR_INVALID_ARG;
  if (a->seqlen > 0 && (!a->x || !a->delta || !a->Bm || !a->Cm || !a->y)) return GLINATTN_ERR_INVALID_ARG;
  if (!glinattn::aligned16(a->A) || !glinattn::aligned16(a->h_T) || (a->h0 && !glinattn::aligned16(a->h0)))
    return GLINATTN_ERR_INVALID_ARG;
  const size_t hbytes = (size_t)a->batch * a->channels * a->state * 4;
  if (a->h0 && a->h0 != a->h_T) {
    const uintptr_t x = (uintptr_t)a->h0, y = (uintptr_t)a->h_T;
    if (x < y + hbytes && y < x + hbytes) return GLINATTN_ERR_INVALID_ARG;  // partial overlap
  }
  if (a->seqlen == 0) {  // an empty segment hands its start state on
    if (a->h0 == a->h_T) return GLINATTN_OK;
    const cudaError_t e = a->h0 ? cudaMemcpyAsync(a->h_T, a->h0, hbytes, cudaMemcpyDeviceToDevice,
                                                  (cudaStream_t)stream)
                                : cudaMemsetAsync(a->h_T, 0, hbytes, (cudaStream_t)stream);
    return e == cudaSuccess ? GLINATTN_OK : GLINATTN_ERR_CUDA;
  }
  size_t off_sdt = 0, off_hs = 0;
  const size_t need = scan_workspace(a, &off_sdt, &off_hs);
  if (!a->workspace || a->workspace_bytes < need || !glinattn::aligned16(a->workspace))
    return GLINATTN_ERR_INVALID_ARG;
  glinattn::ScanParams p;
  p.x = a->x;
  p.delta = a->delta;
  p.Bm = a->Bm;
  p.Cm = a->Cm;
  p.A = a->A;
  p.h0 = a->h0;
  p.h_T = a->h_T;
  p.y = a->y;
  uint8_t *ws = static_cast<uint8_t *>(a->workspace);
  p.h_end = reinterpret_cast<float *>(ws);
  p.sdt = reinterpret_cast<float *>(ws + off_sdt);
  p.h_start = reinterpret_cast<float *>(ws + off_hs);
  p.B = a->batch;
  p.T = a->seqlen;
  p.D = a->channels;
  p.nc = (a->seqlen + glinattn::kL - 1) / glinattn::kL;
  p.in_bf16 = a->in_dtype == GLINATTN_BF16;
  p.out_bf16 = a->out_dtype == GLINATTN_BF16;
  const cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  switch (a->state) {
    case 8: e = glinattn::launch_scan<8>(p, s); break;
    case 16: e = glinattn::launch_scan<16>(p, s); break;
    default: e = glinattn::launch_scan<32>(p, s); break;
  }
  return e == cudaSuccess ? GLINATTN_OK : GLINATTN_ERR_CUDA;
}

extern "C" glinattn_status glinattn_selective_scan_decode(const glinattn_scan_decode_args *a,
                                                          glinattn_stream_t stream) {
  if (!a) return GLINATTN_ERR_INVALID_ARG;
  if ((a->in_dtype != GLINATTN_F32 && a->in_dtype != GLINATTN_BF16) ||
      (a->out_dtype != GLINATTN_F32 && a->out_dtype != GLINATTN_BF16))
    return GLINATTN_ERR_INVALID_ARG;
  if (a->num_req < 0 || a->channels <= 0 || a->state <= 0 || a->pool_slots <= 0) return GLINATTN_ERR_INVALID_ARG;
  if (!glinattn::state_ok(a->state)) return GLINATTN_ERR_UNSUPPORTED;
  if (a->num_req > 65535) return GLINATTN_ERR_UNSUPPORTED;
  if (a->num_req == 0) return GLINATTN_OK;
  if (!a->x || !a->delta || !a->Bm || !a->Cm || !a->A || !a->state_pool || !a->slot_ids || !a->y)
    return GLINATTN_ERR_INVALID_ARG;
  if (!glinattn::aligned16(a->state_pool)) return GLINATTN_ERR_INVALID_ARG;
  glinattn::ScanDecodeParams p;
  p.x = a->x;
  p.delta = a->delta;
  p.Bm = a->Bm;
  p.Cm = a->Cm;
  p.A = a->A;
  p.pool = a->state_pool;
  p.slot_ids = a->slot_ids;
  p.y = a->y;
  p.dev_status = a->dev_status;
  p.R = a->num_req;
  p.D = a->channels;
  p.P = a->pool_slots;
  p.in_bf16 = a->in_dtype == GLINATTN_BF16;
  p.out_bf16 = a->out_dtype == GLINATTN_BF16;
  const unsigned per_cta = 256u / (unsigned)(a->state / 4);  // channels per CTA
  const dim3 grid((unsigned)((a->channels + per_cta - 1) / per_cta), (unsigned)a->num_req);
  cudaStream_t s = (cudaStream_t)stream;
  switch (a->state) {
    case 8: glinattn::ssm_decode_kernel<8><<<grid, 256, 0, s>>>(p); break;
    case 16: glinattn::ssm_decode_kernel<16><<<grid, 256, 0, s>>>(p); break;
    default: glinattn::ssm_decode_kernel<32><<<grid, 256, 0, s>>>(p); break;
  }
  return cudaGetLastError() == cudaSuccess ? GLINATTN_OK : GLINATTN_ERR_CUDA;
}
