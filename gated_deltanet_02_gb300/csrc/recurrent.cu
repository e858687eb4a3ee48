// recurrent.cu -- token-serial kernel for recurrent decode, speculative decode
// with one state per draft position, and the fp32 prefill path.
//
// "Inference for linear attention and hybrid architectures", section "Two
// ways to write the same computation": decode reads the state once and does
// one rank-one update per token, so each step is memory-bound and constant in
// the context length:
//   GLA:  S <- alpha S + k^T v                      o = q S = alpha (q S_old) + (q.k) v
//   GDN:  u = beta (v - alpha (k S_old))            S <- alpha S_old + k^T u
//         o = q S = alpha (q S_old) + (q.k) u
// (the Gated DeltaNet update alpha (I - beta k^T k) S + beta k^T v written as a
// rank-one correction of the decayed state).  Section "Speculative decoding
// and PD disaggregation": one state is kept per draft position, and batched
// kernels read and write the state pool by slot index.
//
// One CTA owns one (request, head) state, d x d fp32, held in registers for
// all of its steps: thread (rg, cg) holds rows rg + ROWG*i of column group cg
// (4 consecutive columns, one 16-byte vector), so every warp-wide load or
// store of a state row is contiguous.  k S and q S are reduced in one pass
// over the registers, across row groups through shared memory in a fixed
// order (deterministic, no atomics).  Decode (1 step, in place) and
// speculative decode (D steps, a write after each) run this same code, so a
// draft state equals the state of repeated decode steps bit for bit.
#include "common.cuh"

namespace glinattn {
namespace {

template <int D>
struct Shape {
  static constexpr int NT = (D * D / 4 < 256) ? D * D / 4 : 256;  // threads per CTA
  static constexpr int COLG = D / 4;                               // 16-byte column groups
  static constexpr int ROWG = NT / COLG;                           // row groups
  static constexpr int RPT = D / ROWG;                             // rows per thread
  static_assert(RPT >= 1 && ROWG * RPT == D, "shape");
};

__device__ __forceinline__ float load_act(const void *base, size_t idx, int bf16) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[idx]);
  return reinterpret_cast<const float *>(base)[idx];
}

__device__ __forceinline__ void store_act(void *base, size_t idx, float x, int bf16) {
  if (bf16)
    reinterpret_cast<__nv_bfloat16 *>(base)[idx] = __float2bfloat16_rn(x);
  else
    reinterpret_cast<float *>(base)[idx] = x;
}

__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int D>
__global__ void __launch_bounds__(Shape<D>::NT) recurrent_kernel(const RecurParams p) {
  using Sh = Shape<D>;
  constexpr int NW = (Sh::NT + 31) / 32;
  const int unit = blockIdx.x;
  const int n = unit / p.H, h = unit - n * p.H;
  const int tid = threadIdx.x;
  const int cg = tid % Sh::COLG, rg = tid / Sh::COLG;
  const size_t DD = (size_t)D * D;

  __shared__ float s_act[3 * D];      // q | k | v of the current token after the front end
  __shared__ float s_raw[3 * D];      // raw inputs of the current token
  __shared__ float s_hist[3][3 * D];  // conv history, oldest first
  __shared__ float s_red[Sh::ROWG][2][D];
  __shared__ float s_wsum[2][NW];
  __shared__ float s_qk;
  __shared__ int s_bad;

  // ---- unit validation: slots in range, gates in (0, 1] ----------------------
  if (tid == 0) s_bad = 0;
  __syncthreads();
  int bad = 0;
  if (p.pool_slots > 0) {
    if (p.src_slot && tid == 0) {
      const int s = p.src_slot[n];
      if (s < 0 || s >= p.pool_slots) bad |= GLINATTN_DEV_BAD_SLOT;
    }
    if (p.dst_slot) {
      const int nd = p.dst_per_step ? p.steps : 1;
      for (int t = tid; t < nd; t += Sh::NT) {
        const int s = p.dst_slot[(size_t)n * nd + t];
        if (s < 0 || s >= p.pool_slots) bad |= GLINATTN_DEV_BAD_SLOT;
      }
    }
  }
  for (int t = tid; t < p.steps; t += Sh::NT) {
    const float a = p.alpha[((size_t)n * p.steps + t) * p.H + h];
    if (!(a > 0.f && a <= 1.f)) bad |= GLINATTN_DEV_BAD_GATE;
  }
  if (bad) atomicOr(&s_bad, bad);
  __syncthreads();
  if (s_bad) {
    if (tid == 0 && p.dev_status) atomicOr(p.dev_status, (uint32_t)s_bad);
    return;
  }

  // ---- load the state into registers ------------------------------------------
  float4 S[Sh::RPT];
  {
    const float *src = nullptr;
    if (p.S_src) {
      const size_t slot = p.src_slot ? (size_t)p.src_slot[n] : (size_t)n;
      src = p.S_src + (slot * p.H + h) * DD;
    }
#pragma unroll
    for (int i = 0; i < Sh::RPT; ++i) {
      const int r = rg + Sh::ROWG * i;
      S[i] = src ? *reinterpret_cast<const float4 *>(src + (size_t)r * D + 4 * cg)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  // channel of this head for local channel c = part * D + i
  auto chan = [&](int c) { return (c / D) * p.H * D + h * D + (c % D); };

  // ---- conv history ----------------------------------------------------------
  const bool conv = p.conv_w != nullptr;
  if (conv) {
    const size_t cslot = p.src_slot ? (size_t)p.src_slot[n] : (size_t)n;
    for (int c = tid; c < 3 * D; c += Sh::NT)
#pragma unroll
      for (int j = 0; j < 3; ++j)
        s_hist[j][c] = p.conv_src ? load_act(p.conv_src, (cslot * 3 + j) * p.Cch + chan(c), p.in_bf16)
                                  : 0.f;
  }

  for (int t = 0; t < p.steps; ++t) {
    const size_t row = ((size_t)n * p.steps + t) * p.H + h;  // (n, t, h)
    // ---- front end: conv, L2 norm, bf16 rounding --------------------------------
    for (int c = tid; c < 3 * D; c += Sh::NT) {
      const int part = c / D, i = c % D;
      const void *src = part == 0 ? p.q : (part == 1 ? p.k : p.v);
      const float x = load_act(src, row * D + i, p.in_bf16);
      float y = x;
      if (conv) {
        const float *w = p.conv_w + (size_t)chan(c) * 4;
        y = w[0] * s_hist[0][c] + w[1] * s_hist[1][c] + w[2] * s_hist[2][c] + w[3] * x;
      }
      s_raw[c] = x;
      s_act[c] = y;
    }
    __syncthreads();
    if (conv) {
      for (int c = tid; c < 3 * D; c += Sh::NT) {
        s_hist[0][c] = s_hist[1][c];
        s_hist[1][c] = s_hist[2][c];
        s_hist[2][c] = s_raw[c];
      }
    }
    if (p.qk_l2norm) {
      // sum of squares of q (part 0) and k (part 1), fixed order
      float sq = 0.f, sk = 0.f;
      for (int i = tid; i < D; i += Sh::NT) {
        sq += s_act[i] * s_act[i];
        sk += s_act[D + i] * s_act[D + i];
      }
      sq = warp_sum(sq);
      sk = warp_sum(sk);
      if ((tid & 31) == 0) {
        s_wsum[0][tid >> 5] = sq;
        s_wsum[1][tid >> 5] = sk;
      }
      __syncthreads();
      float tq = 0.f, tk = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        tq += s_wsum[0][w];
        tk += s_wsum[1][w];
      }
      const float iq = 1.f / sqrtf(tq + 1e-6f), ik = 1.f / sqrtf(tk + 1e-6f);
      __syncthreads();  // everyone has read s_wsum before s_act changes
      for (int i = tid; i < D; i += Sh::NT) {
        s_act[i] *= iq;
        s_act[D + i] *= ik;
      }
    }
    if (p.in_bf16 && (conv || p.qk_l2norm)) {
      __syncthreads();
      for (int c = tid; c < 3 * D; c += Sh::NT) s_act[c] = round_bf16(s_act[c]);
    }
    __syncthreads();

    // ---- q.k (one warp, fixed order) and the partial k S, q S ------------------
    if (tid < 32) {
      float acc = 0.f;
      for (int i = tid; i < D; i += 32) acc += s_act[i] * s_act[D + i];
      acc = warp_sum(acc);
      if (tid == 0) s_qk = acc;
    }
    const float *sq = s_act, *sk = s_act + D, *sv = s_act + 2 * D;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
#pragma unroll
    for (int i = 0; i < Sh::RPT; ++i) {
      const int r = rg + Sh::ROWG * i;
      const float kr = sk[r], qr = sq[r];
      x.x += kr * S[i].x; x.y += kr * S[i].y; x.z += kr * S[i].z; x.w += kr * S[i].w;
      y.x += qr * S[i].x; y.y += qr * S[i].y; y.z += qr * S[i].z; y.w += qr * S[i].w;
    }
    *reinterpret_cast<float4 *>(&s_red[rg][0][4 * cg]) = x;
    *reinterpret_cast<float4 *>(&s_red[rg][1][4 * cg]) = y;
    __syncthreads();
    x = make_float4(0.f, 0.f, 0.f, 0.f);
    y = x;
#pragma unroll
    for (int r = 0; r < Sh::ROWG; ++r) {
      const float4 a = *reinterpret_cast<const float4 *>(&s_red[r][0][4 * cg]);
      const float4 b = *reinterpret_cast<const float4 *>(&s_red[r][1][4 * cg]);
      x.x += a.x; x.y += a.y; x.z += a.z; x.w += a.w;
      y.x += b.x; y.y += b.y; y.z += b.z; y.w += b.w;
    }

    // ---- update -----------------------------------------------------------------
    const float a = p.alpha[row];
    const float4 vv = *reinterpret_cast<const float4 *>(sv + 4 * cg);
    float4 u = vv;
    if (p.variant == GLINATTN_GDN) {
      const float b = p.beta[row];
      u.x = b * (vv.x - a * x.x);
      u.y = b * (vv.y - a * x.y);
      u.z = b * (vv.z - a * x.z);
      u.w = b * (vv.w - a * x.w);
    }
#pragma unroll
    for (int i = 0; i < Sh::RPT; ++i) {
      const float kr = sk[rg + Sh::ROWG * i];
      S[i].x = a * S[i].x + kr * u.x;
      S[i].y = a * S[i].y + kr * u.y;
      S[i].z = a * S[i].z + kr * u.z;
      S[i].w = a * S[i].w + kr * u.w;
    }
    if (rg == 0) {
      const float qk = s_qk;
      const size_t ob = row * D + 4 * cg;
      store_act(p.o, ob + 0, a * y.x + qk * u.x, p.out_bf16);
      store_act(p.o, ob + 1, a * y.y + qk * u.y, p.out_bf16);
      store_act(p.o, ob + 2, a * y.z + qk * u.z, p.out_bf16);
      store_act(p.o, ob + 3, a * y.w + qk * u.w, p.out_bf16);
    }

    // ---- per-step destination (one state per draft position) ------------------
    const bool last = (t == p.steps - 1);
    if (p.dst_per_step || last) {
      const size_t slot = p.dst_slot ? (size_t)p.dst_slot[(size_t)n * (p.dst_per_step ? p.steps : 1) +
                                                          (p.dst_per_step ? t : 0)]
                                     : (size_t)n;
      float *dst = p.S_dst + (slot * p.H + h) * DD;
#pragma unroll
      for (int i = 0; i < Sh::RPT; ++i)
        *reinterpret_cast<float4 *>(dst + (size_t)(rg + Sh::ROWG * i) * D + 4 * cg) = S[i];
      if (conv && p.conv_dst) {
        __syncthreads();  // s_hist shift complete
        for (int c = tid; c < 3 * D; c += Sh::NT)
#pragma unroll
          for (int j = 0; j < 3; ++j)
            store_act(p.conv_dst, (slot * 3 + j) * p.Cch + chan(c), s_hist[j][c], p.in_bf16);
      }
    }
    __syncthreads();  // shared buffers are rewritten by the next step
  }

  if (p.steps == 0) {  // a zero-length segment hands its inputs straight on
    float *dst = p.S_dst + ((size_t)n * p.H + h) * DD;
#pragma unroll
    for (int i = 0; i < Sh::RPT; ++i)
      *reinterpret_cast<float4 *>(dst + (size_t)(rg + Sh::ROWG * i) * D + 4 * cg) = S[i];
    if (conv && p.conv_dst)
      for (int c = tid; c < 3 * D; c += Sh::NT)
#pragma unroll
        for (int j = 0; j < 3; ++j)
          store_act(p.conv_dst, ((size_t)n * 3 + j) * p.Cch + chan(c), s_hist[j][c], p.in_bf16);
  }
}

template <int D>
cudaError_t launch(const RecurParams &p, cudaStream_t stream) {
  const unsigned units = (unsigned)p.N * (unsigned)p.H;
  recurrent_kernel<D><<<units, Shape<D>::NT, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

glinattn_status launch_recurrent(const RecurParams &p, int d, cudaStream_t stream) {
  if ((long long)p.N * p.H == 0) return GLINATTN_OK;
  cudaError_t e;
  switch (d) {
    case 16: e = launch<16>(p, stream); break;
    case 32: e = launch<32>(p, stream); break;
    case 64: e = launch<64>(p, stream); break;
    case 128: e = launch<128>(p, stream); break;
    default: return GLINATTN_ERR_UNSUPPORTED;
  }
  return e == cudaSuccess ? GLINATTN_OK : GLINATTN_ERR_CUDA;
}

}  // namespace glinattn
