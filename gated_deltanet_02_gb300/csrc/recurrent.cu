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
// One CTA owns one (request, head) state, d x d fp32.  Its source is fetched
// into shared memory by a single bulk copy (cp.async.bulk) issued as soon as
// the slot id is known, so the copy engine moves the 64 KiB while the threads
// run the front end (short convolution, L2 norm); registers stay low enough
// for two CTAs per SM, i.e. two states in flight per SM besides the stores.
// Thread (rg, cg) owns rows rg + ROWG*i of column group cg (4 consecutive
// columns, one 16-byte vector), so every warp-wide access to a state row is
// contiguous, in shared and in global memory.  k S and q S are reduced in one
// pass, across row groups through shared memory in a fixed order
// (deterministic, no atomics).  Decode (1 step, in place) and speculative
// decode (D steps, a write after each) run this same code, so a draft state
// equals the state of repeated decode steps bit for bit.
#include "common.cuh"
#include "sm100.cuh"

namespace glinattn {
namespace {

using namespace sm100;

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
  constexpr uint32_t kStateBytes = D * D * 4;
  const int unit = blockIdx.x;
  const int n = unit / p.H, h = unit - n * p.H;
  const int tid = threadIdx.x;
  const int cg = tid % Sh::COLG, rg = tid / Sh::COLG;
  const size_t DD = (size_t)D * D;

  extern __shared__ __align__(128) float4 s_state4[];  // the d x d state, row-major
  __shared__ float s_act[3 * D];                        // q | k | v after the front end
  __shared__ float s_raw[3 * D];                        // raw inputs of the current token
  __shared__ float s_hist[3][3 * D];                    // conv history, oldest first
  __shared__ float s_red[Sh::ROWG][2][D];
  __shared__ float s_wsum[2][NW];
  __shared__ float s_qk;
  __shared__ int s_bad, s_has_src;
  __shared__ __align__(8) uint64_t s_bar;

  // ---- thread 0 checks the source slot and starts the state copy at once ----
  if (tid == 0) {
    int bad0 = 0;
    const float *src = nullptr;
    if (p.S_src) {
      size_t slot = (size_t)n;
      if (p.src_slot) {
        const int s = p.src_slot[n];
        if (p.pool_slots > 0 && (s < 0 || s >= p.pool_slots)) bad0 = GLINATTN_DEV_BAD_SLOT;
        slot = (size_t)s;
      }
      if (!bad0) src = p.S_src + (slot * p.H + h) * DD;
    }
    mbar_init(&s_bar, 1);
    fence_mbar_init();
    if (src) {
      mbar_arrive_expect_tx(&s_bar, kStateBytes);
      bulk_load(s_state4, src, kStateBytes, &s_bar);
    }
    s_bad = bad0;
    s_has_src = src != nullptr;
  }
  __syncthreads();

  // ---- the rest of the unit validation: destination slots, gates in (0, 1] --
  int bad = 0;
  if (p.pool_slots > 0 && p.dst_slot) {
    const int nd = p.dst_per_step ? p.steps : 1;
    for (int t = tid; t < nd; t += Sh::NT) {
      const int s = p.dst_slot[(size_t)n * nd + t];
      if (s < 0 || s >= p.pool_slots) bad |= GLINATTN_DEV_BAD_SLOT;
    }
  }
  for (int t = tid; t < p.steps; t += Sh::NT) {
    const float a = p.alpha[((size_t)n * p.steps + t) * p.H + h];
    if (!(a > 0.f && a <= 1.f)) bad |= GLINATTN_DEV_BAD_GATE;
  }
  if (bad) atomicOr(&s_bad, bad);
  __syncthreads();
  const bool has_src = s_has_src != 0;
  if (s_bad) {
    if (has_src) mbar_wait(&s_bar, 0);  // let the copy land before the CTA exits
    if (tid == 0 && p.dev_status) atomicOr(p.dev_status, (uint32_t)s_bad);
    return;
  }
  if (!has_src) {
#pragma unroll
    for (int i = 0; i < Sh::RPT; ++i)
      s_state4[(rg + Sh::ROWG * i) * Sh::COLG + cg] = make_float4(0.f, 0.f, 0.f, 0.f);
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
    if (t == 0 && has_src) {  // the state copy must have landed
      const bool ok = mbar_wait(&s_bar, 0);
      if (!__syncthreads_and(ok)) {
        if (tid == 0 && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_WAIT_TIMEOUT);
        return;
      }
    } else {
      __syncthreads();
    }

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
      const float4 S = s_state4[r * Sh::COLG + cg];
      const float kr = sk[r], qr = sq[r];
      x.x += kr * S.x; x.y += kr * S.y; x.z += kr * S.z; x.w += kr * S.w;
      y.x += qr * S.x; y.y += qr * S.y; y.z += qr * S.z; y.w += qr * S.w;
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

    // ---- update: shared memory copy for the next step, global copy if due ------
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
    const bool last = (t == p.steps - 1);
    const bool emit = p.dst_per_step || last;
    float *dst = nullptr;
    size_t dslot = (size_t)n;
    if (emit) {
      if (p.dst_slot)
        dslot = (size_t)p.dst_slot[(size_t)n * (p.dst_per_step ? p.steps : 1) + (p.dst_per_step ? t : 0)];
      dst = p.S_dst + (dslot * p.H + h) * DD;
    }
#pragma unroll
    for (int i = 0; i < Sh::RPT; ++i) {
      const int r = rg + Sh::ROWG * i;
      const float kr = sk[r];
      float4 S = s_state4[r * Sh::COLG + cg];
      S.x = a * S.x + kr * u.x;
      S.y = a * S.y + kr * u.y;
      S.z = a * S.z + kr * u.z;
      S.w = a * S.w + kr * u.w;
      if (!last) s_state4[r * Sh::COLG + cg] = S;
      if (emit) *reinterpret_cast<float4 *>(dst + (size_t)r * D + 4 * cg) = S;
    }
    if (rg == 0) {
      const float qk = s_qk;
      const size_t ob = row * D + 4 * cg;
      store_act(p.o, ob + 0, a * y.x + qk * u.x, p.out_bf16);
      store_act(p.o, ob + 1, a * y.y + qk * u.y, p.out_bf16);
      store_act(p.o, ob + 2, a * y.z + qk * u.z, p.out_bf16);
      store_act(p.o, ob + 3, a * y.w + qk * u.w, p.out_bf16);
    }
    if (emit && conv && p.conv_dst) {
      __syncthreads();  // s_hist shift complete
      for (int c = tid; c < 3 * D; c += Sh::NT)
#pragma unroll
        for (int j = 0; j < 3; ++j)
          store_act(p.conv_dst, (dslot * 3 + j) * p.Cch + chan(c), s_hist[j][c], p.in_bf16);
    }
    __syncthreads();  // shared buffers are rewritten by the next step
  }

  if (p.steps == 0) {  // a zero-length segment hands its inputs straight on
    if (has_src && !mbar_wait(&s_bar, 0)) {
      if (tid == 0 && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_WAIT_TIMEOUT);
      return;
    }
    __syncthreads();
    float *dst = p.S_dst + ((size_t)n * p.H + h) * DD;
#pragma unroll
    for (int i = 0; i < Sh::RPT; ++i) {
      const int r = rg + Sh::ROWG * i;
      *reinterpret_cast<float4 *>(dst + (size_t)r * D + 4 * cg) = s_state4[r * Sh::COLG + cg];
    }
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
  constexpr int smem = D * D * 4;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(recurrent_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  recurrent_kernel<D><<<units, Shape<D>::NT, smem, stream>>>(p);
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
