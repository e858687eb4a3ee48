// verify128.cu -- the outputs of D draft tokens from one read of the start
// state: verify-only speculative decode for 128 x 128 fp32 head states.
//
// "Inference for linear attention and hybrid architectures", section
// "Speculative decoding and PD disaggregation": verifying D draft tokens is a
// prefill of D tokens from the request's state, and section "Two ways to
// write the same computation" gives that prefill in chunked form.  With the
// draft tokens as one chunk of C = D tokens from start state S, g the
// cumulative log decay, gamma = exp(g) and D_ij = exp(g_i - g_j) [j <= i]:
//   GLA:  O = diag(gamma) Q S + ((Q K^T) * D) V
//   GDN:  (I + A) U = diag(beta) V - diag(beta gamma) K S,
//         A_ij = beta_i D_ij (k_i . k_j) for j < i,
//         O = diag(gamma) Q S + ((Q K^T) * D) U
// so the state is read once and enters only through the 2D row products Q S
// and K S, where the per-step form reads it D times and rewrites it D - 1
// times.  The outputs equal those of D decode steps up to fp32 rounding; the
// per-step form remains the one that writes states (spec decode with one
// state per draft, replay), whose states are bit-identical to decode steps.
//
// Kernel design (sm_103a): one CTA of 256 threads per (request, head) unit.
// Warp w keeps rows 16w .. 16w + 15 of the state in registers (lane = a
// 16-byte column group), loaded with coalesced 512-byte rows before the front
// end runs.  The front end (width-4 causal convolution over the conv cache
// and the earlier drafts, L2 norm, bf16 rounding) is the decode kernel's
// arithmetic in the decode kernel's order: thread t owns q channel t (t <
// 128) or k channel t - 128, and threads t < 128 also v channel t, so the
// pairwise sums of squares run over the same lanes and warps.  The D x D
// scalars (Gram products, the unit-lower inverse by forward substitution,
// the decay factors) are formed by single warps; each of the 128 columns then
// needs only O(D^2) scalar work.
#include <cuda_bf16.h>

#include "common.cuh"
#include "frontend.cuh"

namespace glinattn {
namespace {

constexpr int kD = 128;
constexpr int kVT = 256;       // threads per CTA
constexpr int kMaxD = 16;      // drafts per call handled here
constexpr int kG = 4;          // drafts per pass of the row products

// shared memory, in floats
constexpr int kOffAct = 0;                            // [kMaxD][3 kD]: q | k | v after the front end
constexpr int kOffWsum = kOffAct + kMaxD * 3 * kD;    // [kMaxD][8]: sums of squares per warp
constexpr int kOffRed = kOffWsum + kMaxD * 8;         // [8 warps][2 kG][kD]: row-product partials
constexpr int kOffKS = kOffRed + 8 * 2 * kG * kD;     // [kMaxD][kD]: K S
constexpr int kOffQS = kOffKS + kMaxD * kD;           // [kMaxD][kD]: Q S
constexpr int kOffGkk = kOffQS + kMaxD * kD;          // [kMaxD][kMaxD]: k_i . k_j
constexpr int kOffGqk = kOffGkk + kMaxD * kMaxD;      // [kMaxD][kMaxD]: q_i . k_j
constexpr int kOffT = kOffGqk + kMaxD * kMaxD;        // [kMaxD][kMaxD]: (I + A)^-1
constexpr int kOffP = kOffT + kMaxD * kMaxD;          // [kMaxD][kMaxD]: (q_i . k_j) D_ij
constexpr int kOffGam = kOffP + kMaxD * kMaxD;        // [kMaxD]: gamma
constexpr int kOffBet = kOffGam + kMaxD;              // [kMaxD]: beta
constexpr int kSmemFloats = kOffBet + kMaxD;
// before the row products, the reduction buffer holds the unit's raw inputs,
// copied in with cp.async at the start: D rows of q | k | v, the conv history
// (3 rows of q | k | v) and the D gates alpha, beta (as raw bytes, bf16 or fp32)
constexpr int kRawRow = 3 * kD;                               // elements per row
constexpr int kOffRawX = kOffRed;                             // [kMaxD][3 kD] elements
constexpr int kOffRawH = kOffRawX + kMaxD * kRawRow;          // [3][3 kD] elements (fp32 worst case)
constexpr int kOffRawG = kOffRawH + 3 * kRawRow;              // alpha [kMaxD], beta [kMaxD] (fp32)
static_assert(kOffRawG + 2 * kMaxD <= kOffRed + 8 * 2 * kG * kD, "raw inputs fit the reduction buffer");

__device__ __forceinline__ float ld_in(const void *base, size_t idx, int bf16) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[idx]);
  return reinterpret_cast<const float *>(base)[idx];
}

__device__ __forceinline__ void cp16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_commit_wait() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void st_out(void *base, size_t idx, float x, int bf16) {
  if (bf16)
    reinterpret_cast<__nv_bfloat16 *>(base)[idx] = __float2bfloat16_rn(x);
  else
    reinterpret_cast<float *>(base)[idx] = x;
}

template <bool kGdn>
__global__ void __launch_bounds__(kVT, 2) verify128_kernel(const RecurParams p) {
  extern __shared__ __align__(16) float vsm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H, D = p.steps;
  const int n = blockIdx.x / H, h = blockIdx.x - n * H;
  const int slot = p.src_slot[n];

  // ---- the slot (uniform); a slot outside the pool skips the unit ---------------
  if (slot < 0 || slot >= p.pool_slots) {
    if (tid == 0 && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_BAD_SLOT);
    return;
  }
  const int in_bf16 = p.in_bf16, esz = in_bf16 ? 2 : 4;
  const bool conv = p.conv_w != nullptr;

  // ---- raw inputs into shared memory (cp.async), then the state's rows ---------
  // 16-byte pieces: D token rows and 3 history rows of q | k | v, each part
  // kD elements (16 pieces of bf16 or 32 of fp32)
  {
    uint8_t *rawx = reinterpret_cast<uint8_t *>(vsm + kOffRawX);
    uint8_t *rawh = reinterpret_cast<uint8_t *>(vsm + kOffRawH);
    const int ppp = kD * esz / 16;        // pieces per part
    const int rows = D + (conv ? 3 : 0);  // token rows, then history rows
    for (int e = tid; e < rows * 3 * ppp; e += kVT) {
      const int r = e / (3 * ppp), part = (e / ppp) % 3, pc = e % ppp;
      if (r < D) {
        const size_t row = ((size_t)n * D + r) * H + h;
        const uint8_t *src = reinterpret_cast<const uint8_t *>(part == 0 ? p.q : part == 1 ? p.k : p.v) +
                             (row * kD) * esz + pc * 16;
        cp16(rawx + ((size_t)r * kRawRow + part * kD) * esz + pc * 16, src);
      } else {
        const int j = r - D;
        const uint8_t *src = reinterpret_cast<const uint8_t *>(p.conv_src) +
                             (((size_t)slot * 3 + j) * p.Cch + part * H * kD + h * kD) * esz + pc * 16;
        cp16(rawh + ((size_t)j * kRawRow + part * kD) * esz + pc * 16, src);
      }
    }
    float *rawg = vsm + kOffRawG;
    if (tid < D) cp4(&rawg[tid], &p.alpha[((size_t)n * D + tid) * H + h]);
    else if (kGdn && tid >= 32 && tid < 32 + D)
      cp4(&rawg[kMaxD + tid - 32], &p.beta[((size_t)n * D + tid - 32) * H + h]);
  }
  // the state's rows 16 warp .. + 15, columns 4 lane .. + 3 (in flight meanwhile)
  float4 S[16];
  {
    const float4 *src = reinterpret_cast<const float4 *>(p.S_src + ((size_t)slot * H + h) * kD * kD);
#pragma unroll
    for (int r = 0; r < 16; ++r) S[r] = src[(16 * warp + r) * (kD / 4) + lane];
  }
  cp_commit_wait();
  __syncthreads();

  // ---- the gates in (0, 1] (uniform); a bad gate skips the unit ------------------
  {
    const float a = tid < D ? vsm[kOffRawG + tid] : 1.f;
    if (__syncthreads_or(!(a > 0.f && a <= 1.f))) {
      if (tid == 0 && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_BAD_GATE);
      return;
    }
  }

  // ---- front end: thread t owns q / k channel t and (t < 128) v channel t ------
  {
    const bool round_act = in_bf16 && (conv || p.qk_l2norm);
    // local channels of this thread: a (q or k) and, for t < 128, v
    const int ca = tid, cv = 2 * kD + tid;
    const bool has_v = tid < kD;
    auto gch = [&](int c) {  // the channel's row in the conv weights
      return c < 2 * kD ? (c / kD) * H * kD + h * kD + (c % kD) : 2 * H * kD + h * kD + (c - 2 * kD);
    };
    const void *rawx = vsm + kOffRawX, *rawh = vsm + kOffRawH;
    float wa[4] = {0.f, 0.f, 0.f, 1.f}, wv[4] = {0.f, 0.f, 0.f, 1.f};
    float ha[3] = {0.f, 0.f, 0.f}, hv[3] = {0.f, 0.f, 0.f};
    if (conv) {
      const float4 a4 = *reinterpret_cast<const float4 *>(p.conv_w + (size_t)gch(ca) * 4);
      wa[0] = a4.x; wa[1] = a4.y; wa[2] = a4.z; wa[3] = a4.w;
      if (has_v) {
        const float4 v4 = *reinterpret_cast<const float4 *>(p.conv_w + (size_t)gch(cv) * 4);
        wv[0] = v4.x; wv[1] = v4.y; wv[2] = v4.z; wv[3] = v4.w;
      }
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        ha[j] = ld_in(rawh, j * kRawRow + ca, in_bf16);
        if (has_v) hv[j] = ld_in(rawh, j * kRawRow + cv, in_bf16);
      }
    }
    float *act = vsm + kOffAct;
    // tokens in groups of 8: their squares summed over the lanes together
    // (the same pairwise tree per token as one reduction each)
    for (int t0 = 0; t0 < D; t0 += 8) {
      float sq[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int t = t0 + k;
        sq[k] = 0.f;
        if (t < D) {
          const float xa = ld_in(rawx, t * kRawRow + ca, in_bf16);
          const float ya = conv ? fe::conv4(wa[0], wa[1], wa[2], wa[3], ha[0], ha[1], ha[2], xa) : xa;
          ha[0] = ha[1];
          ha[1] = ha[2];
          ha[2] = xa;
          act[t * 3 * kD + ca] = ya;
          sq[k] = __fmul_rn(ya, ya);
          if (has_v) {
            const float xv = ld_in(rawx, t * kRawRow + cv, in_bf16);
            const float yv = conv ? fe::conv4(wv[0], wv[1], wv[2], wv[3], hv[0], hv[1], hv[2], xv) : xv;
            hv[0] = hv[1];
            hv[1] = hv[2];
            hv[2] = xv;
            act[t * 3 * kD + cv] = round_act ? __bfloat162float(__float2bfloat16_rn(yv)) : yv;
          }
        }
      }
      if (p.qk_l2norm) {  // pairwise sums of squares: lanes, then the 4 warps of q (or k)
        const float r = fe::warp_pairwise_sum8(sq, lane);
        const int row = 4 * (lane & 1) + 2 * ((lane >> 1) & 1) + ((lane >> 2) & 1);  // the row lane l holds
        if (lane < 8 && t0 + row < D) vsm[kOffWsum + (t0 + row) * 8 + warp] = r;
      }
    }
    __syncthreads();
    // the inverse norms, once per token: warp 0, lane t (q) and 16 + t (k)
    float *s_inv = vsm + kOffKS;  // free until the row products
    if (p.qk_l2norm && warp == 0 && (lane & 15) < D) {
      const int t = lane & 15;
      s_inv[lane] = fe::inv_norm(fe::pairwise_sum<4>(vsm + kOffWsum + t * 8 + (lane < 16 ? 0 : 4)));
    }
    if (p.qk_l2norm) __syncthreads();
    for (int t = 0; t < D; ++t) {
      float y = act[t * 3 * kD + ca];
      const float inv = p.qk_l2norm ? s_inv[(ca < kD ? 0 : 16) + t] : 1.f;
      y = __fmul_rn(y, inv);
      if (round_act) y = __bfloat162float(__float2bfloat16_rn(y));
      act[t * 3 * kD + ca] = y;
    }
  }
  // the gates of draft `lane` (warp 0 uses them below; the raw area is reused)
  const float ga = lane < D ? vsm[kOffRawG + lane] : 1.f;
  const float gb = kGdn && lane < D ? vsm[kOffRawG + kMaxD + lane] : 0.f;
  __syncthreads();
  const float *act = vsm + kOffAct;

  // ---- Gram products k_i . k_j and q_i . k_j (j <= i): a warp per pair ---------
  for (int pi = warp; pi < D * D; pi += kVT / 32) {
    const int i = pi / D, j = pi - (pi / D) * D;
    if (j > i) continue;
    float sqk = 0.f, skk = 0.f;
#pragma unroll
    for (int c = lane; c < kD; c += 32) {
      const float kj = act[j * 3 * kD + kD + c];
      sqk = fmaf(act[i * 3 * kD + c], kj, sqk);
      skk = fmaf(act[i * 3 * kD + kD + c], kj, skk);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sqk += __shfl_xor_sync(0xffffffffu, sqk, o);
      skk += __shfl_xor_sync(0xffffffffu, skk, o);
    }
    if (lane == 0) {
      vsm[kOffGqk + i * kMaxD + j] = sqk;
      vsm[kOffGkk + i * kMaxD + j] = skk;
    }
  }

  // ---- K S and Q S: this warp's 16 rows, then the sum over the 8 warps --------
  for (int g0 = 0; g0 < D; g0 += kG) {
    // fused multiply-adds on column pairs (two lanes of one instruction)
    float2 kp[kG][2], qp[kG][2];
#pragma unroll
    for (int i = 0; i < kG; ++i)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) kp[i][h2] = qp[i][h2] = make_float2(0.f, 0.f);
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int row = 16 * warp + r;
      const float2 s01 = make_float2(S[r].x, S[r].y), s23 = make_float2(S[r].z, S[r].w);
#pragma unroll
      for (int i = 0; i < kG; ++i) {
        const int t = g0 + i < D ? g0 + i : D - 1;  // past D: a repeat, never used
        const float kv = act[t * 3 * kD + kD + row], qv = act[t * 3 * kD + row];
        const float2 k2 = make_float2(kv, kv), q2 = make_float2(qv, qv);
        kp[i][0] = __ffma2_rn(k2, s01, kp[i][0]);
        kp[i][1] = __ffma2_rn(k2, s23, kp[i][1]);
        qp[i][0] = __ffma2_rn(q2, s01, qp[i][0]);
        qp[i][1] = __ffma2_rn(q2, s23, qp[i][1]);
      }
    }
    float4 *red4 = reinterpret_cast<float4 *>(vsm + kOffRed);
#pragma unroll
    for (int i = 0; i < kG; ++i) {
      red4[((warp * 2 * kG) + 2 * i) * (kD / 4) + lane] = make_float4(kp[i][0].x, kp[i][0].y, kp[i][1].x, kp[i][1].y);
      red4[((warp * 2 * kG) + 2 * i + 1) * (kD / 4) + lane] = make_float4(qp[i][0].x, qp[i][0].y, qp[i][1].x, qp[i][1].y);
    }
    __syncthreads();
    // the sums over the warps; in the last group warp 0 forms the D x D scalars
    // (lane = draft) meanwhile and warps 1-7 add
    const bool last = g0 + kG >= D;
    if (last && warp == 0) {
      const float a = lane < D ? ga : 1.f;
      float g = log2f(a);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, g, o);
        if (lane >= o) g += y;
      }
      if (lane < D) {
        vsm[kOffGam + lane] = exp2f(g);
        vsm[kOffBet + lane] = kGdn ? gb : 0.f;
      }
      // P_ij = (q_i . k_j) 2^(g_i - g_j) for j <= i: lane j of row i
      for (int i = 0; i < D; ++i) {
        const float gi = __shfl_sync(0xffffffffu, g, i);
        if (lane <= i) vsm[kOffP + i * kMaxD + lane] = vsm[kOffGqk + i * kMaxD + lane] * exp2f(gi - g);
      }
      if (kGdn) {
        // A_ij = beta_i 2^(g_i - g_j) (k_i . k_j), j < i; T = (I + A)^-1 by forward
        // substitution, lane = column j: x = e_j, then x_m -= A_mi x_i for m > i
        const float bl = lane < D ? gb : 0.f;
        float x[kMaxD];
#pragma unroll
        for (int m = 0; m < kMaxD; ++m) x[m] = m == lane ? 1.f : 0.f;
#pragma unroll
        for (int i = 0; i < kMaxD; ++i) {
          if (i >= D) break;
          const float gi = __shfl_sync(0xffffffffu, g, i);
#pragma unroll
          for (int m = i + 1; m < kMaxD; ++m) {
            if (m >= D) break;
            const float gm = __shfl_sync(0xffffffffu, g, m), bm = __shfl_sync(0xffffffffu, bl, m);
            const float amj = bm * exp2f(gm - gi) * vsm[kOffGkk + m * kMaxD + i];
            x[m] = fmaf(-amj, x[i], x[m]);
          }
        }
#pragma unroll
        for (int m = 0; m < kMaxD; ++m)
          if (m < D && lane < D) vsm[kOffT + m * kMaxD + lane] = x[m];
      }
    } else {
      const int e0 = last ? tid - 32 : tid, step = last ? kVT - 32 : kVT;
      for (int e = e0; e < 2 * kG * kD; e += step) {
        const int v = e / kD, c = e - (e / kD) * kD, t = g0 + v / 2;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += vsm[kOffRed + (w * 2 * kG + v) * kD + c];
        if (t < D) vsm[((v & 1) ? kOffQS : kOffKS) + t * kD + c] = s;
      }
    }
    __syncthreads();
  }

  // ---- outputs: column c, drafts of parity tid >> 7 ---------------------------------
  {
    const int c = tid & (kD - 1), par = tid >> 7;
    float u[kMaxD];
#pragma unroll
    for (int j = 0; j < kMaxD; ++j) {
      if (j >= D) break;
      const float vj = act[j * 3 * kD + 2 * kD + c];
      if (kGdn) {
        // U_j = sum over m <= j of T_jm beta_m (v_m - gamma_m (K S)_m)
        float s = 0.f;
        for (int m = 0; m <= j; ++m) {
          const float bm = vsm[kOffBet + m];
          const float rhs = bm * (act[m * 3 * kD + 2 * kD + c] - vsm[kOffGam + m] * vsm[kOffKS + m * kD + c]);
          s = fmaf(vsm[kOffT + j * kMaxD + m], rhs, s);
        }
        u[j] = s;
      } else {
        u[j] = vj;
      }
    }
#pragma unroll
    for (int i = 0; i < kMaxD; ++i) {
      if (i >= D) break;
      if ((i & 1) != par) continue;
      float o = vsm[kOffGam + i] * vsm[kOffQS + i * kD + c];
#pragma unroll
      for (int j = 0; j < kMaxD; ++j) {
        if (j > i) break;
        o = fmaf(vsm[kOffP + i * kMaxD + j], u[j], o);
      }
      st_out(p.o, (((size_t)n * D + i) * H + h) * kD + c, o, p.out_bf16);
    }
  }
}

}  // namespace

bool verify128_supports(const RecurParams &p, int d) {
  return d == kD && (p.variant == GLINATTN_GLA || p.variant == GLINATTN_GDN) && p.S_dst == nullptr &&
         p.dst_slot == nullptr && p.step_count == nullptr && p.o != nullptr && p.src_slot != nullptr &&
         p.S_src != nullptr && p.steps >= 1 && p.steps <= kMaxD && p.pool_slots > 0 && p.Hq == p.H &&
         (p.conv_w == nullptr || p.conv_src != nullptr) && p.S_blocks == nullptr && p.alpha != nullptr &&
         (p.variant != GLINATTN_GDN || p.beta != nullptr) && ((uintptr_t)p.S_src & 15u) == 0;
}

cudaError_t launch_verify128(const RecurParams &p, cudaStream_t stream) {
  const int bytes = kSmemFloats * 4;
  auto kernel = p.variant == GLINATTN_GDN ? verify128_kernel<true> : verify128_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  kernel<<<(unsigned)((long long)p.N * p.H), kVT, bytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace glinattn
