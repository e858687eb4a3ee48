// gdn_tc.cu -- chunked Gated DeltaNet prefill on the 5th-generation tensor cores.
//
// "Inference for linear attention and hybrid architectures", section "Two
// ways to write the same computation": DeltaNet's chunked form must first
// write the error-correcting updates inside a chunk in matrix form.  With the
// recurrence S_t = alpha_t S_{t-1} + k_t^T u_t, u_t = beta_t (v_t - alpha_t k_t
// S_{t-1}) and, inside a chunk with start state S, g = cumulative log decay,
// gamma = exp(g), D_ij = exp(g_i - g_j) [j <= i], r_j = exp(g_C - g_j):
//
//   (I + A) U = diag(beta) V - diag(beta gamma) K S,
//        A_ij = beta_i D_ij (k_i . k_j) for j < i
//   U = U~ - W S,  U~ = (I+A)^-1 diag(beta) V,  W = (I+A)^-1 diag(beta gamma) K
//   O      = diag(gamma) Q S + ((Q K^T) * D) U
//   S_next = gamma_C S + K^T diag(r) U
//
// Everything but U - W S is independent of the state, so the work is split:
//
//   pass A (gdn_prep_kernel), one CTA per (batch, head, chunk), all chunks in
//     parallel: the front end (short causal convolution, L2 norm of q and k,
//     rounding to bf16), [Q; K] K^T as one M = 128 MMA, A, the unit-lower
//     inverse (I + A)^-1 in fp32, and W and U~ as MMAs.  Q', K', W (bf16), U~
//     (fp32) and the log2 gates go to a caller-provided workspace.
//   pass B (gdn_scan_kernel), one CTA per (batch, head, 32-wide d_v slice),
//     serial over chunks with the fp32 state in registers: U = U~ - W S, the
//     outputs and the state carry.  The two output terms share one
//     accumulator, O = c_i (Q' S + P'' U) with P''_ij = (Q'K'^T)_ij
//     exp(g_i - g_j) / c_i and the row scale c_i = gamma_i (2^-100 for a row
//     whose own decay is below that: its Q' S term then carries 2^-100 in
//     place of gamma_i, a difference below 2^-100 |Q' S|).  Three threads
//     issue MMAs: one the state chain (W S, K'^T r U), one Q'K'^T as soon as
//     a chunk lands, one the outputs -- Q'S once W S of the chunk is done and
//     P''U once K'^T r U is done, so the chain's MMAs never wait behind the
//     outputs' in the tensor pipe.  The M = 64 accumulators are read with the
//     16x256b TMEM shape (every lane of a warp holds two rows).
//
// Operands derived in fp32 (S, P'', U, r U, the inverse) enter the MMAs as a
// bf16 high part plus a bf16 remainder.
#include <cuda.h>
#include <cuda_bf16.h>
#include <string.h>

#include "common.cuh"
#include "frontend.cuh"
#include "prefill_tc.cuh"
#include "sm100.cuh"
#include "tc_common.cuh"

namespace glinattn {
namespace {

using namespace sm100;
using namespace tc;

constexpr int kC = 64;   // chunk length
constexpr int kD = 128;  // head size (d_k = d_v)

// 1024-byte aligned pointer into the shared array, derived by pointer
// arithmetic so the compiler keeps accesses through it in the shared space.
__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

// ================================ pass A ====================================

constexpr int kPrepThreads = 256;
constexpr int kBlk = 32;                         // the inverse works on 32 x 32 blocks
constexpr uint32_t kBlkBytes = kBlk * (kBlk + 1) * 4;  // one fp32 block, rows padded to 33
constexpr uint32_t kOffRaw = 0;                  // the chunk's raw q, k, v rows: 3 x 2 swizzled 8 KiB blocks
constexpr uint32_t kRawBytes = 3 * 16384;        // (dead after the front end; A, T, Tm reuse it)
constexpr uint32_t kOffA = 0;                    // A00, A10, A11 (A00 later holds X = A10 T00)
constexpr uint32_t kOffT = 3 * kBlkBytes;        // T00, T10, T11 of T = (I + A)^-1
constexpr uint32_t kOffTm = 25600;               // T diag(beta gamma) hi, lo and T diag(beta) hi, lo: 4 x 8 KiB
constexpr uint32_t kOffQK = 61440;               // stacked [Q'; K']: 2 column blocks x 128 rows x 128 B
constexpr uint32_t kOffVp = kOffQK + 32768;      // V': 2 column blocks x 64 rows x 128 B
constexpr uint32_t kOffMisc = kOffVp + 16384;    // g2[64], beta[64], barrier, TMEM slot
constexpr uint32_t kPrepSmem = kOffMisc + 1024 + 1024;
static_assert(kOffT + 3 * kBlkBytes <= kOffTm && kOffTm + 4 * 8192 <= kOffQK, "pass A layout");
static_assert(kOffRaw + kRawBytes <= kOffQK, "raw tile");
static_assert(kOffQK % 1024 == 0 && kOffVp % 1024 == 0 && kOffTm % 1024 == 0, "alignment");

struct PrepParams {
  int B, T, H, nchunks, Tp, qk_l2norm, has_conv;
  const __nv_bfloat16 *q, *k, *v;
  const float *alpha, *beta, *conv_w;
  const __nv_bfloat16 *conv_in;
  __nv_bfloat16 *Qp, *Kp, *Wp;  // [B*H, Tp, 128]
  float *Up;                    // [B*H, Tp, 128]
  float *Gp;                    // [B*H, Tp]
  uint32_t *dev_status;
};

// kConv, kL2: the front end's convolution and L2 norm as template parameters
// (one code path per instance)
template <bool kConv, bool kL2>
__global__ void __launch_bounds__(kPrepThreads)
    gdn_prep_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const PrepParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = c * kC, H = p.H, T = p.T;
  const int Cch = 3 * H * kD;
  const size_t unit = (size_t)b * H + h;
  float *g2s = reinterpret_cast<float *>(smem + kOffMisc);
  float *betas = g2s + kC;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kOffMisc + 512);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + kOffMisc + 520);
  uint64_t *bar_raw = reinterpret_cast<uint64_t *>(smem + kOffMisc + 528);
  float *colbg = reinterpret_cast<float *>(smem + kOffMisc + 768);  // beta_k 2^g_k, 64 columns
  uint8_t *raw = smem + kOffRaw;

  // the chunk's 64 raw rows of q, k and v by TMA (rows past T arrive as zeros)
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(bar_raw, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar_raw, kRawBytes);
    const CUtensorMap *maps[3] = {&tq, &tk, &tv};
#pragma unroll
    for (int part = 0; part < 3; ++part)
#pragma unroll
      for (int blk = 0; blk < 2; ++blk)
        tma_load_4d(raw + part * 16384 + blk * 8192, maps[part], bar_raw, 64 * blk, h, t0, b);
  }
  if (warp == 0) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  __syncthreads();  // both mbarriers are initialised before any thread waits on them

  // ---- front end: y_t = sum_j w_j x_{t-3+j}; L2 norm of q, k rows; bf16 -------
  // A task is (part, 8 consecutive tokens) of the chunk: a warp slides the
  // 4-tap window along its tokens, lane l owning channels 4l .. 4l+3, so every
  // access is 8 bytes per lane and the L2 norm is one warp reduction.  The
  // chunk's rows come from the TMA tile; the 3 rows before the chunk (first
  // task of each part only) from global memory, or conv_in before the
  // sequence (zero without it).
  struct FeTask {
    uint2 hist[3];  // rows -3, -2, -1 of the chunk when r0 == 0
    float4 w[4];    // the 4 taps of channels 4l .. 4l+3
  };
  auto fe_load = [&](int task, FeTask &f) {
    const int part = task % 3, r0 = (task / 3) * 8;
    const __nv_bfloat16 *src = part == 0 ? p.q : (part == 1 ? p.k : p.v);
#pragma unroll
    for (int m = 0; m < 3; ++m) {
      const int t = t0 - 3 + m;
      uint2 v = make_uint2(0u, 0u);
      if (r0 == 0) {
        if (t >= 0)
          v = *reinterpret_cast<const uint2 *>(src + (((size_t)b * T + t) * H + h) * kD + 4 * lane);
        else if (kConv && p.conv_in)
          v = *reinterpret_cast<const uint2 *>(p.conv_in + ((size_t)b * 3 + (t + 3)) * Cch + part * H * kD +
                                               h * kD + 4 * lane);
      }
      f.hist[m] = v;
    }
#pragma unroll
    for (int c2 = 0; c2 < 4; ++c2)
      f.w[c2] = kConv ? *reinterpret_cast<const float4 *>(
                                 p.conv_w + ((size_t)part * H * kD + h * kD + 4 * lane + c2) * 4)
                           : make_float4(0.f, 0.f, 0.f, 1.f);
  };
  uint8_t *qk = smem + kOffQK;
  uint8_t *vp = smem + kOffVp;
  auto fe_compute = [&](int task, const FeTask &f) {
    const int part = task % 3, r0 = (task / 3) * 8;
    // channels 4l .. 4l+3: column block l / 16, 16-byte chunk (l % 16) / 2, half l % 2
    const uint32_t cb = (uint32_t)(lane >> 4), ch = (uint32_t)((lane & 15) >> 1), hb = (uint32_t)(lane & 1) * 8;
    uint2 xrow[11];  // rows r0 - 3 .. r0 + 7
#pragma unroll
    for (int m = 0; m < 11; ++m) {
      const int tr = r0 - 3 + m;
      xrow[m] = tr >= 0 ? *reinterpret_cast<const uint2 *>(raw + part * 16384 + cb * 8192 + swz(tr, ch) + hb)
                        : f.hist[m < 3 ? m : 0];
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float y[4];
#pragma unroll
      for (int c2 = 0; c2 < 4; ++c2) {
        // bf16 channel c2 of row m: low or high half of word c2 / 2
        auto xv = [&](int m) {
          const uint32_t wd = (c2 >> 1) ? xrow[m].y : xrow[m].x;
          return __uint_as_float((c2 & 1) ? (wd & 0xffff0000u) : (wd << 16));
        };
        const float4 wc = f.w[c2];
        y[c2] = fe::conv4(wc.x, wc.y, wc.z, wc.w, xv(r), xv(r + 1), xv(r + 2), xv(r + 3));
      }
      if (part < 2 && kL2) {
        // pairwise sum of squares: this lane's 4 channels, then adjacent lanes
        const float ss = fe::warp_pairwise_sum(__fadd_rn(__fadd_rn(__fmul_rn(y[0], y[0]), __fmul_rn(y[1], y[1])),
                                                         __fadd_rn(__fmul_rn(y[2], y[2]), __fmul_rn(y[3], y[3]))));
        const float inv = fe::inv_norm(ss);
#pragma unroll
        for (int c2 = 0; c2 < 4; ++c2) y[c2] = __fmul_rn(y[c2], inv);
      }
      const bool valid = t0 + r0 + r < T;
      uint2 pk;
      pk.x = bits(__floats2bfloat162_rn(valid ? y[0] : 0.f, valid ? y[1] : 0.f));
      pk.y = bits(__floats2bfloat162_rn(valid ? y[2] : 0.f, valid ? y[3] : 0.f));
      const int t = r0 + r;
      if (part < 2)
        *reinterpret_cast<uint2 *>(qk + cb * 16384 + swz(part * kC + t, ch) + hb) = pk;
      else
        *reinterpret_cast<uint2 *>(vp + cb * 8192 + swz(t, ch) + hb) = pk;
    }
  };
  FeTask fa, fb;
  fe_load(warp, fa);  // 24 tasks, three per warp
  // ---- gates of the chunk (warp 0): g2 = cumsum(log2 alpha); alpha = 1, beta = 0 past T
  if (warp == 0) {
    const int ta = t0 + 2 * lane, tb = ta + 1;
    const size_t ia = ((size_t)b * T + ta) * H + h, ib = ((size_t)b * T + tb) * H + h;
    const float a0 = ta < T ? p.alpha[ia] : 1.f, a1 = tb < T ? p.alpha[ib] : 1.f;
    const float l0 = log2f(a0), l1 = log2f(a1);
    float incl = l0 + l1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.f;
    const float ga = excl + l0, gb = ga + l1;
    g2s[2 * lane] = ga;
    g2s[2 * lane + 1] = gb;
    betas[2 * lane] = ta < T ? p.beta[ia] : 0.f;
    betas[2 * lane + 1] = tb < T ? p.beta[ib] : 0.f;
    p.Gp[unit * p.Tp + t0 + 2 * lane] = ga;
    p.Gp[unit * p.Tp + t0 + 2 * lane + 1] = gb;
  }

  const bool raw_ok = mbar_wait(bar_raw, 0);  // visibility of the raw tile to this thread
  fe_load(warp + 8, fb);
  fe_compute(warp, fa);
  fe_load(warp + 16, fa);
  fe_compute(warp + 8, fb);
  fe_compute(warp + 16, fa);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  // Q', K' rows to the workspace: 2 x 64 rows x 16 chunks of 16 bytes
  for (int it = tid; it < 2 * kC * 16; it += kPrepThreads) {
    const int part = it >> 10, rem = it & 1023, t = rem >> 4, ch = rem & 15;
    const uint4 v = *reinterpret_cast<const uint4 *>(qk + (ch >> 3) * 16384 + swz(part * kC + t, ch & 7));
    __nv_bfloat16 *dst = (part == 0 ? p.Qp : p.Kp) + (unit * p.Tp + t0 + t) * kD + ch * 8;
    *reinterpret_cast<uint4 *>(dst) = v;
  }

  // ---- [Q'; K'] K'^T: M = 128 (rows 0-63 Q'K'^T, rows 64-127 K'K'^T), N = 64
  if (tid == 0) {
    const uint64_t dA = desc_sw128(smem_u32(qk), 16, 1024);
    const uint64_t dB = desc_sw128(smem_u32(qk + 8192), 16, 1024);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t off = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
      umma_bf16(tm, dA + off, dB + off, idesc_bf16(128, 64, false, false), ks > 0);
    }
    umma_commit(bar);
  }
  bool ok = __syncthreads_and(mbar_wait(bar, 0) && raw_ok);
  tc_fence_after();

  // ---- A_ij = beta_i 2^(g_i - g_j) (k_i . k_j) for j < i (rows from TMEM lanes 64..127)
  // stored as the blocks A00, A10, A11 of 32 x 32 (A01 is zero)
  float *A00 = reinterpret_cast<float *>(smem + kOffA);
  float *A10 = A00 + kBlk * (kBlk + 1);
  float *A11 = A10 + kBlk * (kBlk + 1);
  float *T00 = reinterpret_cast<float *>(smem + kOffT);
  float *T10 = T00 + kBlk * (kBlk + 1);
  float *T11 = T10 + kBlk * (kBlk + 1);
  constexpr int kLd = kBlk + 1;
  if (ok && warp < 2) {  // column scales of T diag(beta gamma)
    const int k = 32 * warp + lane;
    colbg[k] = betas[k] * exp2f(g2s[k]);
  }
  // warps 2 and 6 read TMEM lanes 64-95 (K'K'^T rows 0-31), warps 3 and 7
  // lanes 96-127 (rows 32-63); warp w >> 2 takes column half w >> 2.  Rows
  // 0-31 x columns 32-63 form the zero block A01, so warp 6 has no work.
  if (ok && (warp & 3) >= 2 && warp != 6) {
    const int lq = warp & 3, half = warp >> 2;
    const int i = 32 * (lq - 2) + lane;
    float kk[32];
    tmem_ld32(tm + ((uint32_t)(32 * lq) << 16) + 32 * half, kk);
    const float gi = g2s[i], bi = betas[i];
    if (lq == 2) {
#pragma unroll
      for (int j = 0; j < 32; ++j) A00[lane * kLd + j] = (j < i) ? bi * exp2f(gi - g2s[j]) * kk[j] : 0.f;
    } else if (half == 0) {
#pragma unroll
      for (int j = 0; j < 32; ++j) A10[lane * kLd + j] = bi * exp2f(gi - g2s[j]) * kk[j];
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        A11[lane * kLd + j] = (32 + j < i) ? bi * exp2f(gi - g2s[32 + j]) * kk[j] : 0.f;
    }
  }
  __syncthreads();

  // ---- T = (I + A)^-1 in 32 x 32 blocks ---------------------------------------
  // T00 = (I + A00)^-1 and T11 = (I + A11)^-1 by forward substitution, both at
  // once: 4 lanes solve column kc of one block, lane `sub` holding x_j for
  // j = sub (mod 4), the partial sums combined with two shuffles per row.
  // Then T10 = -T11 A10 T00 as two fp32 products (T01 = 0).
  if (ok) {
    const int k = tid >> 2, sub = tid & 3, blk = k >> 5, kc = k & 31;
    const float *Ab = blk ? A11 : A00;
    float xs[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) xs[m] = 0.f;
#pragma unroll
    for (int i = 0; i < kBlk; ++i) {
      // x_j of rows not solved yet are still 0 and A is strictly lower, so
      // the bounds can be the compile-time 4m < i: every index stays static
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int m = 0; m < 8; m += 2) {
        if (4 * m < i) s0 = fmaf(Ab[i * kLd + 4 * m + sub], xs[m], s0);
        if (4 * (m + 1) < i) s1 = fmaf(Ab[i * kLd + 4 * (m + 1) + sub], xs[m + 1], s1);
      }
      float sum = s0 + s1;
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      if ((i & 3) == sub) xs[i >> 2] = (i == kc ? 1.f : 0.f) - sum;
    }
    float *Tb = blk ? T11 : T00;
#pragma unroll
    for (int m = 0; m < 8; ++m) Tb[(4 * m + sub) * kLd + kc] = xs[m];
  }
  __syncthreads();
  float *X = A00;  // A00 is no longer needed: X = A10 T00 takes its place
  // a warp computes rows warp, warp + 8, +16, +24 of a product, lane = column;
  // each element of the right factor is loaded once for the four rows
  if (ok) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int j = 0; j < kBlk; ++j) {
      const float t = T00[j * kLd + lane];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) acc[rr] += A10[(warp + 8 * rr) * kLd + j] * t;
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) X[(warp + 8 * rr) * kLd + lane] = acc[rr];
  }
  __syncthreads();
  if (ok) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int j = 0; j < kBlk; ++j) {
      const float x = X[j * kLd + lane];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) acc[rr] += T11[(warp + 8 * rr) * kLd + j] * x;
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) T10[(warp + 8 * rr) * kLd + lane] = -acc[rr];
  }
  __syncthreads();
  // ---- T diag(beta gamma) and T diag(beta) as bf16 hi / lo MMA tiles ------------
  if (ok) {
    uint8_t *tm1 = smem + kOffTm;  // T diag(beta gamma): hi, lo
    uint8_t *tm2 = tm1 + 16384;    // T diag(beta): hi, lo
    for (int it = tid; it < kC * 8; it += kPrepThreads) {  // (row i, 8-column chunk)
      const int i = it >> 3, chk = it & 7;
      float w1[8], w2[8];
#pragma unroll
      for (int e2 = 0; e2 < 8; ++e2) {
        const int k = 8 * chk + e2;
        float tv;
        if (i < kBlk) tv = k < kBlk ? T00[i * kLd + k] : 0.f;
        else tv = k < kBlk ? T10[(i - kBlk) * kLd + k] : T11[(i - kBlk) * kLd + (k - kBlk)];
        w1[e2] = tv * colbg[k];
        w2[e2] = tv * betas[k];
      }
      uint32_t h1[4], l1[4], h2[4], l2[4];
#pragma unroll
      for (int q2 = 0; q2 < 4; ++q2) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(w1[2 * q2], w1[2 * q2 + 1]);
        const __nv_bfloat162 c2 = __floats2bfloat162_rn(w2[2 * q2], w2[2 * q2 + 1]);
        h1[q2] = bits(a);
        h2[q2] = bits(c2);
        l1[q2] = bits(__floats2bfloat162_rn(w1[2 * q2] - __low2float(a), w1[2 * q2 + 1] - __high2float(a)));
        l2[q2] = bits(__floats2bfloat162_rn(w2[2 * q2] - __low2float(c2), w2[2 * q2 + 1] - __high2float(c2)));
      }
      const uint32_t off = swz(i, chk);
      *reinterpret_cast<uint4 *>(tm1 + off) = make_uint4(h1[0], h1[1], h1[2], h1[3]);
      *reinterpret_cast<uint4 *>(tm1 + 8192 + off) = make_uint4(l1[0], l1[1], l1[2], l1[3]);
      *reinterpret_cast<uint4 *>(tm2 + off) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
      *reinterpret_cast<uint4 *>(tm2 + 8192 + off) = make_uint4(l2[0], l2[1], l2[2], l2[3]);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- W = Tm1 K' (TMEM cols 0-127), U~ = Tm2 V' (cols 128-255): M = 64, N = 128
  if (ok && tid == 0) {
    const uint32_t id = idesc_bf16(64, 128, false, true);
    const uint64_t dT1 = desc_sw128(smem_u32(smem + kOffTm), 16, 1024);
    const uint64_t dT2 = desc_sw128(smem_u32(smem + kOffTm + 16384), 16, 1024);
    const uint64_t dK = desc_sw128(smem_u32(qk + 8192), 16384, 1024);
    const uint64_t dV = desc_sw128(smem_u32(vp), 8192, 1024);
#pragma unroll
    for (int part = 0; part < 2; ++part)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint32_t aoff = (part * 8192 + ks * 32) >> 4, boff = (ks * 2048) >> 4;
        umma_bf16(tm, dT1 + aoff, dK + boff, id, (part | ks) != 0);
        umma_bf16(tm + 128, dT2 + aoff, dV + boff, id, (part | ks) != 0);
      }
    umma_commit(bar);
  }
  if (ok) ok = __syncthreads_and(mbar_wait(bar, 1));
  tc_fence_after();

  // ---- W (bf16) and U~ (fp32) rows to the workspace ----------------------------
  if (ok) {
    // 16x256b reads of the M = 64 accumulators: rows r0 and r0 + 8, columns
    // 8m + cq and + 1 of each 64-column half
    const int q4 = warp & 3, r0 = 16 * q4 + (lane >> 2), cq = 2 * (lane & 3);
    const uint32_t base = tm + ((uint32_t)(32 * q4) << 16) + (warp < 4 ? 0u : 128u);
    const size_t row0 = unit * p.Tp + t0 + r0, row1 = row0 + 8;
    float v0[32], v1[32];
    tmem_ld16x256b_x8x2(base, base + 64, v0, v1);
    if (warp < 4) {
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float *v = m < 8 ? v0 : v1;
        const int mm = m & 7, col = 8 * m + cq;
        *reinterpret_cast<__nv_bfloat162 *>(p.Wp + row0 * kD + col) = __floats2bfloat162_rn(v[4 * mm], v[4 * mm + 1]);
        *reinterpret_cast<__nv_bfloat162 *>(p.Wp + row1 * kD + col) =
            __floats2bfloat162_rn(v[4 * mm + 2], v[4 * mm + 3]);
      }
    } else {
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float *v = m < 8 ? v0 : v1;
        const int mm = m & 7, col = 8 * m + cq;
        *reinterpret_cast<float2 *>(p.Up + row0 * kD + col) = make_float2(v[4 * mm], v[4 * mm + 1]);
        *reinterpret_cast<float2 *>(p.Up + row1 * kD + col) = make_float2(v[4 * mm + 2], v[4 * mm + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (!ok && tid == 0 && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_WAIT_TIMEOUT);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tm, 256);
  }
}

// ================================ pass B ====================================

constexpr int kBV = 32;          // d_v columns per CTA
constexpr int kNV = kD / kBV;    // CTAs per (batch, head)
constexpr int kStages = 2;
constexpr int kPrefetch = 3;  // chunks prefetched into L2 beyond the shared-memory ring
// warp 0 TMA, warp 1 MMA issuer of the state chain (W S, K'^T r U), warps 2-5 P,
// warps 6-9 U / state / outputs, warp 10 MMA issuer of the outputs (Q'S + P U),
// warp 11 MMA issuer of Q'K'^T (a thread issues one small MMA about every 85
// cycles, so the MMAs of a chunk are spread over three issuers)
constexpr int kThreads = 384;
constexpr uint32_t kTile = kC * kD * 2;        // Q', K' or W tile: 16 KiB (2 column blocks)
constexpr uint32_t kTileU = kC * kBV * 4;      // U~ slice, fp32: 8 KiB
constexpr uint32_t kStageBytes = 3 * kTile + kTileU;
constexpr uint32_t kTileP = kC * kC * 2;       // 8 KiB (one of hi / lo)
// A d_v slice of 32 bf16 high parts and its 32 remainders share one 128-byte
// swizzled row, so [hi | lo] is a single 64-wide MMA operand.
constexpr uint32_t kTileHL = kC * 128;         // [U_hi | U_lo] or [rU_hi | rU_lo]: 8 KiB
constexpr uint32_t kTileS = kD * 128;          // [S_hi | S_lo]: 16 KiB
constexpr uint32_t kOffStage = 0;
constexpr uint32_t kOffP = kStages * kStageBytes;   // P hi, lo
constexpr uint32_t kOffU = kOffP + 2 * kTileP;      // [U_hi | U_lo]
constexpr uint32_t kOffRU = kOffU + kTileHL;        // [rU_hi | rU_lo]
constexpr uint32_t kOffS = kOffRU + kTileHL;        // [S_hi | S_lo], double-buffered
constexpr uint32_t kOffG = kOffS + 2 * kTileS;      // gate rows [warp][2][64]
constexpr uint32_t kOffBar = kOffG + (kThreads / 32) * 2 * kC * 4;
constexpr uint32_t kScanSmem = kOffBar + 256 + 1024;
static_assert(kScanSmem <= 232448, "shared memory budget");
static_assert(kOffP % 1024 == 0 && kOffU % 1024 == 0 && kOffRU % 1024 == 0 && kOffS % 1024 == 0, "alignment");
// TMEM (64 columns each, the hi and lo products side by side): Q'K'^T,
// W[S_hi|S_lo], K'^T[rU_hi|rU_lo], and the outputs Q'[S_hi|S_lo] + P''[U_hi|U_lo]
constexpr uint32_t kColQK = 0, kColWS = 64, kColDS = 128, kColO = 192;
constexpr uint32_t kScanTmCols = 256;

struct ScanParams {
  int B, T, H, nchunks, Tp, out_bf16;
  int state_every, nblocks;  // states emitted after every state_every tokens (a multiple of 64)
  float *S_blocks;
  const float *alpha;
  const float *Gp;
  const float *S0;
  float *S_T;
  void *o;
  // conv cache hand-over (written by the vblk-0 CTA of each (b, h))
  int has_conv;
  const __nv_bfloat16 *q, *k, *v, *conv_in;
  __nv_bfloat16 *conv_out;
  uint32_t *dev_status;
};

struct ScanBars {
  uint64_t full[kStages], empty[kStages];
  uint64_t qk_ready, qk_free, p_ready, o_ready, o_free;
  uint64_t ws_ready, u_ready, ds_ready, s_ready, p_free;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(ScanBars) <= 256, "barrier block");

struct GateRow {
  float g0n, g1n;  // next chunk's g2 values, prefetched
};

__device__ __forceinline__ void grow_prefetch(GateRow &G, const ScanParams &p, size_t unit, int c,
                                              int lane) {
  const size_t base = unit * p.Tp + (size_t)c * kC + 2 * lane;
  const bool in = c < p.nchunks;
  G.g0n = in ? p.Gp[base] : 0.f;
  G.g1n = in ? p.Gp[base + 1] : 0.f;
}

__device__ __forceinline__ float grow_chunk(GateRow &G, const ScanParams &p, size_t unit, int c,
                                            int lane, float *row) {
  const float a = G.g0n, b = G.g1n;
  grow_prefetch(G, p, unit, c + 1, lane);
  __syncwarp();
  row[2 * lane] = a;
  row[2 * lane + 1] = b;
  __syncwarp();
  return row[kC - 1];
}

// kOutBf16, kEmit: output dtype and block-state emission as template
// parameters, so each instance carries only its own epilogue paths
template <bool kOutBf16, bool kEmit>
__global__ void __launch_bounds__(kThreads, 1)
    gdn_scan_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tu,
                    const ScanParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  ScanBars *bars = reinterpret_cast<ScanBars *>(smem + kOffBar);
  float *s_g = reinterpret_cast<float *>(smem + kOffG);
  volatile int *abort = &bars->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int vblk = blockIdx.x % kNV;
  const int bh = blockIdx.x / kNV;
  const int b = bh / p.H, h = bh - b * p.H;
  const size_t unit = (size_t)bh;
  const int T = p.T, nchunks = p.nchunks;

  // ---- the unit is skipped when a gate is outside (0, 1] ---------------------
  {
    int bad = 0;
    for (int t = tid; t < T; t += kThreads) {
      const float a = p.alpha[((size_t)b * T + t) * p.H + h];
      bad |= !(a > 0.f && a <= 1.f);
    }
    if (__syncthreads_or(bad)) {
      if (tid == 0 && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_BAD_GATE);
      return;
    }
  }
  // ---- conv cache hand-over: the last 3 raw inputs of this head's channels -----
  if (p.has_conv && p.conv_out && vblk == 0) {
    const int Cch = 3 * p.H * kD;
    __nv_bfloat16 vals[6];  // up to 2 (row, channel) items per thread: 3 x 384 / 320
    int n = 0;
    for (int it = tid; it < 3 * 3 * kD; it += kThreads, ++n) {
      const int j = it / (3 * kD), rem = it - j * 3 * kD, part = rem / kD, ch = rem - part * kD;
      const int t = T - 3 + j;
      __nv_bfloat16 x = __float2bfloat16_rn(0.f);
      if (t >= 0) {
        const __nv_bfloat16 *src = part == 0 ? p.q : (part == 1 ? p.k : p.v);
        x = src[(((size_t)b * T + t) * p.H + h) * kD + ch];
      } else if (p.conv_in) {
        x = p.conv_in[((size_t)b * 3 + (t + 3)) * Cch + part * p.H * kD + h * kD + ch];
      }
      vals[n] = x;
    }
    __syncthreads();  // every read of conv_in precedes the writes (they may alias)
    n = 0;
    for (int it = tid; it < 3 * 3 * kD; it += kThreads, ++n) {
      const int j = it / (3 * kD), rem = it - j * 3 * kD, part = rem / kD, ch = rem - part * kD;
      p.conv_out[((size_t)b * 3 + j) * Cch + part * p.H * kD + h * kD + ch] = vals[n];
    }
  }

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 3);  // one commit from each MMA issuer
    }
    // arrivals: one commit, or one per warp of a warpgroup
    mbar_init(&bars->qk_ready, 1);
    mbar_init(&bars->o_ready, 1);
    mbar_init(&bars->qk_free, 4);
    mbar_init(&bars->p_ready, 4);
    mbar_init(&bars->o_free, 4);
    mbar_init(&bars->ws_ready, 1);
    mbar_init(&bars->ds_ready, 1);
    mbar_init(&bars->p_free, 2);
    mbar_init(&bars->u_ready, 4);
    mbar_init(&bars->s_ready, 4);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kScanTmCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      prefetch_tensormap(&tq);
      prefetch_tensormap(&tk);
      prefetch_tensormap(&tw);
      prefetch_tensormap(&tu);
      auto prefetch = [&](int c) {  // chunk c's tiles into L2, ahead of the ring
        if (c >= nchunks) return;
        const int r0 = c * kC;
        tma_prefetch_l2_3d(&tq, 0, r0, (int)unit);
        tma_prefetch_l2_3d(&tq, 64, r0, (int)unit);
        tma_prefetch_l2_3d(&tk, 0, r0, (int)unit);
        tma_prefetch_l2_3d(&tk, 64, r0, (int)unit);
        tma_prefetch_l2_3d(&tw, 0, r0, (int)unit);
        tma_prefetch_l2_3d(&tw, 64, r0, (int)unit);
        tma_prefetch_l2_3d(&tu, vblk * kBV, r0, (int)unit);
      };
      for (int c = 0; c < kPrefetch; ++c) prefetch(kStages + c);
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % kStages;
        prefetch(c + kStages + kPrefetch);
        if (!wait_bar(&bars->empty[s], ((uint32_t)(c / kStages) & 1u) ^ 1u, abort)) break;
        uint8_t *st = smem + kOffStage + s * kStageBytes;
        uint64_t *fb = &bars->full[s];
        mbar_arrive_expect_tx(fb, kStageBytes);
        const int r0 = c * kC;
        tma_load_3d(st, &tq, fb, 0, r0, (int)unit);
        tma_load_3d(st + kTile / 2, &tq, fb, 64, r0, (int)unit);
        tma_load_3d(st + kTile, &tk, fb, 0, r0, (int)unit);
        tma_load_3d(st + kTile + kTile / 2, &tk, fb, 64, r0, (int)unit);
        tma_load_3d(st + 2 * kTile, &tw, fb, 0, r0, (int)unit);
        tma_load_3d(st + 2 * kTile + kTile / 2, &tw, fb, 64, r0, (int)unit);
        tma_load_3d(st + 3 * kTile, &tu, fb, vblk * kBV, r0, (int)unit);
      }
    }
  } else if (warp == 1) {
    // ============ MMA issuer A: the state chain, W S and K'^T r U ============
    // Its own thread, so these are issued the moment their inputs are ready
    // instead of queueing behind Q'K'^T, Q'S and P U.  S buffer c & 1 holds
    // the state before chunk c.
    if (lane == 0) {
      constexpr uint32_t id_xs = idesc_bf16(64, 2 * kBV, false, true);    // W [S_hi|S_lo]
      constexpr uint32_t id_ds = idesc_bf16(128, 2 * kBV, true, true);    // K'^T [rU_hi|rU_lo]
      const uint32_t sbase = smem_u32(smem);
      const uint64_t dRU = desc_sw128(sbase + kOffRU, 16, 1024);  // [rU_hi | rU_lo]
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % kStages;
        const uint32_t pc = (uint32_t)c & 1u;
        const uint32_t aQ = sbase + kOffStage + s * kStageBytes;
        const uint64_t dKm = desc_sw128(aQ + kTile, kTile / 2, 1024);
        const uint64_t dW = desc_sw128(aQ + 2 * kTile, 16, 1024);
        const uint64_t dS = desc_sw128(sbase + kOffS + (c & 1) * kTileS, 16, 1024);  // [S_hi | S_lo]
        if (!wait_bar(&bars->full[s], (uint32_t)(c / kStages) & 1u, abort)) break;
        if (!wait_bar(&bars->s_ready, pc, abort)) break;
        tc_fence_after();
        // W [S_hi | S_lo]: M = 64, N = 64, K = d_k (W tile K-major, S tile MN-major)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t aoff = ((ks >> 2) * (kTile / 2) + (ks & 3) * 32) >> 4;
          umma_bf16(tmem + kColWS, dW + aoff, dS + ((ks * 2048) >> 4), id_xs, ks > 0);
        }
        umma_commit(&bars->ws_ready);
        if (!wait_bar(&bars->u_ready, pc, abort)) break;
        tc_fence_after();
        // dS = K'^T [rU_hi | rU_lo]: M = d_k (K' tile read M-major), N = 64, K = 64 tokens
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tmem + kColDS, dKm + ((ks * 2048) >> 4), dRU + ((ks * 2048) >> 4), id_ds, ks > 0);
        umma_commit(&bars->ds_ready);
        umma_commit(&bars->p_free);    // r U may be rewritten
        umma_commit(&bars->empty[s]);  // W and K' of this stage are read
      }
    }
  } else if (warp < 6) {
    // ============ warpgroup A: P'' = (Q' K'^T) masked and scaled ============
    // P''_ij = (Q'K'^T)_ij 2^(g_i - g_j) / c_i for j <= i with the row scale
    // c_i = 2^max(g_i, -100): the outputs are c_i (Q' S + P'' U), both terms in
    // one accumulator.  16x256b layout: rows r0, r0 + 8, columns 8m + cq, + 1.
    const int q4 = warp & 3;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const int r0 = 16 * q4 + (lane >> 2), cq = 2 * (lane & 3);
    const uint32_t phi = smem_u32(smem + kOffP), plo = phi + kTileP;
    float *grow = s_g + warp * 2 * kC;
    GateRow G;
    grow_prefetch(G, p, unit, 0, lane);
    for (int c = 0; c < nchunks; ++c) {
      const uint32_t pc = (uint32_t)c & 1u;
      const float gC = grow_chunk(G, p, unit, c, lane, grow);
      if (!wait_bar_warp(&bars->qk_ready, pc, abort)) break;
      tc_fence_after();
      float qk[32];
      tmem_ld16x256b_x8(tmem + kColQK + lane_base, qk);
      tc_fence_before();
      warp_arrive(&bars->qk_free);
      const bool factored = gC > kRowScaleFloor;  // 2^-g <= 2^100: no overflow
      float *cfrow = grow + kC;
      if (factored) {
        cfrow[2 * lane] = exp2f(-grow[2 * lane]);
        cfrow[2 * lane + 1] = exp2f(-grow[2 * lane + 1]);
      }
      __syncwarp();
      if (factored) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int col = 8 * m + cq;
          const float f0 = cfrow[col], f1 = cfrow[col + 1];
          qk[4 * m + 0] = col <= r0 ? qk[4 * m + 0] * f0 : 0.f;
          qk[4 * m + 1] = col + 1 <= r0 ? qk[4 * m + 1] * f1 : 0.f;
          qk[4 * m + 2] = col <= r0 + 8 ? qk[4 * m + 2] * f0 : 0.f;
          qk[4 * m + 3] = col + 1 <= r0 + 8 ? qk[4 * m + 3] * f1 : 0.f;
        }
      } else {
        const float g0 = grow[r0], g1 = grow[r0 + 8];
        const float m0 = fmaxf(g0, kRowScaleFloor), m1 = fmaxf(g1, kRowScaleFloor);  // log2 c_i
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int col = 8 * m + cq;
          const float ga = grow[col], gb = grow[col + 1];
          qk[4 * m + 0] = col <= r0 ? qk[4 * m + 0] * exp2f((g0 - ga) - m0) : 0.f;
          qk[4 * m + 1] = col + 1 <= r0 ? qk[4 * m + 1] * exp2f((g0 - gb) - m0) : 0.f;
          qk[4 * m + 2] = col <= r0 + 8 ? qk[4 * m + 2] * exp2f((g1 - ga) - m1) : 0.f;
          qk[4 * m + 3] = col + 1 <= r0 + 8 ? qk[4 * m + 3] * exp2f((g1 - gb) - m1) : 0.f;
        }
      }
      if (!wait_bar_warp(&bars->p_free, pc ^ 1u, abort)) break;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        uint32_t h0, l0, h1, l1;
        split2(qk[4 * m + 0], qk[4 * m + 1], h0, l0);
        split2(qk[4 * m + 2], qk[4 * m + 3], h1, l1);
        const uint32_t o0 = swz(r0, m) + 2 * cq, o1 = swz(r0 + 8, m) + 2 * cq;
        sts32(phi + o0, h0);
        sts32(plo + o0, l0);
        sts32(phi + o1, h1);
        sts32(plo + o1, l1);
      }
      fence_proxy_async_smem();
      warp_arrive(&bars->p_ready);
    }
  } else if (warp < 10) {
    // ============ warpgroup B: U, the state chain and the outputs ============
    const int q4 = warp & 3;
    const int srow = 32 * q4 + lane;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    // the M = 64 accumulators in the 16x256b layout: rows r0, r0 + 8 and, of the
    // 32 slice columns, 8m + cq and + 1 (m = 0..3: high parts; + 32: remainders)
    const int r0 = 16 * q4 + (lane >> 2), cq = 2 * (lane & 3);
    float *grow = s_g + warp * 2 * kC;
    GateRow G;
    grow_prefetch(G, p, unit, 0, lane);
    float S[kBV];
    {
      const float *src = p.S0 ? p.S0 + ((unit * kD) + srow) * kD + vblk * kBV : nullptr;
#pragma unroll
      for (int j = 0; j < kBV; j += 4) {
        const float4 v4 = src ? *reinterpret_cast<const float4 *>(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        S[j] = v4.x; S[j + 1] = v4.y; S[j + 2] = v4.z; S[j + 3] = v4.w;
      }
    }
    // S row srow as [hi | lo]: 16-byte chunks 0-3 hold the high parts, 4-7 the remainders
    auto write_state = [&](int buf) {
      const uint32_t sb = smem_u32(smem + kOffS + buf * kTileS);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint4 vh, vl;
        split8(&S[8 * ch], vh, vl);
        sts128(sb + swz(srow, ch), vh);
        sts128(sb + swz(srow, 4 + ch), vl);
      }
      fence_proxy_async_smem();
      warp_arrive(&bars->s_ready);
    };
    write_state(0);
    bool ok = true;
    const uint32_t ub = smem_u32(smem + kOffU), rb = smem_u32(smem + kOffRU);
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % kStages;
      const uint32_t pc = (uint32_t)c & 1u;
      const uint32_t sph = (uint32_t)(c / kStages) & 1u;
      const int t0 = c * kC;
      const float gC = grow_chunk(G, p, unit, c, lane, grow);
      const float g0 = grow[r0], g1 = grow[r0 + 8];

      // ---- U = U~ - W S (the hi and lo products summed), r U -----------------------
      if (!wait_bar_warp(&bars->ws_ready, pc, abort)) { ok = false; break; }
      tc_fence_after();
      float ws[32];
      tmem_ld16x256b_x8(tmem + kColWS + lane_base, ws);
      if (!wait_bar_warp(&bars->full[s], sph, abort)) { ok = false; break; }
      if (!wait_bar_warp(&bars->p_free, pc ^ 1u, abort)) { ok = false; break; }
      {
        // the U~ slice rows are 128 bytes (32 fp32), loaded with the 128-byte swizzle
        const uint32_t ut = smem_u32(smem + kOffStage + s * kStageBytes + 3 * kTile);
        const float ra = exp2f(gC - g0), rc = exp2f(gC - g1);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int col = 8 * m + cq;
          const uint32_t uo = 4 * (col & 3);
          const float2 ua = lds64f(ut + swz(r0, col >> 2) + uo), uc = lds64f(ut + swz(r0 + 8, col >> 2) + uo);
          const float a0 = ua.x - (ws[4 * m + 0] + ws[4 * m + 16]), a1 = ua.y - (ws[4 * m + 1] + ws[4 * m + 17]);
          const float c0 = uc.x - (ws[4 * m + 2] + ws[4 * m + 18]), c1 = uc.y - (ws[4 * m + 3] + ws[4 * m + 19]);
          uint32_t h, l;
          split2(a0, a1, h, l);
          sts32(ub + swz(r0, m) + 2 * cq, h);
          sts32(ub + swz(r0, 4 + m) + 2 * cq, l);
          split2(c0, c1, h, l);
          sts32(ub + swz(r0 + 8, m) + 2 * cq, h);
          sts32(ub + swz(r0 + 8, 4 + m) + 2 * cq, l);
          split2(ra * a0, ra * a1, h, l);
          sts32(rb + swz(r0, m) + 2 * cq, h);
          sts32(rb + swz(r0, 4 + m) + 2 * cq, l);
          split2(rc * c0, rc * c1, h, l);
          sts32(rb + swz(r0 + 8, m) + 2 * cq, h);
          sts32(rb + swz(r0 + 8, 4 + m) + 2 * cq, l);
        }
      }
      fence_proxy_async_smem();
      warp_arrive(&bars->u_ready);

      // ---- S <- gamma_C S + K'^T diag(r) U (hi and lo products summed) -----------
      if (!wait_bar_warp(&bars->ds_ready, pc, abort)) { ok = false; break; }
      tc_fence_after();
      {
        const float gam = exp2f(gC);
        float dh[32], dl[32];
        tmem_ld32x2(tmem + kColDS + lane_base, tmem + kColDS + kBV + lane_base, dh, dl);
#pragma unroll
        for (int jj = 0; jj < kBV; ++jj) S[jj] = gam * S[jj] + (dh[jj] + dl[jj]);
      }
      // buffer (c + 1) & 1 was last read by W S and Q' S of the previous chunk,
      // both complete before that chunk's outputs were ready
      if (c + 1 < nchunks) write_state((c + 1) & 1);
      if (kEmit && ((c + 1) * kC) % p.state_every == 0 && (c + 1) * kC <= T) {
        // the state after this chunk closes a block: this thread's row slice goes out
        float *dst = p.S_blocks +
                     ((((size_t)b * p.nblocks + (c + 1) * kC / p.state_every - 1) * p.H + h) * kD + srow) * kD +
                     vblk * kBV;
#pragma unroll
        for (int j = 0; j < kBV; j += 4)
          *reinterpret_cast<float4 *>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
      }

      // ---- o = c_i (Q' S + P'' U), the hi and lo columns summed -----------------------
      if (!wait_bar_warp(&bars->o_ready, pc, abort)) { ok = false; break; }
      tc_fence_after();
      float ov[32];
      tmem_ld16x256b_x8(tmem + kColO + lane_base, ov);
      tc_fence_before();
      warp_arrive(&bars->o_free);
      {
        const float f0 = exp2f(fmaxf(g0, kRowScaleFloor)), f1 = exp2f(fmaxf(g1, kRowScaleFloor));
        const int ta = t0 + r0, tb2 = ta + 8;
        const size_t oa = (((size_t)b * T + ta) * p.H + h) * kD + vblk * kBV + cq;
        const size_t ob2 = (((size_t)b * T + tb2) * p.H + h) * kD + vblk * kBV + cq;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float x0 = f0 * (ov[4 * m + 0] + ov[4 * m + 16]), x1 = f0 * (ov[4 * m + 1] + ov[4 * m + 17]);
          const float y0 = f1 * (ov[4 * m + 2] + ov[4 * m + 18]), y1 = f1 * (ov[4 * m + 3] + ov[4 * m + 19]);
          if (kOutBf16) {
            __nv_bfloat16 *o16 = reinterpret_cast<__nv_bfloat16 *>(p.o);
            if (ta < T) *reinterpret_cast<__nv_bfloat162 *>(o16 + oa + 8 * m) = __floats2bfloat162_rn(x0, x1);
            if (tb2 < T) *reinterpret_cast<__nv_bfloat162 *>(o16 + ob2 + 8 * m) = __floats2bfloat162_rn(y0, y1);
          } else {
            float *o32 = reinterpret_cast<float *>(p.o);
            if (ta < T) *reinterpret_cast<float2 *>(o32 + oa + 8 * m) = make_float2(x0, x1);
            if (tb2 < T) *reinterpret_cast<float2 *>(o32 + ob2 + 8 * m) = make_float2(y0, y1);
          }
        }
      }
    }
    if (ok) {
      float *dst = p.S_T + ((unit * kD) + srow) * kD + vblk * kBV;
#pragma unroll
      for (int j = 0; j < kBV; j += 4)
        *reinterpret_cast<float4 *>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
  } else if (warp == 10) {
    // ============ MMA issuer B: the outputs Q'S + P'' U ============
    // Each output MMA group is issued right after the state-chain MMA it may
    // not delay has completed (Q'S after W S, P''U after K'^T r U), so the
    // chain's MMAs never wait behind the outputs' in the tensor pipe.
    if (lane == 0) {
      constexpr uint32_t id_xs = idesc_bf16(64, 2 * kBV, false, true);    // Q' [S_hi|S_lo]
      constexpr uint32_t id_pu = idesc_bf16(64, 2 * kBV, false, true);    // P'' [U_hi|U_lo]
      const uint32_t sbase = smem_u32(smem);
      const uint64_t dP = desc_sw128(sbase + kOffP, 16, 1024);
      const uint64_t dU = desc_sw128(sbase + kOffU, 16, 1024);    // [U_hi | U_lo]
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % kStages;
        const uint32_t pc = (uint32_t)c & 1u;
        const uint32_t aQ = sbase + kOffStage + s * kStageBytes;
        const uint64_t dQ = desc_sw128(aQ, 16, 1024);
        const uint64_t dS = desc_sw128(sbase + kOffS + (c & 1) * kTileS, 16, 1024);
        // Q' [S_hi | S_lo] once W S of this chunk is done (S_c is in place), and
        // the previous chunk's outputs are read
        if (!wait_bar(&bars->ws_ready, pc, abort)) break;
        if (!wait_bar(&bars->o_free, pc ^ 1u, abort)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t aoff = ((ks >> 2) * (kTile / 2) + (ks & 3) * 32) >> 4;
          umma_bf16(tmem + kColO, dQ + aoff, dS + ((ks * 2048) >> 4), id_xs, ks > 0);
        }
        // (P''hi + P''lo) [U_hi | U_lo] into the same columns, once K'^T r U is done
        if (!wait_bar(&bars->ds_ready, pc, abort)) break;
        if (!wait_bar(&bars->p_ready, pc, abort)) break;
        if (!wait_bar(&bars->u_ready, pc, abort)) break;
        tc_fence_after();
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_bf16(tmem + kColO, dP + ((part * kTileP + ks * 32) >> 4), dU + ((ks * 2048) >> 4), id_pu, 1u);
        umma_commit(&bars->o_ready);
        umma_commit(&bars->p_free);    // P'' and U may be rewritten
        umma_commit(&bars->empty[s]);  // Q' of this stage is read
      }
    }
  } else {
    // ============ MMA issuer QK: Q'K'^T of each chunk as soon as it may ============
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16(64, 64, false, false);        // Q' K'^T
      const uint32_t sbase = smem_u32(smem);
      for (int c = 0; c < nchunks; ++c) {  // M = 64 tokens, N = 64 tokens, K = d_k
        const int s = c % kStages;
        if (!wait_bar(&bars->full[s], (uint32_t)(c / kStages) & 1u, abort)) break;
        if (!wait_bar(&bars->qk_free, ((uint32_t)c & 1u) ^ 1u, abort)) break;
        tc_fence_after();
        const uint32_t aQ = sbase + kOffStage + s * kStageBytes;
        const uint64_t dQ = desc_sw128(aQ, 16, 1024), dK = desc_sw128(aQ + kTile, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = ((ks >> 2) * (kTile / 2) + (ks & 3) * 32) >> 4;
          umma_bf16(tmem + kColQK, dQ + off, dK + off, id_qk, ks > 0);
        }
        umma_commit(&bars->qk_ready);
        umma_commit(&bars->empty[s]);  // Q' and K' of this stage are read by Q'K'^T
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort && tid == 0 && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_WAIT_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kScanTmCols);
  }
}

// ================================ host ======================================

struct Workspace {
  __nv_bfloat16 *Qp, *Kp, *Wp;
  float *Up, *Gp;
  size_t bytes;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

Workspace carve(void *base, int B, int H, int Tp) {
  Workspace w;
  const size_t rows = (size_t)B * H * Tp;
  size_t off = 0;
  uint8_t *p = reinterpret_cast<uint8_t *>(base);
  w.Qp = reinterpret_cast<__nv_bfloat16 *>(p + off);
  off = align256(off + rows * kD * 2);
  w.Kp = reinterpret_cast<__nv_bfloat16 *>(p + off);
  off = align256(off + rows * kD * 2);
  w.Wp = reinterpret_cast<__nv_bfloat16 *>(p + off);
  off = align256(off + rows * kD * 2);
  w.Up = reinterpret_cast<float *>(p + off);
  off = align256(off + rows * kD * 4);
  w.Gp = reinterpret_cast<float *>(p + off);
  off = align256(off + rows * 4);
  w.bytes = off;
  return w;
}

}  // namespace

bool gdn_tc_supports(const glinattn_prefill_args &a) {
  return a.variant == GLINATTN_GDN && a.in_dtype == GLINATTN_BF16 && a.dk == kD && a.dv == kD &&
         (a.qk_heads == 0 || a.qk_heads == a.heads) && a.seqlen > 0;
}

size_t gdn_tc_workspace_bytes(const glinattn_prefill_args &a) {
  const int Tp = (a.seqlen + kC - 1) / kC * kC;
  return carve(nullptr, a.batch, a.heads, Tp).bytes;
}

glinattn_status launch_gdn_tc(const glinattn_prefill_args &a, cudaStream_t stream) {
  const int B = a.batch, T = a.seqlen, H = a.heads;
  const int nchunks = (T + kC - 1) / kC, Tp = nchunks * kC;
  const Workspace w = carve(a.workspace, B, H, Tp);
  if (!a.workspace || a.workspace_bytes < w.bytes) return GLINATTN_ERR_INVALID_ARG;

  PrepParams pp;
  pp.B = B; pp.T = T; pp.H = H; pp.nchunks = nchunks; pp.Tp = Tp;
  pp.qk_l2norm = a.qk_l2norm != 0;
  pp.has_conv = a.conv_w != nullptr;
  pp.q = static_cast<const __nv_bfloat16 *>(a.q);
  pp.k = static_cast<const __nv_bfloat16 *>(a.k);
  pp.v = static_cast<const __nv_bfloat16 *>(a.v);
  pp.alpha = a.alpha; pp.beta = a.beta; pp.conv_w = a.conv_w;
  pp.conv_in = static_cast<const __nv_bfloat16 *>(a.conv_in);
  pp.Qp = w.Qp; pp.Kp = w.Kp; pp.Wp = w.Wp; pp.Up = w.Up; pp.Gp = w.Gp;
  pp.dev_status = a.dev_status;
  auto prep = pp.has_conv ? (pp.qk_l2norm ? gdn_prep_kernel<true, true> : gdn_prep_kernel<true, false>)
                          : (pp.qk_l2norm ? gdn_prep_kernel<false, true> : gdn_prep_kernel<false, false>);
  if (cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kPrepSmem) != cudaSuccess)
    return GLINATTN_ERR_CUDA;
  CUtensorMap rq, rk, rv;  // raw activations, 64-token x 64-channel boxes
  if (!make_act_map(&rq, a.q, B, T, H, kD) || !make_act_map(&rk, a.k, B, T, H, kD) ||
      !make_act_map(&rv, a.v, B, T, H, kD))
    return GLINATTN_ERR_CUDA;
  prep<<<dim3(nchunks, H, B), kPrepThreads, kPrepSmem, stream>>>(rq, rk, rv, pp);
  if (cudaGetLastError() != cudaSuccess) return GLINATTN_ERR_CUDA;

  CUtensorMap tq, tk, tw, tu;
  const int rows_bh = B * H;
  if (!encode_rows_map(&tq, w.Qp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, Tp, rows_bh, 64, true) ||
      !encode_rows_map(&tk, w.Kp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, Tp, rows_bh, 64, true) ||
      !encode_rows_map(&tw, w.Wp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, Tp, rows_bh, 64, true) ||
      !encode_rows_map(&tu, w.Up, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, kD, Tp, rows_bh, kBV, true))
    return GLINATTN_ERR_CUDA;
  ScanParams sp;
  sp.B = B; sp.T = T; sp.H = H; sp.nchunks = nchunks; sp.Tp = Tp;
  sp.out_bf16 = a.out_dtype == GLINATTN_BF16;
  sp.alpha = a.alpha; sp.Gp = w.Gp; sp.S0 = a.S0; sp.S_T = a.S_T; sp.o = a.o;
  sp.has_conv = a.conv_w != nullptr;
  sp.q = pp.q; sp.k = pp.k; sp.v = pp.v; sp.conv_in = pp.conv_in;
  sp.conv_out = static_cast<__nv_bfloat16 *>(a.conv_out);
  sp.dev_status = a.dev_status;
  sp.state_every = a.state_every > 0 && T / a.state_every > 0 ? a.state_every : 0;
  sp.nblocks = sp.state_every ? T / sp.state_every : 0;
  sp.S_blocks = a.S_blocks;
  auto scan = sp.out_bf16 ? (sp.state_every ? gdn_scan_kernel<true, true> : gdn_scan_kernel<true, false>)
                          : (sp.state_every ? gdn_scan_kernel<false, true> : gdn_scan_kernel<false, false>);
  if (cudaFuncSetAttribute(scan, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kScanSmem) != cudaSuccess)
    return GLINATTN_ERR_CUDA;
  scan<<<(unsigned)(B * H * kNV), kThreads, kScanSmem, stream>>>(tq, tk, tw, tu, sp);
  return cudaGetLastError() == cudaSuccess ? GLINATTN_OK : GLINATTN_ERR_CUDA;
}

}  // namespace glinattn
